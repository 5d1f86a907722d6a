// noalloc.cu -- pp_sched_eval_noalloc: the GPipe / 1F1B evaluation without
// any device allocation.
//
// pp_sched_eval keeps each shape's schedule tables in device memory it
// allocates the first time it sees the shape.  Some callers cannot let a
// library call cudaMalloc: a caller whose device memory is owned by another
// allocator (a framework's caching pool that must account for every byte), a
// process that must not grow or fragment its device footprint once it is
// running, or code on a path where allocating would synchronize the device.
// For them this entry point builds the schedule tables inside one fixed
// array that the library declares at file scope, so the only device memory it
// touches besides the caller's own buffers is reserved when the library is
// loaded.
//
// The array is a static __device__ symbol: every GPU that loads the library
// holds its 4 MiB until the process exits.  Host code cannot use the symbol's
// name as a device address (it names a host-side stand-in), so the device
// address is fetched with cudaGetSymbolAddress, once per device, with that
// device current, on the first call made on that device.
#include <cstdio>
#include <mutex>

#include "eval_common.cuh"

namespace pps {
namespace {

// 4 MiB of schedule tables (plan + per-stride kernel tables).
constexpr int64_t kNoAllocWords = (int64_t)1 << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint32_t g_noalloc_tables[kNoAllocWords];

// Per-device state: the array's device address and what the array holds now
// (so a repeated call with the same shape and strides reuses the tables).
struct DeviceScratch {
    uint32_t *addr = nullptr;
    bool valid = false;
    int policy = -1, P = 0, M = 0;
    int64_t s_stage = -1, s_mb = -1;
    bool with_ktab = false;
    ScratchPlan sp{};
};

std::mutex g_mu;
DeviceScratch g_dev[kMaxDevices];

// Device address of the array on the current device (fetched once per device).
int scratch_for_current_device(DeviceScratch **out) {
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return PP_ERR_SIZE;
    DeviceScratch &d = g_dev[dev];
    if (!d.addr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_tables);
        if (e != cudaSuccess || !p) return cuda_status(e);
        d.addr = static_cast<uint32_t *>(p);
    }
    *out = &d;
    return PP_OK;
}

}  // namespace
}  // namespace pps

extern "C" int pp_sched_eval_noalloc(pp_policy_t policy, int P, int M, const int32_t *cost_f,
                                     const int32_t *cost_b, int64_t stride_inst, int64_t stride_stage,
                                     int64_t stride_mb, const int32_t *comm, int64_t comm_stride_inst,
                                     int64_t comm_stride_bnd, int64_t n_instances, int32_t *makespan,
                                     int32_t *idle, int64_t *bub_num, int64_t *bub_den, int32_t *peak,
                                     int8_t *status, cudaStream_t stream) {
    using namespace pps;
    if (policy != PP_GPIPE && policy != PP_1F1B) return PP_ERR_ARG;
    int rc = check_shape((int)policy, P, M, 1);
    if (rc) return rc;
    if (n_instances < 0) return PP_ERR_ARG;
    if (n_instances > 0 && (!cost_f || !cost_b)) return PP_ERR_ARG;
    if (stride_inst < 0 || stride_stage < 0 || stride_mb < 0 || comm_stride_inst < 0 || comm_stride_bnd < 0)
        return PP_ERR_ARG;

    std::lock_guard<std::mutex> lk(g_mu);
    DeviceScratch *d = nullptr;
    rc = scratch_for_current_device(&d);
    if (rc) return rc;

    const bool vec = stride_inst == 1 && (reinterpret_cast<uintptr_t>(cost_f) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(cost_b) & 15) == 0 && stride_stage % 4 == 0 &&
                     stride_mb % 4 == 0 &&
                     (int64_t)(P - 1) * stride_stage + (int64_t)(M - 1) * stride_mb < ((int64_t)1 << 31);

    // (Re)build the tables unless the array already holds this shape's.
    const bool same_shape = d->valid && d->policy == (int)policy && d->P == P && d->M == M;
    if (!same_shape) {
        d->valid = false;
        rc = plan_into((int)policy, P, M, d->addr, kNoAllocWords, stream, &d->sp);
        if (rc) return rc;
        d->valid = true;
        d->policy = (int)policy; d->P = P; d->M = M;
        d->with_ktab = false; d->s_stage = -1; d->s_mb = -1;
    }

    EvalArgs a{};
    a.desc = d->sp.desc; a.desc2 = nullptr; a.rw = d->sp.rw;
    a.seg = d->sp.seg; a.nseg = d->sp.nseg;
    a.R = d->sp.R; a.P = P; a.M = M; a.v = 1; a.S = P; a.O = 2 * M; a.nslots = 0;
    a.cost_f = cost_f; a.cost_b = cost_b;
    a.s_inst = stride_inst; a.s_stage = stride_stage; a.s_mb = stride_mb;
    a.comm = comm; a.c_inst = comm_stride_inst; a.c_bnd = comm_stride_bnd;
    a.n = n_instances; a.inst_begin = 0;
    a.makespan = makespan; a.idle = idle; a.bub_num = bub_num; a.bub_den = bub_den; a.status = status;
    a.op_start = nullptr; a.op_end = nullptr; a.o_inst = 0; a.o_op = 0;
    a.ktab = nullptr; a.ktab_words = 0;
    if (reg_table_path(d->sp.pmax, a, vec)) {
        if (!d->with_ktab || d->s_stage != stride_stage || d->s_mb != stride_mb) {
            // ktab_into writes right after the plan's tables (used_words, which it
            // does not advance), so another stride pair's tables are replaced in place.
            d->sp.ktab_words = 0;
            d->with_ktab = false;
            rc = ktab_into(&d->sp, stride_stage, stride_mb, stream);
            if (rc) return rc;
            d->with_ktab = true; d->s_stage = stride_stage; d->s_mb = stride_mb;
        }
        a.ktab = reinterpret_cast<const uint4 *>(d->sp.ktab);
        a.ktab_words = d->sp.ktab_words;
    }
    if (peak)
        PPS_CUDA_TRY(cudaMemcpyAsync(peak, d->sp.peak, P * sizeof(int32_t), cudaMemcpyDeviceToDevice, stream));
    if (n_instances == 0) return PP_OK;
    return launch_eval_reg_tables(d->sp.pmax, a, vec, false, stream);
}
