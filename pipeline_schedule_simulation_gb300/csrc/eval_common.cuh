// eval_common.cuh -- pieces shared by the two evaluator kernels.
//
// Work decomposition: one thread per schedule instance, one warp per 32
// instances.  All instances of a call share the plan, so every lane of a warp
// walks the same per-round op table: descriptor loads are warp-uniform and the
// per-op branches never diverge.  A round holds at most one op per device, and
// ops within a round are independent (rounds are a topological order of the
// dependency graph), so a thread evaluates its instance round by round.
//
// Cost staging: each warp keeps a ring of NSLOT round-slices in shared memory,
// laid out [slice][device][lane], filled D = NSLOT-1 rounds ahead with
// cp.async.  With the instance-minor cost layout (stride_inst == 1) a group of
// 8 lanes copies the 128 contiguous bytes of one (stage, microbatch) row for
// the warp's 32 instances in 16-byte pieces, so every global load is
// coalesced and 128-bit; the compute reads its own word conflict-free.
#pragma once

#include <cstdint>

#include "checks.cuh"
#include "internal.cuh"

namespace pps {

struct EvalArgs {
    const uint32_t *desc;    // [R][PMAX]
    const uint32_t *desc2;   // [R][PMAX] (generic evaluator)
    const uint64_t *rw;      // [R] per-round kind words and patterns
    const uint4 *seg;        // [nseg] segments
    int nseg;
    const uint4 *ktab;       // register evaluator's tables for these strides
    int ktab_words;
    int R, P, M, v, S, O, nslots;
    const int32_t *cost_f, *cost_b;
    int64_t s_inst, s_stage, s_mb;
    const int32_t *comm;
    const int32_t *comm_b;   // latency of the backward edges (same strides), null: comm
    int64_t c_inst, c_bnd;
    int64_t n;
    int64_t inst_begin;      // first instance of this launch
    int64_t tasks;           // register evaluator: > 0 when block b takes warp tasks
                             // [b*tasks/grid, (b+1)*tasks/grid); 0: one per warp in grid order
    int32_t *makespan, *idle;
    int64_t *bub_num, *bub_den;
    int8_t *status;
    int32_t *op_start, *op_end;
    int64_t o_inst, o_op;
    const int32_t *peak_src;  // the plan's peak held activations per device [P]
    int32_t *peak_dst;        // the caller's copy of it, written by block 0; null: none
};

// The cost-independent peak of the plan goes to the caller's array from inside
// the evaluation kernel, so a call is one launch (no separate copy on the
// stream).  Block 0's first P threads, before any early exit; every block has
// at least one warp and P <= 16.
__device__ __forceinline__ void copy_peak(const EvalArgs &a, int64_t bid) {
    if (a.peak_dst && bid == 0 && threadIdx.x < (unsigned)a.P) a.peak_dst[threadIdx.x] = a.peak_src[threadIdx.x];
}
__device__ __forceinline__ void copy_peak(const EvalArgs &a) { copy_peak(a, blockIdx.x); }

// One problem of a fused launch over many problems (pp_sched_many_*): its
// arguments as pp_sched_eval would pass them, the lane evaluator's table and
// block count (unused by the register kernel), and the problem's first CTA in
// the fused grid.  A fused kernel finds its problem by binary search over
// block_begin (ascending) and runs the single-problem body with the CTA's
// index within the problem.
struct ManyJob {
    EvalArgs a;
    const uint4 *tab;
    int nblocks;
    int64_t block_begin;
};

__device__ __forceinline__ int many_job_of(const ManyJob *jobs, int njobs, int64_t cta) {
    int lo = 0, hi = njobs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (jobs[mid].block_begin <= cta) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Loader-table entry of an idle (round, device) slot.
constexpr uint32_t kLtIdle = 0xFFFFFFFFu;

// Round slices kept per warp: enough prefetch depth to cover HBM latency
// while the ring stays at 8 KB per warp.
template <int PMAX, int NI = 1>
struct Ring {
    static constexpr int kSlices = PMAX == 4 ? 16 : 8;
    static constexpr int kAhead = kSlices - 1;   // kernels that step one round at a time
    static constexpr int kAhead2 = kSlices - 2;  // kernels that may step two rounds at once
    static constexpr int kWords = kSlices * PMAX * NI * 32;
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

// 16 bytes, or 16 zero bytes without reading the source when `zero` is set.
__device__ __forceinline__ void cp_async16_or_zero(uint32_t dst, const void *src, bool zero) {
    asm volatile(
        "{\n .reg .pred z;\n setp.ne.b32 z, %2, 0;\n cp.async.cg.shared.global [%0], [%1], 16, z;\n}\n" ::"r"(dst),
        "l"(src), "r"((uint32_t)zero)
        : "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// The loader's view of one round: the descriptors of the devices this lane
// copies for (vector path: devices 4i + lane/8; scalar path: every device).
template <int PMAX, bool VEC>
struct LoadDesc {
    static constexpr int kN = VEC ? PMAX / 4 : PMAX;
    uint32_t d[kN];
};

template <int PMAX, bool VEC>
__device__ __forceinline__ void fetch_load_desc(const EvalArgs &a, int rl, int lane, LoadDesc<PMAX, VEC> &ld) {
    const uint32_t *drow = a.desc + (int64_t)rl * PMAX;
#pragma unroll
    for (int i = 0; i < LoadDesc<PMAX, VEC>::kN; ++i)
        ld.d[i] = __ldg(drow + (VEC ? 4 * i + (lane >> 3) : i));
}

// Issue the copies of round `rl`'s costs into ring slice rl % kSlices.  The
// vector path needs every element offset to fit in 32 bits (checked on the
// host) and computes it in 32-bit arithmetic.
template <int PMAX, bool VEC>
__device__ __forceinline__ void load_round(const EvalArgs &a, int rl, const LoadDesc<PMAX, VEC> &ld,
                                           int32_t *ring, int64_t inst0, int lane) {
    using RG = Ring<PMAX>;
    int32_t *slice = ring + (rl % RG::kSlices) * (PMAX * 32);
    if constexpr (VEC) {
        // lanes 8q..8q+7 cover device 4*i + q, 4 instances each
        const int g = lane & 7;
        const int64_t x0 = inst0 + 4 * g;
        const int64_t left = a.n - x0;
        const uint32_t bytes_in = left <= 0 ? 0u : (left >= 4 ? 16u : (uint32_t)left * 4u);
        const int s_stage = (int)a.s_stage, s_mb = (int)a.s_mb;
#pragma unroll
        for (int i = 0; i < PMAX / 4; ++i) {
            const int k = 4 * i + (lane >> 3);
            const uint32_t d = ld.d[i];
            const uint32_t kind = desc_kind(d);
            const int32_t *base = kind == kBwd ? a.cost_b : a.cost_f;
            const int s = (int)desc_chunk(d) * a.P + k;
            const int32_t *src = base;
            uint32_t nb = 0;
            if (kind != kIdle && bytes_in) {
                const int64_t off = (int64_t)(s * s_stage + (int)desc_mb(d) * s_mb) + x0;
                if (PPS_CHECK(off + bytes_in / 4 <= cost_reach(a.n, a.S, a.M, a.s_inst, a.s_stage, a.s_mb),
                              kChkCostRead, off)) {
                    src = base + off;
                    nb = bytes_in;
                }
            }
            cp_async16(smem_addr(slice + k * 32 + 4 * g), src, nb);
        }
    } else {
        const int64_t x = inst0 + lane;
        const bool live = x < a.n;
#pragma unroll
        for (int k = 0; k < PMAX; ++k) {
            const uint32_t d = ld.d[k];
            const uint32_t kind = desc_kind(d);
            const int32_t *base = kind == kBwd ? a.cost_b : a.cost_f;
            const int32_t *src = base;
            uint32_t nb = 0;
            if (kind != kIdle && live) {
                const int64_t s = (int64_t)desc_chunk(d) * a.P + k;
                const int64_t off = s * a.s_stage + (int64_t)desc_mb(d) * a.s_mb + x * a.s_inst;
                if (PPS_CHECK(off < cost_reach(a.n, a.S, a.M, a.s_inst, a.s_stage, a.s_mb), kChkCostRead, off)) {
                    src = base + off;
                    nb = 4;
                }
            }
            cp_async4(smem_addr(slice + k * 32 + lane), src, nb);
        }
    }
}

// Loader table (see k_ktab in plan.cu): for every (round, device) the element
// offset of the op's cost row relative to its array, shifted left by one with
// bit 0 set for a backward op; kLtIdle for an idle slot.  Offsets stay below
// 2^30 (checked on the host).

// Vector loader driven by the table: a row (one device's cost for the warp's
// 32*NI instances) takes 8*NI lanes, 16 bytes (4 instances) each; lane copies
// row 32/(8*NI)*i + lane/(8*NI) for i = 0 .. PMAX*NI/4 - 1.  The slice is laid
// out [device][instance]; fbase/bbase already point at this lane's instances.
// (x0, reach: the element offset of fbase / bbase from the tables' bases and
// the elements the strides reach; used by the checked build only.)
template <int PMAX, int NI>
__device__ __forceinline__ void load_round_lt(const uint32_t *lt, int rl, int32_t *ring, const int32_t *fbase,
                                              const int32_t *bbase, uint32_t bytes_in, int lane,
                                              [[maybe_unused]] int64_t x0, [[maybe_unused]] int64_t reach) {
    using RG = Ring<PMAX, NI>;
    constexpr int kLanesPerRow = 8 * NI, kRowsPerInst = 32 / kLanesPerRow;
    int32_t *slice = ring + (rl % RG::kSlices) * (PMAX * NI * 32);
    const int g = lane % kLanesPerRow;
#pragma unroll
    for (int i = 0; i < PMAX / kRowsPerInst; ++i) {
        const int k = kRowsPerInst * i + lane / kLanesPerRow;
        const uint32_t e = lt[rl * PMAX + k];
        const int32_t *src = (e & 1u) ? bbase : fbase;
        uint32_t nb = 0;
        if (e != kLtIdle && PPS_CHECK(x0 + (e >> 1) + bytes_in / 4 <= reach, kChkCostRead, x0 + (e >> 1))) {
            src += e >> 1;
            nb = bytes_in;
        }
        cp_async16(smem_addr(slice + k * (NI * 32) + 4 * g), src, nb);
    }
}

// The same loader for a warp whose 32*NI instances all exist: every copy is a
// whole 16 bytes, and an idle slot is zero-filled without a read.  `e` holds
// this lane's table entries of the round (rows 32/(8*NI)*i + lane/(8*NI)),
// read ahead by the caller; `dst` is the shared address of this lane's first
// chunk in the round's slice.
template <int PMAX, int NI>
__device__ __forceinline__ void load_round_lt_q(const uint32_t (&e)[PMAX * NI / 4], uint32_t dst, const int32_t *fbase,
                                                const int32_t *bbase, [[maybe_unused]] int64_t x0,
                                                [[maybe_unused]] int64_t reach) {
    constexpr int kRowsPerInst = 32 / (8 * NI);
#pragma unroll
    for (int i = 0; i < PMAX * NI / 4; ++i) {
        const bool idle = e[i] == kLtIdle || !PPS_CHECK(e[i] == kLtIdle || x0 + (e[i] >> 1) + 4 <= reach,
                                                        kChkCostRead, x0 + (e[i] >> 1));
        const int32_t *src = ((e[i] & 1u) ? bbase : fbase) + (idle ? 0u : (e[i] >> 1));
        cp_async16_or_zero(dst + (uint32_t)(i * kRowsPerInst * NI * 32 * 4), src, idle);
    }
}

// True if any cost of instance x is negative (read from global memory; used
// only to classify an instance whose sticky sign flag was raised).
static __device__ __noinline__ bool any_negative_cost(const EvalArgs &a, int64_t x) {
    for (int s = 0; s < a.S; ++s)
        for (int i = 0; i < a.M; ++i) {
            const int64_t off = x * a.s_inst + (int64_t)s * a.s_stage + (int64_t)i * a.s_mb;
            if (a.cost_f[off] < 0 || a.cost_b[off] < 0) return true;
        }
    return false;
}

// Per-instance reductions for the unsigned evaluators.  `flag` carries the
// sign bits of every op's start tick and cost (see k_eval_reg): it is clear
// exactly when no cost is negative and every tick fits in int32.  A raised
// flag is classified by re-reading the instance's costs.
template <int PMAX>
__device__ __forceinline__ void write_results_u(const EvalArgs &a, int64_t x, const uint32_t (&fr)[PMAX],
                                                const uint32_t (&busy)[PMAX], uint32_t flag, bool neg_comm) {
    uint32_t mk = 0;
#pragma unroll
    for (int k = 0; k < PMAX; ++k) mk = max(mk, fr[k]);
    flag |= mk;
    int64_t num = 0;
#pragma unroll
    for (int k = 0; k < PMAX; ++k) {
        if (k < a.P) {
            const int idle = (int)(mk - busy[k]);
            num += idle;
            if (a.idle) a.idle[x * a.P + k] = idle;
        }
    }
    if (a.makespan) a.makespan[x] = (int)mk;
    if (a.bub_num) a.bub_num[x] = num;
    if (a.bub_den) a.bub_den[x] = (int64_t)a.P * (int)mk;
    if (a.status) {
        int8_t st = PP_ST_OK;
        if (neg_comm) st = PP_ST_NEG_COST;
        else if (flag >> 31) st = any_negative_cost(a, x) ? PP_ST_NEG_COST : PP_ST_OVERFLOW;
        a.status[x] = st;
    }
}

// Warp-cooperative version of write_results_u for the warp's 32 instances
// starting at x0 (this lane's instance is x0 + lane): the [n][P] idle block of
// the warp is contiguous, so it is staged through `scratch` (32*P words of the
// warp's own shared memory, free at this point) and written with consecutive
// lanes on consecutive words.  Called by all 32 lanes.
template <int PMAX>
__device__ __forceinline__ void write_results_warp(const EvalArgs &a, int64_t x0, int lane,
                                                   const uint32_t (&fr)[PMAX], const uint32_t (&busy)[PMAX],
                                                   uint32_t flag, bool neg_comm, int32_t *scratch) {
    const int64_t x = x0 + lane;
    const bool live = x < a.n;
    uint32_t mk = 0;
#pragma unroll
    for (int k = 0; k < PMAX; ++k) mk = max(mk, fr[k]);
    flag |= mk;
    int64_t num = 0;
#pragma unroll
    for (int k = 0; k < PMAX; ++k) {
        if (k < a.P) {
            const int idle = (int)(mk - busy[k]);
            num += idle;
            scratch[lane * a.P + k] = idle;
        }
    }
    if (live) {
        if (a.makespan) a.makespan[x] = (int)mk;
        if (a.bub_num) a.bub_num[x] = num;
        if (a.bub_den) a.bub_den[x] = (int64_t)a.P * (int)mk;
        if (a.status) {
            int8_t st = PP_ST_OK;
            if (neg_comm) st = PP_ST_NEG_COST;
            else if (flag >> 31) st = any_negative_cost(a, x) ? PP_ST_NEG_COST : PP_ST_OVERFLOW;
            a.status[x] = st;
        }
    }
    __syncwarp();
    if (a.idle) {
        const int64_t valid = (a.n - x0 < 32 ? a.n - x0 : 32) * a.P;
        int32_t *dst = a.idle + x0 * a.P;
        for (int w = lane; w < valid; w += 32) dst[w] = scratch[w];
    }
    __syncwarp();
}

// Load the round's descriptors (identical for every lane of the warp).
template <int PMAX>
__device__ __forceinline__ void load_desc(const uint32_t *row, uint32_t (&d)[PMAX]) {
    const uint4 *r4 = reinterpret_cast<const uint4 *>(row);
#pragma unroll
    for (int i = 0; i < PMAX / 4; ++i) {
        const uint4 q = __ldg(r4 + i);
        d[4 * i + 0] = q.x; d[4 * i + 1] = q.y; d[4 * i + 2] = q.z; d[4 * i + 3] = q.w;
    }
}

// Write the per-instance reductions ("2. 1F1B" §4.3 and M040 §04: the window is
// the last end tick; each stage's idle time is the window minus its busy time;
// the bubble is total idle over P windows).
template <int PMAX>
__device__ __forceinline__ void write_results(const EvalArgs &a, int64_t x, const int (&fr)[PMAX],
                                              const int (&busy)[PMAX], uint32_t neg_bits,
                                              uint32_t ovf_bits) {
    int mk = 0;
#pragma unroll
    for (int k = 0; k < PMAX; ++k) mk = max(mk, fr[k]);
    int64_t num = 0;
#pragma unroll
    for (int k = 0; k < PMAX; ++k) {
        if (k < a.P) {
            const int idle = mk - busy[k];
            num += idle;
            if (a.idle) a.idle[x * a.P + k] = idle;
        }
    }
    if (a.makespan) a.makespan[x] = mk;
    if (a.bub_num) a.bub_num[x] = num;
    if (a.bub_den) a.bub_den[x] = (int64_t)a.P * mk;
    if (a.status) {
        int8_t st = PP_ST_OK;
        if (neg_bits >> 31) st = PP_ST_NEG_COST;
        else if (ovf_bits >> 31) st = PP_ST_OVERFLOW;
        a.status[x] = st;
    }
}

// int32 add without C++ signed-overflow semantics; overflow is detected by the
// sign bit of the result (all true values are >= 0 and < 2^31, so a sum of two
// wraps past INT32_MAX exactly when its sign bit is set).
__device__ __forceinline__ int wrap_add(int x, int y) {
    return static_cast<int>(static_cast<uint32_t>(x) + static_cast<uint32_t>(y));
}

// SMs of device `dev` (cached per device and translation unit).
inline int sm_count(int dev) {
    static int cached[64] = {};
    if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = 1;
    }
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
}

// Launchers (defined in eval_reg.cu / eval_slot.cu / eval_lane.cu / eval_split.cu).
int launch_eval_reg(pp_plan *plan, EvalArgs &a, bool vec, bool ops, cudaStream_t st);
bool reg_table_path(int pmax, const EvalArgs &a, bool vec);
int launch_eval_reg_tables(int pmax, const EvalArgs &a, bool vec, bool ops, cudaStream_t st);
int launch_eval_slot(const pp_plan *plan, const EvalArgs &a, bool vec, bool ops, cudaStream_t st);
bool lane_path(const pp_plan *plan, const EvalArgs &a);
int launch_eval_split8(const EvalArgs &a, cudaStream_t st);
int launch_eval_lane(pp_plan *plan, const EvalArgs &a, bool vec, bool ops, cudaStream_t st);

// Fused launches over many problems (pp_sched_many_*).  *_ok answers whether
// the fused kernel takes a problem (lane_mbz_ok also sets a.nslots); its
// tables are built by build_tables (register evaluator's for reg, lane
// evaluator's with one instance set per lane for lane); *_warps is the warps its
// instances fill, *_ctas the CTAs of `warps` warps it needs, *_smem the
// dynamic shared memory of such a CTA; launch_*_many runs a group of jobs of
// one table width, already in device memory, with CTAs of `warps` warps (at
// most kManyRegWarps / kManyLaneWarps).
constexpr int kManyRegWarps = 4, kManyLaneWarps = 2;
bool reg_mbz_ok(const pp_plan *plan, const EvalArgs &a);
int64_t reg_mbz_warps(const EvalArgs &a);
int64_t reg_mbz_ctas(const EvalArgs &a, int warps);
size_t reg_mbz_smem(int pmax, const EvalArgs &a, int warps);
int launch_reg_mbz_many(int pmax, int warps, const ManyJob *d_jobs, int njobs, int64_t ctas, size_t smem,
                        cudaStream_t st);
bool lane_mbz_ok(const pp_plan *plan, EvalArgs &a);
int64_t lane_mbz_warps(int pmax, const EvalArgs &a);
int64_t lane_mbz_ctas(int pmax, const EvalArgs &a, int warps);
size_t lane_mbz_smem(int pmax, const EvalArgs &a, int warps);
int launch_lane_mbz_many(int pmax, int warps, const ManyJob *d_jobs, int njobs, int64_t ctas, size_t smem,
                         cudaStream_t st);

// Argument checks and EvalArgs of pp_sched_eval (eval_reg.cu), shared with
// the multi-problem entry points.
int eval_check(pp_policy_t policy, int P, int M, int v, const int32_t *cost_f, const int32_t *cost_b,
               int64_t stride_inst, int64_t stride_stage, int64_t stride_mb, int64_t comm_stride_inst,
               int64_t comm_stride_bnd, int64_t n_instances);
EvalArgs eval_args(const pp_plan *plan, const int32_t *cost_f, const int32_t *cost_b, int64_t stride_inst,
                   int64_t stride_stage, int64_t stride_mb, const int32_t *comm, const int32_t *comm_b,
                   int64_t comm_stride_inst, int64_t comm_stride_bnd, int64_t n_instances, int32_t *makespan,
                   int32_t *idle, int64_t *bub_num, int64_t *bub_den, int32_t *peak, int32_t *op_start,
                   int32_t *op_end, int64_t op_stride_inst, int64_t op_stride_op, int8_t *status);

}  // namespace pps
