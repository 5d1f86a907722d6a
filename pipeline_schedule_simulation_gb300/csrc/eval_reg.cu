// eval_reg.cu -- the register evaluator (GPipe and 1F1B) and pp_sched_eval.
//
// The max-plus recurrence, per op in round order ("Pipeline parallelism: from
// GPipe to 1F1B and Zero Bubble", GPipe figure text and M040 §01/§08: the
// backward needs the downstream backward and its own forward; each stage runs
// one op at a time):
//     start = max(end of the device's previous op, arrival of its input)
//     end   = start + cost
// where the input of F(k,i) is F(k-1,i), arriving comm[k-1] after it ends, and
// the input of B(k,i) is B(k+1,i), arriving comm[k] after it ends (B's need of
// F(k,i) is covered by the device order).  For these two policies the plan
// verified that an op's input is always the latest result of its kind on the
// neighbouring device at the start of the op's round, so the whole state of an
// instance is four registers per device: the device's free tick, the arrival
// tick of its latest F and latest B at the neighbour, and its busy ticks.
#include "eval_common.cuh"

namespace pps {

template <int PMAX, bool VEC, bool OPS>
__global__ void __launch_bounds__(128) k_eval_reg(const EvalArgs a) {
    using RG = Ring<PMAX>;
    extern __shared__ __align__(16) int32_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t *ring = smem + warp * RG::kWords;
    const int64_t inst0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + warp) * 32;
    if (inst0 >= a.n) return;  // warp-uniform
    const int64_t x = inst0 + lane;
    const bool live = x < a.n;

    // Outgoing comm per device: a forward result of device k crosses boundary k,
    // a backward result of device k crosses boundary k-1.
    int cF[PMAX], cB[PMAX];
    uint32_t neg = 0;
#pragma unroll
    for (int k = 0; k < PMAX; ++k) {
        cF[k] = 0;
        cB[k] = 0;
        if (a.comm && live) {
            if (k < a.P - 1) cF[k] = a.comm[x * a.c_inst + (int64_t)k * a.c_bnd];
            if (k >= 1 && k < a.P) cB[k] = a.comm[x * a.c_inst + (int64_t)(k - 1) * a.c_bnd];
        }
        neg |= (uint32_t)cF[k] | (uint32_t)cB[k];
    }
    int fr[PMAX], rf[PMAX], rb[PMAX], busy[PMAX], cnt[PMAX];
#pragma unroll
    for (int k = 0; k < PMAX; ++k) { fr[k] = 0; rf[k] = 0; rb[k] = 0; busy[k] = 0; cnt[k] = 0; }
    uint32_t accE = 0, accC = 0;

    const int R = a.R;
#pragma unroll 1
    for (int q = 0; q < RG::kAhead; ++q) {
        if (q < R) load_round<PMAX, VEC>(a, q, ring, inst0, lane);
        cp_async_commit();
    }
#pragma unroll 1
    for (int r = 0; r < R; ++r) {
        if (r + RG::kAhead < R) load_round<PMAX, VEC>(a, r + RG::kAhead, ring, inst0, lane);
        cp_async_commit();
        uint32_t d[PMAX];
        load_desc<PMAX>(a.desc + (int64_t)r * PMAX, d);
        cp_async_wait<RG::kAhead>();
        __syncwarp();
        const int32_t *slice = ring + (r % RG::kSlices) * (PMAX * 32);
        int rf0[PMAX], rb0[PMAX];  // inputs are read as of the start of the round
#pragma unroll
        for (int k = 0; k < PMAX; ++k) { rf0[k] = rf[k]; rb0[k] = rb[k]; }
#pragma unroll
        for (int k = 0; k < PMAX; ++k) {
            const uint32_t kind = desc_kind(d[k]);
            if (kind == kIdle) continue;
            const int c = slice[k * 32 + lane];
            int arr;
            if (kind == kFwd) arr = k > 0 ? rf0[k > 0 ? k - 1 : 0] : 0;
            else arr = k < PMAX - 1 ? rb0[k < PMAX - 1 ? k + 1 : 0] : 0;
            const int st = max(fr[k], arr);
            const int en = wrap_add(st, c);
            fr[k] = en;
            busy[k] = wrap_add(busy[k], c);
            accE |= (uint32_t)en | (uint32_t)arr;
            accC |= (uint32_t)c;
            if (kind == kFwd) rf[k] = wrap_add(en, cF[k]);
            else rb[k] = wrap_add(en, cB[k]);
            if constexpr (OPS) {
                if (live) {
                    const int64_t off = x * a.o_inst + ((int64_t)k * a.O + cnt[k]) * a.o_op;
                    if (a.op_start) a.op_start[off] = st;
                    if (a.op_end) a.op_end[off] = en;
                }
                ++cnt[k];
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();
    if (live) write_results<PMAX>(a, x, fr, busy, accC | neg, accE);
}

template <int PMAX, bool VEC, bool OPS>
static int launch_reg_t(const EvalArgs &a, cudaStream_t st) {
    constexpr int kWarps = 2;
    const size_t smem = (size_t)kWarps * Ring<PMAX>::kWords * sizeof(int32_t);
    const int64_t warps = (a.n + 31) / 32;
    const int64_t blocks = (warps + kWarps - 1) / kWarps;
    if (blocks > 0x7FFFFFFF) return PP_ERR_SIZE;
    k_eval_reg<PMAX, VEC, OPS><<<(unsigned)blocks, kWarps * 32, smem, st>>>(a);
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}

template <int PMAX>
static int launch_reg_p(const EvalArgs &a, bool vec, bool ops, cudaStream_t st) {
    if (vec) return ops ? launch_reg_t<PMAX, true, true>(a, st) : launch_reg_t<PMAX, true, false>(a, st);
    return ops ? launch_reg_t<PMAX, false, true>(a, st) : launch_reg_t<PMAX, false, false>(a, st);
}

int launch_eval_reg(const pp_plan *plan, const EvalArgs &a, bool vec, bool ops, cudaStream_t st) {
    switch (plan->pmax) {
        case 4: return launch_reg_p<4>(a, vec, ops, st);
        case 8: return launch_reg_p<8>(a, vec, ops, st);
        case 16: return launch_reg_p<16>(a, vec, ops, st);
        default: return PP_ERR_INTERNAL;
    }
}

}  // namespace pps

extern "C" int pp_sched_eval(pp_policy_t policy, int P, int M, int v, const int32_t *cost_f,
                             const int32_t *cost_b, int64_t stride_inst, int64_t stride_stage,
                             int64_t stride_mb, const int32_t *comm, int64_t comm_stride_inst,
                             int64_t comm_stride_bnd, int64_t n_instances, int32_t *makespan,
                             int32_t *idle, int64_t *bub_num, int64_t *bub_den, int32_t *peak,
                             int32_t *op_start, int32_t *op_end, int64_t op_stride_inst,
                             int64_t op_stride_op, int8_t *status, cudaStream_t stream) {
    using namespace pps;
    int rc = check_shape((int)policy, P, M, v);
    if (rc) return rc;
    if (n_instances < 0) return PP_ERR_ARG;
    if (n_instances > 0 && (!cost_f || !cost_b)) return PP_ERR_ARG;
    if (stride_inst < 0 || stride_stage < 0 || stride_mb < 0 || comm_stride_inst < 0 ||
        comm_stride_bnd < 0)
        return PP_ERR_ARG;
    if ((op_start || op_end) && (op_stride_inst < 0 || op_stride_op < 0)) return PP_ERR_ARG;
    const pp_plan *plan = nullptr;
    rc = cached_plan((int)policy, P, M, v, stream, &plan);
    if (rc) return rc;
    if (peak)
        PPS_CUDA_TRY(cudaMemcpyAsync(peak, plan->d_peak, P * sizeof(int32_t), cudaMemcpyDeviceToDevice, stream));
    if (n_instances == 0) return PP_OK;
    EvalArgs a;
    a.desc = plan->d_desc; a.desc2 = plan->d_desc2;
    a.R = plan->R; a.P = P; a.M = M; a.v = v; a.S = plan->S; a.O = plan->O; a.nslots = plan->nslots;
    a.cost_f = cost_f; a.cost_b = cost_b;
    a.s_inst = stride_inst; a.s_stage = stride_stage; a.s_mb = stride_mb;
    a.comm = comm; a.c_inst = comm_stride_inst; a.c_bnd = comm_stride_bnd;
    a.n = n_instances;
    a.makespan = makespan; a.idle = idle; a.bub_num = bub_num; a.bub_den = bub_den; a.status = status;
    a.op_start = op_start; a.op_end = op_end; a.o_inst = op_stride_inst; a.o_op = op_stride_op;
    const bool vec = stride_inst == 1 && (reinterpret_cast<uintptr_t>(cost_f) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(cost_b) & 15) == 0 && stride_stage % 4 == 0 &&
                     stride_mb % 4 == 0;
    const bool ops = op_start || op_end;
    if (plan->reg_ok) return launch_eval_reg(plan, a, vec, ops, stream);
    return launch_eval_slot(plan, a, vec, ops, stream);
}
