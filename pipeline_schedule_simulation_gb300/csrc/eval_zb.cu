// eval_zb.cu -- the Zero Bubble schedules ZB1P and ZB2P.
//
// [GPipe->ZB] "Zero Bubble" and "ZB1P and ZB2P"; [1F1B] §6.2.  The backward
// of microbatch i on stage k splits into B(k,i) (input gradient, which stage
// k-1 waits for) and W(k,i) (weight gradient, which only needs B(k,i) on the
// same device).  F and B keep 1F1B's order F^w (B F)^(M-w) B^w (w = min(P-k,
// M) for ZB1P, min(2(P-k), M) for ZB2P); a device holds at most L = P (ZB1P)
// or 2P (ZB2P) microbatches whose W has not run; a device that becomes free at
// tick t runs the oldest pending W if its next F/B op is an F and it holds L,
// else that F/B op if its input has arrived by t, else the oldest pending W,
// else it waits for the input.  With no F/B op left it runs its pending W's.
//
// The op order depends on the costs, so there is no plan and no wavefront:
// every device is a small state machine.  One lane per (instance, device), a
// warp holds 32/PMAX instances (lane = device * 32/PMAX + instance).  In each
// step every lane takes at most one decision, and only one the rules already
// fix: its next F/B op's input has been placed (the arrival tick is known), or
// the producer device's current free tick proves the input cannot arrive by
// the decision tick (an F or B costs at least one tick, so a producer op not
// placed yet ends after the producer's free tick plus the costs of the
// producer's ops up to and including it).  Otherwise the lane waits a step.
// Every decision is the one the rules fix, so the result does not depend on
// the order of the steps.  While an instance is unfinished, some
// device of it places an op in every step: following "waits for the input of"
// from any waiting device walks the acyclic dependency graph back to an op
// whose input is known.  An instance therefore takes at most 3*P*M + 1 steps.
//
// Per warp, in shared memory ([row][lane], conflict-free):
//   cost rings  [3 kinds][kRing]: the costs of the next microbatches of each
//               kind, copied by cp.async kAheadC microbatches ahead; each step
//               commits one group and a lane consumes at most one op per step,
//               so the copy of a kind's next microbatch was issued at least
//               kAheadC - 1 steps ago: each step first waits for every group
//               but the last kAheadC - 2
//   arrival rings [2][kQ]: the arrival tick of F(k-1, i) at row i mod kQ of
//               the first ring (written by lane k-1) and of B(k+1, i) in the
//               second (written by lane k+1).  At most 2P results of a kind
//               wait for one device, and kQ = 2*PMAX.
#include "eval_common.cuh"

namespace pps {

template <int PMAX>
struct ZbGeom {
    static constexpr int kIPW = 32 / PMAX;  // instances per warp
    static constexpr int kRing = 8;         // cost ring rows per kind
    static constexpr int kAheadC = kRing - 1;
    static constexpr int kQ = 2 * PMAX;     // arrival ring rows
    static constexpr int kWords = (3 * kRing + 2 * kQ) * 32;  // per warp
    static constexpr int kWarps = 4;
    static_assert((kRing & (kRing - 1)) == 0 && (kQ & (kQ - 1)) == 0, "rings are indexed by masks");
};

constexpr int kZbF = 0, kZbB = 1, kZbW = 2;

// True if instance x has a negative cost or comm (then PP_ST_NEG_COST), or an F
// or B cost below 1 (PP_ST_ZERO_COST); read from global memory, used only to
// classify an instance whose flags were raised.
static __device__ __noinline__ int8_t zb_classify(const EvalArgs &a, const int32_t *cost_w, int64_t x) {
    bool zero = false;
    for (int s = 0; s < a.P; ++s) {
        if (a.comm && s < a.P - 1 && a.comm[x * a.c_inst + (int64_t)s * a.c_bnd] < 0) return PP_ST_NEG_COST;
        for (int i = 0; i < a.M; ++i) {
            const int64_t off = x * a.s_inst + (int64_t)s * a.s_stage + (int64_t)i * a.s_mb;
            const int32_t f = a.cost_f[off], b = a.cost_b[off], w = cost_w[off];
            if (f < 0 || b < 0 || w < 0) return PP_ST_NEG_COST;
            if (f < 1 || b < 1) zero = true;
        }
    }
    return zero ? PP_ST_ZERO_COST : PP_ST_OVERFLOW;
}

template <int PMAX, bool OPS>
__global__ void __launch_bounds__(128) k_eval_zb(const EvalArgs a, const int32_t *cost_w, int32_t *peak_out, int L,
                                                 int zb2) {
    using G = ZbGeom<PMAX>;
    extern __shared__ __align__(16) uint32_t zsm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int j = lane % G::kIPW, k = lane / G::kIPW;
    uint32_t *cring = zsm + warp * G::kWords;   // [3][kRing][32]
    uint32_t *fring = cring + 3 * G::kRing * 32;  // [kQ][32]
    uint32_t *bring = fring + G::kQ * 32;         // [kQ][32]
    const int64_t x = ((int64_t)blockIdx.x * G::kWarps + warp) * G::kIPW + j;
    const int P = a.P, M = a.M;
    const bool dev = x < a.n && k < P;  // this lane simulates a device

    // per-lane constants: warmup, comm on the left / right boundary, cost rows
    const int w = min(zb2 ? 2 * (P - k) : P - k, M);
    uint32_t cmL = 0, cmR = 0, ncomm = 0;
    if (dev && a.comm) {
        if (k > 0) cmL = (uint32_t)a.comm[x * a.c_inst + (int64_t)(k - 1) * a.c_bnd];
        if (k < P - 1) cmR = (uint32_t)a.comm[x * a.c_inst + (int64_t)k * a.c_bnd];
        ncomm = cmL | cmR;
    }
    const int64_t row0 = dev ? x * a.s_inst + (int64_t)k * a.s_stage : 0;
    const int32_t *src[3] = {a.cost_f + row0, a.cost_b + row0, cost_w + row0};
    [[maybe_unused]] const int64_t reach = cost_reach(a.n, P, M, a.s_inst, a.s_stage, a.s_mb);
    auto fetch = [&](int kind, int m) {
        if (dev && m < M && PPS_CHECK(row0 + (int64_t)m * a.s_mb < reach, kChkCostRead, row0 + (int64_t)m * a.s_mb)) {
            const int32_t *p = kind == kZbF ? src[0] : (kind == kZbB ? src[1] : src[2]);
            cp_async4(smem_addr(cring + (kind * G::kRing + (m & (G::kRing - 1))) * 32 + lane),
                      p + (int64_t)m * a.s_mb, 4);
        }
    };
#pragma unroll 1
    for (int m = 0; m < G::kAheadC; ++m) {
        fetch(kZbF, m);
        fetch(kZbB, m);
        fetch(kZbW, m);
    }
    cp_async_commit();
    // Zero arrival rings: the first device's forward input and the last
    // device's backward input have no producer, their column is never
    // written and reads 0 (arrival at tick 0).
#pragma unroll
    for (int q = 0; q < G::kQ; ++q) {
        fring[q * 32 + lane] = 0u;
        bring[q * 32 + lane] = 0u;
    }
    cp_async_wait<0>();
    __syncwarp();

    uint32_t t = 0, busy = 0, flag = 0, zero = 0;
    int nf = 0, nb = 0, nw = 0, held = 0, peak = 0;
    bool done = !dev;
    // After each step every lane publishes its counts and two lower bounds:
    // lbF, the earliest end of its next F, and lbB, of its next B (its free
    // tick plus the costs of the ops its order puts before them).  A consumer
    // whose input is not placed yet knows the producer's next op of that kind
    // is exactly the one it waits for.
    int nfL = 0, nbR = 0;
    uint32_t lbL = 0, lbR = 0;
    const int max_steps = 3 * P * M + 2;
    bool capped = true;
    // whether F/B op number pp of the device's order F^w (B F)^(M-w) B^w is an F
    auto is_fwd = [&](int pp) {
        const int q = pp - w;
        return q < 0 || (q < 2 * (M - w) && (q & 1));
    };
    // carried across steps: F/B ops placed, and whether the next one is an F
    int p = 0;
    bool isF = is_fwd(0);
#pragma unroll 1
    for (int step = 0; step < max_steps; ++step) {
        cp_async_wait<G::kAheadC - 2>();
        __syncwarp();
        // ---- decide (every lane evaluates the rules; no divergent paths)
        const bool pend = nw < nb;
        const bool haveX = p < 2 * M;
        const int mx = isF ? nf : nb;
        // the input's arrival: row mx of the ring of the op's kind (0 for the
        // first device's forward and the last device's backward)
        const uint32_t arr = (isF ? fring : bring)[(mx & (G::kQ - 1)) * 32 + lane];
        const bool known = isF ? (k == 0 || nfL > nf) : (k == P - 1 || nbR > nb);
        // the input has not arrived by t: known and later, or provably later
        const uint32_t lower = isF ? lbL + cmL : lbR + cmR;
        const bool late = known ? arr > t : lower > t;
        const int kX = isF ? kZbF : kZbB;
        int kind = -1;
        uint32_t s = t;
        if (!done) {
            if (!haveX) kind = pend ? kZbW : -1;
            else if (isF && nf - nw >= L) kind = kZbW;
            else if (known && !late) kind = kX;
            else if (late && pend) kind = kZbW;
            else if (known) { kind = kX; s = arr; }
        }
        done = done || (!haveX && !pend);
        // ---- place (predicated on kind >= 0)
        const bool act = kind >= 0;
        const int m = kind == kZbW ? nw : mx;
        const int kr = act ? kind : 0;
        const uint32_t c = cring[(kr * G::kRing + (m & (G::kRing - 1))) * 32 + lane];
        const uint32_t e = s + c;
        if (act) {
            flag |= s | c;
            zero |= (kind != kZbW && c == 0) ? 1u : 0u;
            busy += c;
            t = e;
            fetch(kind, m + G::kAheadC);
            if (kind == kZbF && k + 1 < P) fring[(m & (G::kQ - 1)) * 32 + lane + G::kIPW] = e + cmR;
            if (kind == kZbB && k > 0) bring[(m & (G::kQ - 1)) * 32 + lane - G::kIPW] = e + cmL;
            if constexpr (OPS) {
                const int64_t off = x * a.o_inst + ((int64_t)(k * 3 + kind) * M + m) * a.o_op;
                if (a.op_start) a.op_start[off] = (int32_t)s;
                if (a.op_end) a.op_end[off] = (int32_t)e;
            }
        }
        nf += kind == kZbF;
        nb += kind == kZbB;
        nw += kind == kZbW;
        held += (kind == kZbF) - (kind == kZbW);
        peak = max(peak, held);
        // ---- publish
        p = nf + nb;
        isF = is_fwd(p);
        const uint32_t cF = nf < M ? cring[(kZbF * G::kRing + (nf & (G::kRing - 1))) * 32 + lane] : 0u;
        const uint32_t cB = nb < M ? cring[(kZbB * G::kRing + (nb & (G::kRing - 1))) * 32 + lane] : 0u;
        const bool moreX = p < 2 * M;
        const uint32_t lbF = t + ((moreX && !isF) ? cB : 0u) + cF;
        const uint32_t lbB = t + ((moreX && isF) ? cF : 0u) + cB;
        cp_async_commit();
        __syncwarp();
        nfL = __shfl_up_sync(0xFFFFFFFFu, nf, G::kIPW);
        nbR = __shfl_down_sync(0xFFFFFFFFu, nb, G::kIPW);
        lbL = __shfl_up_sync(0xFFFFFFFFu, lbF, G::kIPW);
        lbR = __shfl_down_sync(0xFFFFFFFFu, lbB, G::kIPW);
        // a finished lane takes no decision, so the end is checked every
        // fourth step
        if ((step & 3) == 3 && __all_sync(0xFFFFFFFFu, done)) { capped = false; break; }
    }
    cp_async_wait<0>();

    // per-instance reductions over the instance's lanes (as the other
    // evaluators: window = last end tick, idle = window - busy, bubble = total
    // idle over P windows)
    uint32_t mk = dev ? t : 0u, fl = flag, zr = zero, nc = ncomm;
    uint32_t cp = capped && !done ? 1u : 0u;
#pragma unroll
    for (int d = G::kIPW; d < 32; d <<= 1) {
        mk = max(mk, __shfl_xor_sync(0xFFFFFFFFu, mk, d));
        fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, d);
        zr |= __shfl_xor_sync(0xFFFFFFFFu, zr, d);
        nc |= __shfl_xor_sync(0xFFFFFFFFu, nc, d);
        cp |= __shfl_xor_sync(0xFFFFFFFFu, cp, d);
    }
    fl |= mk;
    const int idle = dev ? (int)(mk - busy) : 0;
    int64_t num = idle;
#pragma unroll
    for (int d = G::kIPW; d < 32; d <<= 1) num += __shfl_xor_sync(0xFFFFFFFFu, num, d);
    if (!dev) return;
    if (a.idle) a.idle[x * P + k] = idle;
    if (peak_out) peak_out[x * P + k] = peak;  // per instance: the order depends on the costs
    if (k == 0) {
        if (a.makespan) a.makespan[x] = (int)mk;
        if (a.bub_num) a.bub_num[x] = num;
        if (a.bub_den) a.bub_den[x] = (int64_t)P * (int)mk;
        if (a.status) {
            int8_t st = PP_ST_OK;
            if (nc >> 31) st = PP_ST_NEG_COST;
            else if ((fl >> 31) || zr || cp) st = zb_classify(a, cost_w, x);
            a.status[x] = st;
        }
    }
}

namespace {

template <int PMAX, bool OPS>
int launch_zb_t(const EvalArgs &a, const int32_t *cost_w, int32_t *peak, int L, int zb2, cudaStream_t st) {
    using G = ZbGeom<PMAX>;
    const size_t smem = (size_t)G::kWarps * G::kWords * sizeof(uint32_t);
    const int64_t warps = (a.n + G::kIPW - 1) / G::kIPW;
    const int64_t blocks = (warps + G::kWarps - 1) / G::kWarps;
    if (blocks > 0x7FFFFFFF) return PP_ERR_SIZE;
    k_eval_zb<PMAX, OPS><<<(unsigned)blocks, G::kWarps * 32, smem, st>>>(a, cost_w, peak, L, zb2);
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}

template <int PMAX>
int launch_zb_p(const EvalArgs &a, const int32_t *cost_w, int32_t *peak, int L, int zb2, bool ops, cudaStream_t st) {
    return ops ? launch_zb_t<PMAX, true>(a, cost_w, peak, L, zb2, st)
               : launch_zb_t<PMAX, false>(a, cost_w, peak, L, zb2, st);
}

}  // namespace
}  // namespace pps

extern "C" int pp_sched_eval_zb(pp_policy_t policy, int P, int M, const int32_t *cost_f, const int32_t *cost_b,
                                const int32_t *cost_w, int64_t stride_inst, int64_t stride_stage,
                                int64_t stride_mb, const int32_t *comm, int64_t comm_stride_inst,
                                int64_t comm_stride_bnd, int64_t n_instances, int32_t *makespan, int32_t *idle,
                                int64_t *bub_num, int64_t *bub_den, int32_t *peak, int32_t *op_start,
                                int32_t *op_end, int64_t op_stride_inst, int64_t op_stride_op, int8_t *status,
                                cudaStream_t stream) {
    using namespace pps;
    if (policy != PP_ZB1P && policy != PP_ZB2P) return PP_ERR_ARG;
    if (P < 1 || M < 1 || n_instances < 0) return PP_ERR_ARG;
    if (P > PP_MAX_P || M > PP_MAX_MV) return PP_ERR_SIZE;
    if (n_instances > 0 && (!cost_f || !cost_b || !cost_w)) return PP_ERR_ARG;
    if (stride_inst < 0 || stride_stage < 0 || stride_mb < 0 || comm_stride_inst < 0 || comm_stride_bnd < 0)
        return PP_ERR_ARG;
    const bool ops = op_start || op_end;
    if (ops && (op_stride_inst < 0 || op_stride_op < 0)) return PP_ERR_ARG;
    if (n_instances == 0) return PP_OK;
    EvalArgs a{};
    a.R = 0; a.P = P; a.M = M; a.v = 1; a.S = P; a.O = 3 * M; a.nslots = 0;
    a.cost_f = cost_f; a.cost_b = cost_b;
    a.s_inst = stride_inst; a.s_stage = stride_stage; a.s_mb = stride_mb;
    a.comm = comm; a.c_inst = comm_stride_inst; a.c_bnd = comm_stride_bnd;
    a.n = n_instances; a.inst_begin = 0;
    a.makespan = makespan; a.idle = idle; a.bub_num = bub_num; a.bub_den = bub_den; a.status = status;
    a.op_start = op_start; a.op_end = op_end; a.o_inst = op_stride_inst; a.o_op = op_stride_op;
    const int L = policy == PP_ZB1P ? P : 2 * P;
    const int zb2 = policy == PP_ZB2P;
    switch (pmax_for(P)) {
        case 4: return launch_zb_p<4>(a, cost_w, peak, L, zb2, ops, stream);
        case 8: return launch_zb_p<8>(a, cost_w, peak, L, zb2, ops, stream);
        case 16: return launch_zb_p<16>(a, cost_w, peak, L, zb2, ops, stream);
        default: return PP_ERR_INTERNAL;
    }
}
