// eval_dp.cu -- DualPipe: two routes through the same blocks of layers in
// opposite directions.
//
// [GPipe->ZB] "DualPipe (DeepSeek-V3)": route A's microbatches enter at
// device 0 and run blocks 0..P-1 on devices 0..P-1; route B's enter at device
// P-1 and run the same blocks on devices P-1..0.  Device d holds block d of
// route A and block P-1-d of route B.  The page leaves the merged order open;
// the library's reading: each route keeps its 1F1B order at each of its stages
// (F^w (B F)^(Mr-w) B^w, w = min(P - stage, Mr)); a device that is free at tick
// T runs an op at the front of either route whose input has arrived by T,
// taking a backward before a forward and, between two ops of one kind, the
// route in which it is the earlier stage (route A when d <= P-1-d); with no
// input arrived it waits for the first.  comm[l] is the latency of the link
// between devices l and l+1 in both directions.  F and B cost at least one
// tick, so whether an input has arrived by T is fixed by the costs alone.
//
// The order depends on the costs, so there is no plan.  One lane per
// (instance, device), a warp holds 32/PMAX instances (lane = device * 32/PMAX
// + instance).  Two phases, both exact:
//   1. each lane on its own tick, deciding only what the rules already fix
//      (the Zero Bubble kernel's scheme: a neighbour's published lower bound
//      on the end of the op a lane waits for proves that its input has not
//      arrived); capped at cap1 steps (8*M + 64 unless the environment
//      variable PPSCHED_DP_PHASE1_STEPS sets it; the results do not depend on
//      it);
//   2. for instances phase 1 left unfinished, the lanes of the instance step
//      through its event ticks together, at most 4*P*M + 1 steps.
//
// Per warp, in shared memory ([row][lane], conflict-free):
//   cost rings    [4 streams][kRing]: F and B costs of route A's block and of
//                 route B's block, copied by cp.async kAheadC microbatches
//                 ahead (a lane consumes at most one op per step, as in the
//                 Zero Bubble kernel)
//   arrival rings [2 routes][2 kinds][kQ]: the arrival tick of the input of
//                 the consumer's op for local microbatch i at row i mod kQ,
//                 written by the producing neighbour.  Under 1F1B a producer
//                 runs at most w <= P ops of a kind ahead of its consumer, so
//                 kQ = PMAX rows never wrap onto an unread one.
#include <cstdlib>

#include "eval_common.cuh"

namespace pps {

template <int PMAX>
struct DpGeom {
    static constexpr int kIPW = 32 / PMAX;  // instances per warp
    static constexpr int kRing = 8;         // cost ring rows per stream
    static constexpr int kAheadC = kRing - 1;
    static constexpr int kQ = PMAX;         // arrival ring rows
    static constexpr int kWords = (4 * kRing + 4 * kQ) * 32;  // per warp
    static constexpr int kWarps = 4;
    static_assert((kRing & (kRing - 1)) == 0 && (kQ & (kQ - 1)) == 0, "rings are indexed by masks");
};

// Route r's next op at a stage with Mr microbatches and warmup w, after nf
// forwards and nb backwards: present, kind, local microbatch.
__device__ __forceinline__ void dp_front(int nf, int nb, int Mr, int w, bool &has, bool &isF, int &i) {
    const int p = nf + nb, q = p - w;
    has = p < 2 * Mr;
    isF = q < 0 || (q < 2 * (Mr - w) && (q & 1));
    i = isF ? nf : nb;
}

// PP_ST_NEG_COST if instance x has a negative cost or comm, PP_ST_ZERO_COST if
// an F or B cost is below 1, else PP_ST_OVERFLOW; read from global memory,
// used only to classify an instance whose flags were raised.
static __device__ __noinline__ int8_t dp_classify(const EvalArgs &a, int64_t x) {
    bool zero = false;
    for (int s = 0; s < a.P; ++s) {
        if (a.comm && s < a.P - 1 && a.comm[x * a.c_inst + (int64_t)s * a.c_bnd] < 0) return PP_ST_NEG_COST;
        for (int g = 0; g < a.M; ++g) {
            const int64_t off = x * a.s_inst + (int64_t)s * a.s_stage + (int64_t)g * a.s_mb;
            const int32_t f = a.cost_f[off], b = a.cost_b[off];
            if (f < 0 || b < 0) return PP_ST_NEG_COST;
            if (f < 1 || b < 1) zero = true;
        }
    }
    return zero ? PP_ST_ZERO_COST : PP_ST_OVERFLOW;
}

template <int PMAX, bool OPS>
__global__ void __launch_bounds__(128) k_eval_dp(const EvalArgs a, int MA, int32_t *peak_out, int cap1) {
    using G = DpGeom<PMAX>;
    extern __shared__ __align__(16) uint32_t dsm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int j = lane % G::kIPW, d = lane / G::kIPW;
    uint32_t *cring = dsm + warp * G::kWords;      // [4][kRing][32]
    uint32_t *aring = cring + 4 * G::kRing * 32;  // [2][2][kQ][32]
    const int64_t x = ((int64_t)blockIdx.x * G::kWarps + warp) * G::kIPW + j;
    const int P = a.P, M = a.M, MB = M - MA;
    const bool dev = x < a.n && d < P;  // this lane simulates a device

    // per-lane constants of the two routes (A, B): block (= stage index on
    // the route), microbatches, warmup, first global microbatch
    const int blkA = d, blkB = P - 1 - d, MB_ = MB;
    const int wA = min(P - d, MA), wB = min(d + 1, MB);
    const bool prefA = d <= P - 1 - d;
    uint32_t cmL = 0, cmR = 0, ncomm = 0;
    if (dev && a.comm) {
        if (d > 0) cmL = (uint32_t)a.comm[x * a.c_inst + (int64_t)(d - 1) * a.c_bnd];
        if (d < P - 1) cmR = (uint32_t)a.comm[x * a.c_inst + (int64_t)d * a.c_bnd];
        ncomm = cmL | cmR;
    }
    // stream q = route * 2 + kind (0 F, 1 B); srcA / srcB: element offset of
    // the route's first microbatch in its block's cost rows
    const int64_t srcA = dev ? x * a.s_inst + (int64_t)blkA * a.s_stage : 0;
    const int64_t srcB = dev ? x * a.s_inst + (int64_t)blkB * a.s_stage + (int64_t)MA * a.s_mb : 0;
    [[maybe_unused]] const int64_t reach = cost_reach(a.n, P, MA + MB_, a.s_inst, a.s_stage, a.s_mb);
    auto fetch = [&](int q, int i) {
        const bool rb = q >= 2;
        if (dev && i < (rb ? MB_ : MA) &&
            PPS_CHECK((rb ? srcB : srcA) + (int64_t)i * a.s_mb < reach, kChkCostRead, (rb ? srcB : srcA) + (int64_t)i * a.s_mb)) {
            const int32_t *base = (q & 1) ? a.cost_b : a.cost_f;
            cp_async4(smem_addr(cring + (q * G::kRing + (i & (G::kRing - 1))) * 32 + lane),
                      base + (rb ? srcB : srcA) + (int64_t)i * a.s_mb, 4);
        }
    };
#pragma unroll 1
    for (int i = 0; i < G::kAheadC; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) fetch(q, i);
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();

    auto ring = [&](int r, int kind, int i) -> uint32_t * {
        return aring + (((r * 2 + kind) * G::kQ) + (i & (G::kQ - 1))) * 32;
    };

    constexpr uint32_t kInf = 0xFFFFFFFFu;
    auto sat = [](uint32_t x, uint32_t y) -> uint32_t {  // x + y, kInf when it does not fit
        const uint32_t z = x + y;
        return z < x ? kInf : z;
    };
    uint32_t tfree = 0, busy = 0, flag = 0, zero = 0;
    int nfA = 0, nbA = 0, nfB = 0, nbB = 0;
    int held = 0, peak = 0;
    // the neighbours' counts: from the left lane its route-A forwards and
    // route-B backwards, from the right lane its route-A backwards and route-B
    // forwards (the producers of this lane's inputs)
    int nfA_L = 0, nbB_L = 0, nbA_R = 0, nfB_R = 0;
    bool done = !dev;

    // Place the front op of route `rb` (0 A, 1 B), of cost c, at tick `t0`:
    // the arrival tick for the consumer neighbour, op times, counts, ledger.
    auto place = [&](bool rb, bool f, int i, uint32_t t0, uint32_t c) {
        const int q = (rb ? 2 : 0) + (f ? 0 : 1);
        const uint32_t e = t0 + c;
        flag |= t0 | c;
        zero |= c == 0 ? 1u : 0u;
        busy += c;
        tfree = e;
        fetch(q, i + G::kAheadC);
        // the consumer: route A forwards go right, backwards left; route B
        // the other way round
        uint32_t *row = ring(rb ? 1 : 0, f ? 0 : 1, i);
        const bool right = rb != f;
        if (right && d + 1 < P) row[lane + G::kIPW] = e + cmR;
        if (!right && d > 0) row[lane - G::kIPW] = e + cmL;
        if constexpr (OPS) {
            const int blk = rb ? blkB : blkA, g = (rb ? MA : 0) + i;
            const int64_t off = x * a.o_inst + ((int64_t)(blk * 2 + (f ? 0 : 1)) * M + g) * a.o_op;
            if (a.op_start) a.op_start[off] = (int32_t)t0;
            if (a.op_end) a.op_end[off] = (int32_t)e;
        }
        nfA += !rb && f;
        nbA += !rb && !f;
        nfB += rb && f;
        nbB += rb && !f;
        held += f ? 1 : -1;
        peak = max(peak, held);
    };
    // The fronts of both routes: present, kind, local microbatch, input known
    // (no producer on another device -- a route's first forward or last
    // backward -- or the producer has placed it), arrival tick if known.
    struct Front { bool h, f, known; int i; uint32_t arr; };
    auto fronts = [&](Front &A, Front &Bf) {
        dp_front(nfA, nbA, MA, wA, A.h, A.f, A.i);
        dp_front(nfB, nbB, MB_, wB, Bf.h, Bf.f, Bf.i);
        const bool firstA = A.f ? blkA == 0 : blkA == P - 1;
        const bool firstB = Bf.f ? blkB == 0 : blkB == P - 1;
        A.known = firstA || (A.f ? nfA_L : nbA_R) > A.i;
        Bf.known = firstB || (Bf.f ? nfB_R : nbB_L) > Bf.i;
        A.arr = firstA ? 0u : ring(0, A.f ? 0 : 1, A.i)[lane];
        Bf.arr = firstB ? 0u : ring(1, Bf.f ? 0 : 1, Bf.i)[lane];
    };
    auto publish_counts = [&]() {
        const uint32_t toR = (uint32_t)nfA | ((uint32_t)nbB << 16);  // read by the right lane
        const uint32_t toL = (uint32_t)nbA | ((uint32_t)nfB << 16);  // read by the left lane
        const uint32_t fromL = __shfl_up_sync(0xFFFFFFFFu, toR, G::kIPW);
        const uint32_t fromR = __shfl_down_sync(0xFFFFFFFFu, toL, G::kIPW);
        nfA_L = (int)(fromL & 0xFFFFu);
        nbB_L = (int)(fromL >> 16);
        nbA_R = (int)(fromR & 0xFFFFu);
        nfB_R = (int)(fromR >> 16);
    };

    // ---- Phase 1: every lane on its own tick t (no op of the lane starts
    // before t).  A lane decides only what the rules already fix at t: a
    // front whose input has arrived by t runs at t when the other front is
    // absent, provably not arrived by t, or would lose the tie-break anyway;
    // when neither front can have arrived by t, t moves to the earliest tick
    // either could arrive.  "Provably not arrived": the producer neighbour
    // publishes after each step a lower bound on the end of its next op of
    // each (route, kind) -- its own t plus the costs its route order puts up
    // to that op (F and B cost at least one tick) -- and a consumer whose
    // input is not placed yet waits for exactly that op.  A lane that waits
    // does so on a neighbour whose t is smaller (the bound exceeds the
    // neighbour's t), so in every step some lane of each unfinished instance
    // places an op or moves its t.  The step count of this phase has no small
    // bound, so it is capped; an instance still unfinished continues in
    // phase 2, which is exact from any state reached here.
    uint32_t t = 0;
    // the neighbours' bounds this lane's inputs depend on (0 until published)
    uint32_t lbFA_L = 0, lbBB_L = 0, lbBA_R = 0, lbFB_R = 0;
    // each route's front and the costs of its next F and B, kept across
    // steps and refreshed when the route places an op (the ring rows of the
    // next ops were copied at least kAheadC - 1 steps ago)
    struct Route { bool h, f, moreF, moreB; int i; uint32_t cF, cB; };
    auto refresh = [&](int r, Route &S) {
        const int nf = r ? nfB : nfA, nb = r ? nbB : nbA, Mr = r ? MB_ : MA;
        dp_front(nf, nb, Mr, r ? wB : wA, S.h, S.f, S.i);
        S.moreF = nf < Mr;
        S.moreB = nb < Mr;
        S.cF = S.moreF ? cring[((2 * r) * G::kRing + (nf & (G::kRing - 1))) * 32 + lane] : 0u;
        S.cB = S.moreB ? cring[((2 * r + 1) * G::kRing + (nb & (G::kRing - 1))) * 32 + lane] : 0u;
    };
    Route RA, RB;
    refresh(0, RA);
    refresh(1, RB);
#pragma unroll 1
    for (int step = 0; step < cap1; ++step) {
        cp_async_wait<G::kAheadC - 2>();
        __syncwarp();
        if (!done) {
            // input known (no producer on another device, or placed), arrival
            const bool firstA = RA.f ? blkA == 0 : blkA == P - 1;
            const bool firstB = RB.f ? blkB == 0 : blkB == P - 1;
            const bool knownA = firstA || (RA.f ? nfA_L : nbA_R) > RA.i;
            const bool knownB = firstB || (RB.f ? nfB_R : nbB_L) > RB.i;
            const uint32_t arrA = firstA ? 0u : ring(0, RA.f ? 0 : 1, RA.i)[lane];
            const uint32_t arrB = firstB ? 0u : ring(1, RB.f ? 0 : 1, RB.i)[lane];
            // earliest tick each front's input can arrive: known, or the bound
            const uint32_t lowA = knownA ? arrA : (RA.f ? sat(lbFA_L, cmL) : sat(lbBA_R, cmR));
            const uint32_t lowB = knownB ? arrB : (RB.f ? sat(lbFB_R, cmR) : sat(lbBB_L, cmL));
            const bool rA = RA.h && knownA && arrA <= t, rB = RB.h && knownB && arrB <= t;
            const bool uA = RA.h && !knownA && lowA <= t, uB = RB.h && !knownB && lowB <= t;
            // route A's front beats route B's whatever B's readiness (and back)
            const bool aWins = (!RA.f && RB.f) || (RA.f == RB.f && prefA);
            int pick = 0;
            if (rA && rB) pick = aWins ? 1 : 2;
            else if (rA && (!uB || aWins)) pick = 1;
            else if (rB && (!uA || !aWins)) pick = 2;
            if (pick) {
                const bool rb = pick == 2;
                Route &S = rb ? RB : RA;
                place(rb, S.f, S.i, t, S.f ? S.cF : S.cB);
                t = tfree;
                refresh(rb ? 1 : 0, S);
            } else if (!rA && !rB && !uA && !uB) {
                t = min(RA.h ? lowA : kInf, RB.h ? lowB : kInf);
            }
        }
        cp_async_commit();
        __syncwarp();
        publish_counts();
        done = !dev || (!RA.h && !RB.h);
        // the bounds on the ends of this lane's next ops of each (route, kind):
        // t plus the costs of the ops its route order puts up to them
        const uint32_t lbFA = RA.moreF ? sat(sat(t, RA.f ? 0u : RA.cB), RA.cF) : kInf;
        const uint32_t lbBA = RA.moreB ? sat(sat(t, RA.f ? RA.cF : 0u), RA.cB) : kInf;
        const uint32_t lbFB = RB.moreF ? sat(sat(t, RB.f ? 0u : RB.cB), RB.cF) : kInf;
        const uint32_t lbBB = RB.moreB ? sat(sat(t, RB.f ? RB.cF : 0u), RB.cB) : kInf;
        lbFA_L = __shfl_up_sync(0xFFFFFFFFu, lbFA, G::kIPW);
        lbBB_L = __shfl_up_sync(0xFFFFFFFFu, lbBB, G::kIPW);
        lbBA_R = __shfl_down_sync(0xFFFFFFFFu, lbBA, G::kIPW);
        lbFB_R = __shfl_down_sync(0xFFFFFFFFu, lbFB, G::kIPW);
        if (__all_sync(0xFFFFFFFFu, done)) break;
    }

    // ---- Phase 2 (instances phase 1 left unfinished): the lanes of an
    // instance step through its event ticks together.  At the instance's tick
    // T every lane free by T takes the op the rules give it at T (an op placed
    // at T ends after T, so no other decision at T depends on it); the next T
    // is the smallest of the busy lanes' free ticks and the known arrivals the
    // free lanes wait for (an arrival not known yet comes after its
    // producer's end, itself a candidate).  It starts at the smallest t of the
    // instance's unfinished lanes: every op that starts before it is placed,
    // and no lane has an input arrived before its own t.  The ticks increase
    // strictly and each is an op's end or an input's arrival, so the phase
    // takes at most 4*P*M + 1 steps.
    bool capped = false;
    if (!__all_sync(0xFFFFFFFFu, done)) {
        uint32_t T = done ? kInf : t;
#pragma unroll
        for (int o = G::kIPW; o < 32; o <<= 1) T = min(T, __shfl_xor_sync(0xFFFFFFFFu, T, o));
        capped = true;
        const int max_steps = 4 * P * M + 2;
#pragma unroll 1
        for (int step = 0; step < max_steps; ++step) {
            cp_async_wait<G::kAheadC - 2>();
            __syncwarp();
            Front A, Bf;
            fronts(A, Bf);
            // ---- decide at T: 0 none, 1 route A, 2 route B
            int pick = 0;
            if (!done && tfree <= T) {
                const bool rA = A.h && A.known && A.arr <= T;
                const bool rB = Bf.h && Bf.known && Bf.arr <= T;
                if (rA && rB) pick = (A.f != Bf.f) ? (A.f ? 2 : 1) : (prefA ? 1 : 2);
                else if (rA) pick = 1;
                else if (rB) pick = 2;
            }
            if (pick) {
                const bool rb = pick == 2;
                const bool f = rb ? Bf.f : A.f;
                const int i = rb ? Bf.i : A.i, q = (rb ? 2 : 0) + (f ? 0 : 1);
                place(rb, f, i, T, cring[(q * G::kRing + (i & (G::kRing - 1))) * 32 + lane]);
            }
            cp_async_commit();
            __syncwarp();
            publish_counts();
            done = !dev || (nfA + nbA == 2 * MA && nfB + nbB == 2 * MB_);
            // ---- the instance's next event tick
            uint32_t nxt = kInf;
            if (!done) {
                if (tfree > T) {
                    nxt = tfree;
                } else {
                    fronts(A, Bf);
                    if (A.h && A.known && A.arr > T) nxt = min(nxt, A.arr);
                    if (Bf.h && Bf.known && Bf.arr > T) nxt = min(nxt, Bf.arr);
                }
            }
#pragma unroll
            for (int o = G::kIPW; o < 32; o <<= 1) nxt = min(nxt, __shfl_xor_sync(0xFFFFFFFFu, nxt, o));
            if (__all_sync(0xFFFFFFFFu, done)) { capped = false; break; }
            if (nxt != kInf) T = nxt;
        }
    }
    cp_async_wait<0>();

    // per-instance reductions over the instance's lanes (as the other
    // evaluators: window = last end tick, idle = window - busy, bubble = total
    // idle over P windows)
    const bool left_over = dev && (nfA + nbA < 2 * MA || nfB + nbB < 2 * MB);
    uint32_t mk = dev ? tfree : 0u, fl = flag, zr = zero, nc = ncomm;
    uint32_t cp = capped && left_over ? 1u : 0u;
#pragma unroll
    for (int o = G::kIPW; o < 32; o <<= 1) {
        mk = max(mk, __shfl_xor_sync(0xFFFFFFFFu, mk, o));
        fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, o);
        zr |= __shfl_xor_sync(0xFFFFFFFFu, zr, o);
        nc |= __shfl_xor_sync(0xFFFFFFFFu, nc, o);
        cp |= __shfl_xor_sync(0xFFFFFFFFu, cp, o);
    }
    fl |= mk;
    const int idle = dev ? (int)(mk - busy) : 0;
    int64_t num = idle;
#pragma unroll
    for (int o = G::kIPW; o < 32; o <<= 1) num += __shfl_xor_sync(0xFFFFFFFFu, num, o);
    if (!dev) return;
    if (a.idle) a.idle[x * P + d] = idle;
    if (peak_out) peak_out[x * P + d] = peak;  // per instance: the order depends on the costs
    if (d == 0) {
        if (a.makespan) a.makespan[x] = (int)mk;
        if (a.bub_num) a.bub_num[x] = num;
        if (a.bub_den) a.bub_den[x] = (int64_t)P * (int)mk;
        if (a.status) {
            int8_t st = PP_ST_OK;
            if (nc >> 31) st = PP_ST_NEG_COST;
            else if ((fl >> 31) || zr || cp) st = dp_classify(a, x);
            a.status[x] = st;
        }
    }
}

namespace {

template <int PMAX, bool OPS>
int launch_dp_t(const EvalArgs &a, int MA, int32_t *peak, int cap1, cudaStream_t st) {
    using G = DpGeom<PMAX>;
    const size_t smem = (size_t)G::kWarps * G::kWords * sizeof(uint32_t);
    const int64_t warps = (a.n + G::kIPW - 1) / G::kIPW;
    const int64_t blocks = (warps + G::kWarps - 1) / G::kWarps;
    if (blocks > 0x7FFFFFFF) return PP_ERR_SIZE;
    k_eval_dp<PMAX, OPS><<<(unsigned)blocks, G::kWarps * 32, smem, st>>>(a, MA, peak, cap1);
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}

template <int PMAX>
int launch_dp_p(const EvalArgs &a, int MA, int32_t *peak, int cap1, bool ops, cudaStream_t st) {
    return ops ? launch_dp_t<PMAX, true>(a, MA, peak, cap1, st) : launch_dp_t<PMAX, false>(a, MA, peak, cap1, st);
}

}  // namespace
}  // namespace pps

extern "C" int pp_sched_eval_dualpipe(int P, int M, int m_a, const int32_t *cost_f, const int32_t *cost_b,
                                      int64_t stride_inst, int64_t stride_stage, int64_t stride_mb,
                                      const int32_t *comm, int64_t comm_stride_inst, int64_t comm_stride_link,
                                      int64_t n_instances, int32_t *makespan, int32_t *idle, int64_t *bub_num,
                                      int64_t *bub_den, int32_t *peak, int32_t *op_start, int32_t *op_end,
                                      int64_t op_stride_inst, int64_t op_stride_op, int8_t *status,
                                      cudaStream_t stream) {
    using namespace pps;
    if (P < 1 || M < 1 || m_a < 0 || m_a > M || n_instances < 0) return PP_ERR_ARG;
    if (P > PP_MAX_P || M > PP_MAX_MV) return PP_ERR_SIZE;
    if (n_instances > 0 && (!cost_f || !cost_b)) return PP_ERR_ARG;
    if (stride_inst < 0 || stride_stage < 0 || stride_mb < 0 || comm_stride_inst < 0 || comm_stride_link < 0)
        return PP_ERR_ARG;
    const bool ops = op_start || op_end;
    if (ops && (op_stride_inst < 0 || op_stride_op < 0)) return PP_ERR_ARG;
    if (n_instances == 0) return PP_OK;
    EvalArgs a{};
    a.R = 0; a.P = P; a.M = M; a.v = 1; a.S = P; a.O = 2 * M; a.nslots = 0;
    a.cost_f = cost_f; a.cost_b = cost_b;
    a.s_inst = stride_inst; a.s_stage = stride_stage; a.s_mb = stride_mb;
    a.comm = comm; a.c_inst = comm_stride_inst; a.c_bnd = comm_stride_link;
    a.n = n_instances; a.inst_begin = 0;
    a.makespan = makespan; a.idle = idle; a.bub_num = bub_num; a.bub_den = bub_den; a.status = status;
    a.op_start = op_start; a.op_end = op_end; a.o_inst = op_stride_inst; a.o_op = op_stride_op;
    // the first phase's step cap (results do not depend on it; see the kernel)
    int cap1 = 8 * M + 64;
    if (const char *env = std::getenv("PPSCHED_DP_PHASE1_STEPS")) {
        const long v = std::strtol(env, nullptr, 10);
        if (v >= 0 && v <= (1L << 30)) cap1 = (int)v;
    }
    switch (pmax_for(P)) {
        case 4: return launch_dp_p<4>(a, m_a, peak, cap1, ops, stream);
        case 8: return launch_dp_p<8>(a, m_a, peak, cap1, ops, stream);
        case 16: return launch_dp_p<16>(a, m_a, peak, cap1, ops, stream);
        default: return PP_ERR_INTERNAL;
    }
}
