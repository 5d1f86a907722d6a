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
// + instance).  The lanes of an instance step through its event ticks
// together: in a step every lane that is free at the instance's tick T takes
// the op the rules give it at T (an op placed at T ends after T, so no other
// decision at T depends on it), then the instance's next tick is the smallest
// of the busy lanes' free ticks and the known arrivals the free lanes wait for
// (an arrival not known yet comes after its producer ends, which is itself a
// candidate).  The ticks increase strictly and each is an op's end or an
// input's arrival, so an instance takes at most 4*P*M + 1 steps.
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
__global__ void __launch_bounds__(128) k_eval_dp(const EvalArgs a, int MA, int32_t *peak_out) {
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
    auto fetch = [&](int q, int i) {
        const bool rb = q >= 2;
        if (dev && i < (rb ? MB_ : MA)) {
            const int32_t *base = (q & 1) ? a.cost_b : a.cost_f;
            cp_async4(smem_addr(cring + (q * G::kRing + i % G::kRing) * 32 + lane),
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

    uint32_t T = 0, tfree = 0, busy = 0, flag = 0, zero = 0;
    int nfA = 0, nbA = 0, nfB = 0, nbB = 0;
    int held = 0, peak = 0;
    // the neighbours' counts: from the left lane its route-A forwards and
    // route-B backwards, from the right lane its route-A backwards and route-B
    // forwards (the producers of this lane's inputs)
    int nfA_L = 0, nbB_L = 0, nbA_R = 0, nfB_R = 0;
    const int max_steps = 4 * P * M + 2;
    bool capped = true;
#pragma unroll 1
    for (int step = 0; step < max_steps; ++step) {
        cp_async_wait<G::kAheadC - 2>();
        __syncwarp();
        // ---- the fronts of both routes: present, kind, local microbatch,
        // input known, arrival tick
        bool hA, fA, hB, fB;
        int iA, iB;
        dp_front(nfA, nbA, MA, wA, hA, fA, iA);
        dp_front(nfB, nbB, MB_, wB, hB, fB, iB);
        // no producer on another device: a route's first forward, last backward
        const bool firstA = fA ? blkA == 0 : blkA == P - 1;
        const bool firstB = fB ? blkB == 0 : blkB == P - 1;
        const bool knownA = firstA || (fA ? nfA_L : nbA_R) > iA;
        const bool knownB = firstB || (fB ? nfB_R : nbB_L) > iB;
        const uint32_t arrA = firstA ? 0u : ring(0, fA ? 0 : 1, iA)[lane];
        const uint32_t arrB = firstB ? 0u : ring(1, fB ? 0 : 1, iB)[lane];
        // ---- decide at T: 0 none, 1 route A, 2 route B
        int pick = 0;
        if (dev && tfree <= T) {
            const bool rA = hA && knownA && arrA <= T;
            const bool rB = hB && knownB && arrB <= T;
            if (rA && rB) pick = (fA != fB) ? (fA ? 2 : 1) : (prefA ? 1 : 2);
            else if (rA) pick = 1;
            else if (rB) pick = 2;
        }
        // ---- place (predicated on pick)
        if (pick) {
            const bool rb = pick == 2;
            const bool f = rb ? fB : fA;
            const int i = rb ? iB : iA, q = (rb ? 2 : 0) + (f ? 0 : 1);
            const uint32_t c = cring[(q * G::kRing + i % G::kRing) * 32 + lane];
            const uint32_t e = T + c;
            flag |= T | c;
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
                if (a.op_start) a.op_start[off] = (int32_t)T;
                if (a.op_end) a.op_end[off] = (int32_t)e;
            }
            nfA += !rb && f;
            nbA += !rb && !f;
            nfB += rb && f;
            nbB += rb && !f;
            held += f ? 1 : -1;
            peak = max(peak, held);
        }
        cp_async_commit();
        __syncwarp();
        // ---- publish the counts the neighbours' inputs depend on
        const uint32_t toR = (uint32_t)nfA | ((uint32_t)nbB << 16);  // read by the right lane
        const uint32_t toL = (uint32_t)nbA | ((uint32_t)nfB << 16);  // read by the left lane
        const uint32_t fromL = __shfl_up_sync(0xFFFFFFFFu, toR, G::kIPW);
        const uint32_t fromR = __shfl_down_sync(0xFFFFFFFFu, toL, G::kIPW);
        nfA_L = (int)(fromL & 0xFFFFu);
        nbB_L = (int)(fromL >> 16);
        nbA_R = (int)(fromR & 0xFFFFu);
        nfB_R = (int)(fromR >> 16);
        // ---- the instance's next event tick
        const bool done = !dev || (nfA + nbA == 2 * MA && nfB + nbB == 2 * MB_);
        uint32_t nxt = 0xFFFFFFFFu;
        if (!done) {
            if (tfree > T) {
                nxt = tfree;
            } else {
                dp_front(nfA, nbA, MA, wA, hA, fA, iA);
                dp_front(nfB, nbB, MB_, wB, hB, fB, iB);
                const bool fstA = fA ? blkA == 0 : blkA == P - 1;
                const bool fstB = fB ? blkB == 0 : blkB == P - 1;
                if (hA && !fstA && (fA ? nfA_L : nbA_R) > iA) {
                    const uint32_t t = ring(0, fA ? 0 : 1, iA)[lane];
                    if (t > T) nxt = min(nxt, t);
                }
                if (hB && !fstB && (fB ? nfB_R : nbB_L) > iB) {
                    const uint32_t t = ring(1, fB ? 0 : 1, iB)[lane];
                    if (t > T) nxt = min(nxt, t);
                }
            }
        }
#pragma unroll
        for (int o = G::kIPW; o < 32; o <<= 1) nxt = min(nxt, __shfl_xor_sync(0xFFFFFFFFu, nxt, o));
        if (__all_sync(0xFFFFFFFFu, done)) { capped = false; break; }
        if (nxt != 0xFFFFFFFFu) T = nxt;
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
int launch_dp_t(const EvalArgs &a, int MA, int32_t *peak, cudaStream_t st) {
    using G = DpGeom<PMAX>;
    const size_t smem = (size_t)G::kWarps * G::kWords * sizeof(uint32_t);
    const int64_t warps = (a.n + G::kIPW - 1) / G::kIPW;
    const int64_t blocks = (warps + G::kWarps - 1) / G::kWarps;
    if (blocks > 0x7FFFFFFF) return PP_ERR_SIZE;
    k_eval_dp<PMAX, OPS><<<(unsigned)blocks, G::kWarps * 32, smem, st>>>(a, MA, peak);
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}

template <int PMAX>
int launch_dp_p(const EvalArgs &a, int MA, int32_t *peak, bool ops, cudaStream_t st) {
    return ops ? launch_dp_t<PMAX, true>(a, MA, peak, st) : launch_dp_t<PMAX, false>(a, MA, peak, st);
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
    switch (pmax_for(P)) {
        case 4: return launch_dp_p<4>(a, m_a, peak, ops, stream);
        case 8: return launch_dp_p<8>(a, m_a, peak, ops, stream);
        case 16: return launch_dp_p<16>(a, m_a, peak, ops, stream);
        default: return PP_ERR_INTERNAL;
    }
}
