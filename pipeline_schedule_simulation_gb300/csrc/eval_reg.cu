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
#include <utility>

#include "eval_common.cuh"

namespace pps {

// Overflow and negative-cost detection.  All true ticks are >= 0.  Ticks are
// carried as uint32 and compared unsigned, and every op ORs its start tick and
// its cost into one sticky word; the final makespan is ORed in too.  If no cost
// is negative and every true tick is below 2^31, every value is exact and no
// sign bit is ever set.  Otherwise take the first op, in evaluation order,
// whose true end reaches 2^31: its inputs are exact and below 2^31 (an arrival
// is an exact end plus a comm below 2^31, so below 2^32), hence its start is
// exact; if the start reaches 2^31 it is flagged, else its end is exact and
// becomes the free tick of the device, so the next op's start (an unsigned max
// with it) or the final makespan carries the sign bit.  A negative cost carries
// it directly.  So the word's sign bit is set exactly when the instance is
// flagged; which flag is decided by re-reading the costs (rare path).

// Register state of one instance: per device its free tick, the arrival tick
// of its latest forward result at device k+1 (rf) and of its latest backward
// result at device k-1 (rb), its busy ticks, and (per-op output only) its op
// counter.  cF[k] is the comm of boundary k|k+1; a backward result of device k
// crosses boundary k-1, whose comm is cF[k-1].
template <int PMAX>
struct RegState {
    uint32_t fr[PMAX], rf[PMAX], rb[PMAX], busy[PMAX], cF[PMAX];
    int cnt[PMAX];
    uint32_t flag;
};

// One op on device K with input arrival `arr` and cost `c`.
template <int PMAX, bool OPS, bool FWD, int K>
__device__ __forceinline__ void reg_op(RegState<PMAX> &S, uint32_t arr, uint32_t c, const EvalArgs &a,
                                       int64_t x, bool live) {
    const uint32_t st = max(S.fr[K], arr);
    const uint32_t en = st + c;
    S.fr[K] = en;
    S.busy[K] += c;
    S.flag |= st | c;
    if constexpr (FWD) S.rf[K] = en + S.cF[K];
    else S.rb[K] = en + (K > 0 ? S.cF[K > 0 ? K - 1 : 0] : 0u);
    if constexpr (OPS) {
        if (live) {
            const int64_t off = x * a.o_inst + ((int64_t)K * a.O + S.cnt[K]) * a.o_op;
            if (a.op_start) a.op_start[off] = (int)st;
            if (a.op_end) a.op_end[off] = (int)en;
        }
        ++S.cnt[K];
    }
}

// Shared-memory words of the per-CTA tables: loader table [R][PMAX] (padded
// to 16 bytes), round words [R] (padded to 16 bytes), segments [nseg].
template <int PMAX>
__host__ __device__ inline int lt_smem_words(int R, int nseg) {
    return ((R * PMAX + 3) & ~3) + 2 * ((R + 1) & ~1) + 4 * nseg;
}

template <int PMAX, int K>
__device__ __forceinline__ uint32_t in_fwd(const RegState<PMAX> &S) { return K > 0 ? S.rf[K > 0 ? K - 1 : 0] : 0u; }
template <int PMAX, int K>
__device__ __forceinline__ uint32_t in_bwd(const RegState<PMAX> &S) {
    return K < PMAX - 1 ? S.rb[K < PMAX - 1 ? K + 1 : 0] : 0u;
}

// Pattern round bodies.  In the alternating patterns a device's input comes
// from a neighbour that runs the other kind (or nothing) this round, so it is
// unchanged by the round; in all-F (all-B) rounds devices run from the last
// (first) so each reads its input before the neighbour overwrites it.  MASKED
// bodies run only the devices whose bit is set.
template <int PMAX, bool OPS, bool MASKED, bool EVEN_FWD, int K = 0>
__device__ __forceinline__ void round_alt(RegState<PMAX> &S, uint32_t mask, const int32_t *slice, int lane,
                                          const EvalArgs &a, int64_t x, bool live) {
    if constexpr (K < PMAX) {
        if (!MASKED || ((mask >> K) & 1u)) {
            const uint32_t c = (uint32_t)slice[K * 32 + lane];
            constexpr bool fwd = ((K & 1) == 0) == EVEN_FWD;
            if constexpr (fwd) reg_op<PMAX, OPS, true, K>(S, in_fwd<PMAX, K>(S), c, a, x, live);
            else reg_op<PMAX, OPS, false, K>(S, in_bwd<PMAX, K>(S), c, a, x, live);
        }
        round_alt<PMAX, OPS, MASKED, EVEN_FWD, K + 1>(S, mask, slice, lane, a, x, live);
    }
}

template <int PMAX, bool OPS, bool MASKED, int K = PMAX - 1>
__device__ __forceinline__ void round_all_f(RegState<PMAX> &S, uint32_t mask, const int32_t *slice, int lane,
                                            const EvalArgs &a, int64_t x, bool live) {
    if constexpr (K >= 0) {
        if (!MASKED || ((mask >> K) & 1u))
            reg_op<PMAX, OPS, true, K>(S, in_fwd<PMAX, K>(S), (uint32_t)slice[K * 32 + lane], a, x, live);
        round_all_f<PMAX, OPS, MASKED, K - 1>(S, mask, slice, lane, a, x, live);
    }
}

template <int PMAX, bool OPS, bool MASKED, int K = 0>
__device__ __forceinline__ void round_all_b(RegState<PMAX> &S, uint32_t mask, const int32_t *slice, int lane,
                                            const EvalArgs &a, int64_t x, bool live) {
    if constexpr (K < PMAX) {
        if (!MASKED || ((mask >> K) & 1u))
            reg_op<PMAX, OPS, false, K>(S, in_bwd<PMAX, K>(S), (uint32_t)slice[K * 32 + lane], a, x, live);
        round_all_b<PMAX, OPS, MASKED, K + 1>(S, mask, slice, lane, a, x, live);
    }
}

// Any other round: inputs are read as of the start of the round, then each
// device runs its op (or none) by its 2-bit kind.
template <int PMAX, bool OPS>
__device__ __forceinline__ void round_generic(RegState<PMAX> &S, uint32_t kinds, const int32_t *slice, int lane,
                                              const EvalArgs &a, int64_t x, bool live) {
    uint32_t inF[PMAX], inB[PMAX];
#pragma unroll
    for (int k = 0; k < PMAX; ++k) {
        inF[k] = k > 0 ? S.rf[k > 0 ? k - 1 : 0] : 0u;
        inB[k] = k < PMAX - 1 ? S.rb[k < PMAX - 1 ? k + 1 : 0] : 0u;
    }
    [&]<int... K>(std::integer_sequence<int, K...>) {
        ([&] {
            const uint32_t kind = (kinds >> (2 * K)) & 3u;
            const uint32_t c = (uint32_t)slice[K * 32 + lane];
            if (kind == kFwd) reg_op<PMAX, OPS, true, K>(S, inF[K], c, a, x, live);
            else if (kind == kBwd) reg_op<PMAX, OPS, false, K>(S, inB[K], c, a, x, live);
        }(), ...);
    }(std::make_integer_sequence<int, PMAX>{});
}

template <int PMAX, bool OPS>
__device__ __forceinline__ void run_round(RegState<PMAX> &S, uint64_t w, const int32_t *slice, int lane,
                                          const EvalArgs &a, int64_t x, bool live) {
    const uint32_t m = rw_mask(w);
    switch (rw_pattern(w)) {
        case kPatAltA: round_alt<PMAX, OPS, false, true>(S, m, slice, lane, a, x, live); break;
        case kPatAltB: round_alt<PMAX, OPS, false, false>(S, m, slice, lane, a, x, live); break;
        case kPatAllF: round_all_f<PMAX, OPS, false>(S, m, slice, lane, a, x, live); break;
        case kPatAllB: round_all_b<PMAX, OPS, false>(S, m, slice, lane, a, x, live); break;
        case kPatMasked + kPatAltA: round_alt<PMAX, OPS, true, true>(S, m, slice, lane, a, x, live); break;
        case kPatMasked + kPatAltB: round_alt<PMAX, OPS, true, false>(S, m, slice, lane, a, x, live); break;
        case kPatMasked + kPatAllF: round_all_f<PMAX, OPS, true>(S, m, slice, lane, a, x, live); break;
        case kPatMasked + kPatAllB: round_all_b<PMAX, OPS, true>(S, m, slice, lane, a, x, live); break;
        default: round_generic<PMAX, OPS>(S, rw_kinds(w), slice, lane, a, x, live); break;
    }
}

// LT: the vector loader runs from the per-CTA offset table.  Dynamic shared
// memory then holds the table, the round words and the segment list (so no
// global load sits on the warmup / cooldown path), then one ring per warp.
//
// The kernel walks the plan's segments.  Alternating and all-F / all-B
// segments are tight loops over static round bodies (two rounds per iteration
// in the alternating case), so the instance's state stays in the same
// registers across iterations; warmup and cooldown rounds are dispatched one
// at a time by their round word.  Copies run D = kAhead2 rounds ahead.
template <int PMAX, bool VEC, bool OPS, bool LT>
__global__ void __launch_bounds__(128) k_eval_reg(const EvalArgs a) {
    using RG = Ring<PMAX>;
    constexpr int D = RG::kAhead2;
    extern __shared__ __align__(16) int32_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int lt_words = LT ? lt_smem_words<PMAX>(a.R, a.nseg) : 0;
    uint32_t *lt = reinterpret_cast<uint32_t *>(smem);
    const uint64_t *rws = a.rw;
    const uint4 *segs = a.seg;
    if constexpr (LT) {
        const int tw = (a.R * PMAX + 3) & ~3;
        uint64_t *rw_s = reinterpret_cast<uint64_t *>(smem + tw);
        uint4 *seg_s = reinterpret_cast<uint4 *>(smem + tw + 2 * ((a.R + 1) & ~1));
        stage_words(a.seg, seg_s, a.nseg);
        stage_words(reinterpret_cast<const uint4 *>(a.rw), reinterpret_cast<uint4 *>(rw_s), (a.R + 1) / 2);
        build_load_table<PMAX>(a, lt);
        __syncthreads();
        rws = rw_s;
        segs = seg_s;
    }
    int32_t *ring = smem + lt_words + warp * RG::kWords;
    const int64_t inst0 = a.inst_begin + ((int64_t)blockIdx.x * nwarps + warp) * 32;
    if (inst0 >= a.n) return;  // warp-uniform, after the block barrier
    const int64_t x = inst0 + lane;
    const bool live = x < a.n;

    RegState<PMAX> S;
    uint32_t negc = 0;
#pragma unroll
    for (int k = 0; k < PMAX; ++k) {
        int c = 0;
        if (a.comm && live && k < a.P - 1) c = a.comm[x * a.c_inst + (int64_t)k * a.c_bnd];
        negc |= (uint32_t)c;
        S.cF[k] = (uint32_t)c;
        S.fr[k] = 0; S.rf[k] = 0; S.rb[k] = 0; S.busy[k] = 0; S.cnt[k] = 0;
    }
    S.flag = 0;

    // loader state
    const int g = lane & 7;
    const int64_t x0 = inst0 + 4 * g;
    const int64_t left = a.n - x0;
    const uint32_t bytes_in = left <= 0 ? 0u : (left >= 4 ? 16u : (uint32_t)left * 4u);
    const int32_t *fbase = a.cost_f + (bytes_in ? x0 : 0);
    const int32_t *bbase = a.cost_b + (bytes_in ? x0 : 0);
    const int R = a.R;
    auto issue = [&](int rl) {
        if (rl < R) {
            if constexpr (LT) {
                load_round_lt<PMAX>(lt, rl, ring, fbase, bbase, bytes_in, lane);
            } else {
                LoadDesc<PMAX, VEC> ld;
                fetch_load_desc<PMAX, VEC>(a, rl, lane, ld);
                load_round<PMAX, VEC>(a, rl, ld, ring, inst0, lane);
            }
        }
        cp_async_commit();
    };
    auto slice = [&](int r) { return ring + (r % RG::kSlices) * (PMAX * 32); };
    // one round: its copies D ahead, wait for it, run `body`
    auto step1 = [&](int r, auto &&body) {
        issue(r + D);
        cp_async_wait<D>();
        __syncwarp();
        body(slice(r));
        __syncwarp();
    };
    // two rounds: copies for both, then wait for both
    auto step2 = [&](int r, auto &&body0, auto &&body1) {
        issue(r + D);
        issue(r + D + 1);
        cp_async_wait<D>();
        __syncwarp();
        body0(slice(r));
        body1(slice(r + 1));
        __syncwarp();
    };
    auto altA = [&](const int32_t *sl) { round_alt<PMAX, OPS, false, true>(S, 0u, sl, lane, a, x, live); };
    auto altB = [&](const int32_t *sl) { round_alt<PMAX, OPS, false, false>(S, 0u, sl, lane, a, x, live); };
    auto allF = [&](const int32_t *sl) { round_all_f<PMAX, OPS, false>(S, 0u, sl, lane, a, x, live); };
    auto allB = [&](const int32_t *sl) { round_all_b<PMAX, OPS, false>(S, 0u, sl, lane, a, x, live); };

#pragma unroll 1
    for (int q = 0; q < D; ++q) issue(q);
#pragma unroll 1
    for (int si = 0; si < a.nseg; ++si) {
        const uint4 sg = segs[si];
        int r = (int)sg.y;
        const int r1 = (int)sg.z;
        switch (sg.x) {
            case kSegAltA:
#pragma unroll 1
                for (; r + 1 < r1; r += 2) step2(r, altA, altB);
                if (r < r1) step1(r, altA);
                break;
            case kSegAltB:
#pragma unroll 1
                for (; r + 1 < r1; r += 2) step2(r, altB, altA);
                if (r < r1) step1(r, altB);
                break;
            case kSegAllF:
#pragma unroll 1
                for (; r < r1; ++r) step1(r, allF);
                break;
            case kSegAllB:
#pragma unroll 1
                for (; r < r1; ++r) step1(r, allB);
                break;
            default: {
                const uint64_t w = rws[r];
                step1(r, [&](const int32_t *sl) { run_round<PMAX, OPS>(S, w, sl, lane, a, x, live); });
                break;
            }
        }
    }
    cp_async_wait<0>();
    if (live) write_results_u<PMAX>(a, x, S.fr, S.busy, S.flag, (negc >> 31) != 0);
}

template <int PMAX, bool VEC, bool OPS, bool LT>
static int launch_reg_t(const EvalArgs &a, int64_t begin, int64_t end, cudaStream_t st) {
    constexpr int kWarps = 4;
    if (end <= begin) return PP_OK;
    const size_t lt_bytes = LT ? (size_t)lt_smem_words<PMAX>(a.R, a.nseg) * sizeof(uint32_t) : 0;
    const size_t smem = lt_bytes + (size_t)kWarps * Ring<PMAX>::kWords * sizeof(int32_t);
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    static bool attr_set[64] = {};
    if (dev < 64 && !attr_set[dev]) {
        PPS_CUDA_TRY(cudaFuncSetAttribute(k_eval_reg<PMAX, VEC, OPS, LT>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024));
        attr_set[dev] = true;
    }
    const int64_t warps = (end - begin + 31) / 32;
    const int64_t blocks = (warps + kWarps - 1) / kWarps;
    if (blocks > 0x7FFFFFFF) return PP_ERR_SIZE;
    EvalArgs b = a;
    b.inst_begin = begin;
    b.n = end;
    k_eval_reg<PMAX, VEC, OPS, LT><<<(unsigned)blocks, kWarps * 32, smem, st>>>(b);
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}

template <int PMAX, bool OPS>
static int launch_reg_o(const EvalArgs &a, bool vec, bool lt, cudaStream_t st) {
    if (lt) return launch_reg_t<PMAX, true, OPS, true>(a, 0, a.n, st);
    if (vec) return launch_reg_t<PMAX, true, OPS, false>(a, 0, a.n, st);
    return launch_reg_t<PMAX, false, OPS, false>(a, 0, a.n, st);
}

// Largest loader table kept in shared memory (words); bigger plans use the
// in-loop address computation.
constexpr int kMaxLtWords = 8192;

template <int PMAX>
static int launch_reg_p(const EvalArgs &a, bool vec, bool ops, cudaStream_t st) {
    // the table path needs 16-byte aligned rows and offsets below 2^30
    const bool lt = vec && (int64_t)lt_smem_words<PMAX>(a.R, a.nseg) <= kMaxLtWords &&
                    (int64_t)(a.S - 1) * a.s_stage + (int64_t)(a.M - 1) * a.s_mb < ((int64_t)1 << 30);
    return ops ? launch_reg_o<PMAX, true>(a, vec, lt, st) : launch_reg_o<PMAX, false>(a, vec, lt, st);
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
    a.desc = plan->d_desc; a.desc2 = plan->d_desc2; a.rw = plan->d_rw;
    a.seg = plan->d_seg; a.nseg = plan->nseg;
    a.R = plan->R; a.P = P; a.M = M; a.v = v; a.S = plan->S; a.O = plan->O; a.nslots = plan->nslots;
    a.cost_f = cost_f; a.cost_b = cost_b;
    a.s_inst = stride_inst; a.s_stage = stride_stage; a.s_mb = stride_mb;
    a.comm = comm; a.c_inst = comm_stride_inst; a.c_bnd = comm_stride_bnd;
    a.n = n_instances;
    a.inst_begin = 0;
    a.makespan = makespan; a.idle = idle; a.bub_num = bub_num; a.bub_den = bub_den; a.status = status;
    a.op_start = op_start; a.op_end = op_end; a.o_inst = op_stride_inst; a.o_op = op_stride_op;
    const bool vec = stride_inst == 1 && (reinterpret_cast<uintptr_t>(cost_f) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(cost_b) & 15) == 0 && stride_stage % 4 == 0 &&
                     stride_mb % 4 == 0 &&
                     (int64_t)(plan->S - 1) * stride_stage + (int64_t)(M - 1) * stride_mb < ((int64_t)1 << 31);
    const bool ops = op_start || op_end;
    if (plan->reg_ok) return launch_eval_reg(plan, a, vec, ops, stream);
    return launch_eval_slot(plan, a, vec, ops, stream);
}
