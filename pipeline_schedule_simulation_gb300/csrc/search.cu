// search.cu -- candidate contiguous partitions of L layers into P stages,
// scored under 1F1B on the GPU (pp_sched_partition_search).
//
// The pages balance stages by splitting the layer sequence into contiguous
// ranges from profiled costs ("Pipeline parallelism: from GPipe to 1F1B and
// Zero Bubble", PipeDream and GPipe sections; M040 §05: uneven stages make the
// fast stage wait; lpnh: 80 layers into 8 stages).  Here each thread draws one
// seeded candidate split, sums its stages' costs and activation bytes from
// prefix sums, rejects it if a stage would hold more activation bytes than the
// cap, and otherwise evaluates the 1F1B schedule with the register recurrence
// (stage costs are constant over microbatches, so they live in registers).
// The best (makespan, candidate) pair is reduced with warp shuffles and one
// 64-bit atomicMin per warp into the caller's best_idx word, which a one-thread
// kernel then turns into the index, makespan and cut positions.  When only the
// winner is wanted, a candidate whose 1F1B makespan lower bound exceeds the
// word's current best is not evaluated, and an exhaustive range first scores
// every kProbe-th split so that the bound is tight from the start.
#include "internal.cuh"
#include "search_common.cuh"

namespace pps {

namespace {

constexpr int kMaxL = 256;

struct SearchArgs {
    const uint64_t *rw;    // 1F1B plan: per-round kind words
    const uint4 *seg;      // and segments
    int nseg;
    int R, P, M, L;
    const int32_t *ltf, *ltb;
    const int64_t *lact;
    int32_t comm;
    int64_t cap;
    uint64_t seed;
    int64_t begin, n;
    int64_t step;          // candidate ci of a launch is call index ci * step
    uint64_t ncomb;        // C(L-1, P-1)
    int32_t peak[PP_MAX_P];
    int32_t *all_mk;
    unsigned long long *key;  // the caller's best_idx word, used as the reduction cell
};

// Shared tables: prefix sums of layer costs and bytes, and C(n, i) for
// n < L, i < P, computed with the multiplicative formula in 128-bit-safe steps.
struct Tables {
    int64_t pre_tf[kMaxL + 1], pre_tb[kMaxL + 1], pre_act[kMaxL + 1];
    uint64_t C[kMaxL][PP_MAX_P];  // C[n][i]; saturates at ~0
};

__device__ void build_tables(const SearchArgs &a, Tables &t) {
    const int tid = threadIdx.x;
    for (int e = tid; e < a.L * a.P; e += blockDim.x) {
        const int n = e / a.P, i = e % a.P;
        t.C[n][i] = binom_u64(n, i);
    }
    if (tid == 0) {
        int64_t f = 0, b = 0, c = 0;
        t.pre_tf[0] = t.pre_tb[0] = t.pre_act[0] = 0;
        for (int l = 0; l < a.L; ++l) {
            f += a.ltf[l]; b += a.ltb[l]; c += a.lact[l];
            t.pre_tf[l + 1] = f; t.pre_tb[l + 1] = b; t.pre_act[l + 1] = c;
        }
    }
    __syncthreads();
}

// Colex unranking: the largest x with C(x, i) <= r for i = K..1, subtracting
// as it goes; writes the first layer of stages 0..P (first[0] = 0, first[P] = L).
template <int PMAX>
__device__ __forceinline__ void unrank(const SearchArgs &a, const Tables &t, uint64_t r, int (&first)[PMAX + 1]) {
    const int K = a.P - 1;
    int hi = a.L - 2;  // positions 0..L-2
#pragma unroll
    for (int i = PMAX - 1; i >= 1; --i) {
        if (i <= K) {
            int c = hi;
            while (c >= i && t.C[c][i] > r) --c;
            r -= t.C[c][i];
            first[i] = c + 1;
            hi = c - 1;
        }
    }
    first[0] = 0;
#pragma unroll
    for (int i = 1; i <= PMAX; ++i) if (i >= a.P) first[i] = a.L;
}

// 1F1B max-plus recurrence of one candidate.  Stage costs are the same for
// every microbatch, so they stay in registers; the plan's rounds are walked
// segment by segment: the steady state alternates static rounds in which the
// even devices run F and the odd ones B (or the reverse), the warmup and
// cooldown rounds run from their kind words.  The input of an op is the
// latest result of its kind on the neighbouring device (the plan checks that
// this holds for 1F1B).  `acc` collects the sign bits of every end tick and
// arrival (an int32 overflow or a negative stage sum sets it).
template <int PMAX>
struct SState {
    int fr[PMAX], rf[PMAX], rb[PMAX];
    uint32_t acc;
};

template <int PMAX>
__device__ __forceinline__ void s_op_f(SState<PMAX> &S, int k, int arr, int c, int cm) {
    const int st = max(S.fr[k], arr);
    const int en = (int)((uint32_t)st + (uint32_t)c);
    S.fr[k] = en;
    S.acc |= (uint32_t)en | (uint32_t)arr;
    S.rf[k] = (int)((uint32_t)en + (uint32_t)cm);
}

template <int PMAX>
__device__ __forceinline__ void s_op_b(SState<PMAX> &S, int k, int arr, int c, int cm) {
    const int st = max(S.fr[k], arr);
    const int en = (int)((uint32_t)st + (uint32_t)c);
    S.fr[k] = en;
    S.acc |= (uint32_t)en | (uint32_t)arr;
    S.rb[k] = (int)((uint32_t)en + (uint32_t)cm);
}

// Alternating round: F on devices of parity FP, B on the others.  An F reads
// rf of a device that runs B this round and a B reads rb of a device that runs
// F, so no input is overwritten within the round.
template <int PMAX, int FP>
__device__ __forceinline__ void s_alt(SState<PMAX> &S, const int (&cf)[PMAX], const int (&cb)[PMAX], int comm) {
#pragma unroll
    for (int k = 0; k < PMAX; ++k) {
        if ((k & 1) == FP) s_op_f<PMAX>(S, k, k > 0 ? S.rf[k > 0 ? k - 1 : 0] : 0, cf[k], k < PMAX - 1 ? comm : 0);
        else s_op_b<PMAX>(S, k, k < PMAX - 1 ? S.rb[k < PMAX - 1 ? k + 1 : 0] : 0, cb[k], k > 0 ? comm : 0);
    }
}

// Any round, from its kind word (2 bits per device).
template <int PMAX>
__device__ __forceinline__ void s_round(SState<PMAX> &S, uint32_t kinds, const int (&cf)[PMAX],
                                        const int (&cb)[PMAX], int P, int comm) {
    int rf0[PMAX], rb0[PMAX];
#pragma unroll
    for (int k = 0; k < PMAX; ++k) { rf0[k] = S.rf[k]; rb0[k] = S.rb[k]; }
#pragma unroll
    for (int k = 0; k < PMAX; ++k) {
        const uint32_t kind = (kinds >> (2 * k)) & 3u;
        if (kind == kFwd) s_op_f<PMAX>(S, k, k > 0 ? rf0[k > 0 ? k - 1 : 0] : 0, cf[k], k < P - 1 ? comm : 0);
        else if (kind == kBwd) s_op_b<PMAX>(S, k, k < PMAX - 1 ? rb0[k < PMAX - 1 ? k + 1 : 0] : 0, cb[k], k > 0 ? comm : 0);
    }
}

template <int PMAX>
__device__ __forceinline__ int eval_1f1b(const SearchArgs &a, SState<PMAX> &S, const int (&cf)[PMAX],
                                         const int (&cb)[PMAX]) {
#pragma unroll
    for (int k = 0; k < PMAX; ++k) { S.fr[k] = 0; S.rf[k] = 0; S.rb[k] = 0; }
#pragma unroll 1
    for (int si = 0; si < a.nseg; ++si) {
        const uint4 sg = __ldg(a.seg + si);
        int r = (int)sg.y;
        const int r1 = (int)sg.z;
        if (sg.x == kSegAltA || sg.x == kSegAltB) {
            const bool a_first = sg.x == kSegAltA;
#pragma unroll 1
            for (; r + 1 < r1; r += 2) {
                if (a_first) { s_alt<PMAX, 0>(S, cf, cb, a.comm); s_alt<PMAX, 1>(S, cf, cb, a.comm); }
                else { s_alt<PMAX, 1>(S, cf, cb, a.comm); s_alt<PMAX, 0>(S, cf, cb, a.comm); }
            }
            if (r < r1) {
                if (a_first) s_alt<PMAX, 0>(S, cf, cb, a.comm);
                else s_alt<PMAX, 1>(S, cf, cb, a.comm);
            }
        } else {
#pragma unroll 1
            for (; r < r1; ++r) s_round<PMAX>(S, rw_kinds(__ldg(a.rw + r)), cf, cb, a.P, a.comm);
        }
    }
    int mk = 0;
#pragma unroll
    for (int k = 0; k < PMAX; ++k) mk = max(mk, S.fr[k]);
    return mk;
}

// The candidate's rank: a seeded draw (SplitMix64 of seed + index, mod the
// number of splits) or, for the exhaustive search, the index itself.
template <bool EXH>
__device__ __forceinline__ uint64_t cand_rank(const SearchArgs &a, int64_t ci) {
    if constexpr (EXH) return (uint64_t)(a.begin + ci * a.step);
    return splitmix64(a.seed + (uint64_t)(a.begin + ci * a.step)) % a.ncomb;
}

template <int PMAX, bool EXH>
__global__ void __launch_bounds__(256) k_search(const SearchArgs a) {
    __shared__ Tables t;
    build_tables(a, t);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int lane = threadIdx.x & 31;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < a.n; base += stride) {
        const int64_t ci = base + threadIdx.x;  // index within this call
        const bool live = ci < a.n;
        int mk = -1;
        if (live) {
            int first[PMAX + 1];
            unrank<PMAX>(a, t, cand_rank<EXH>(a, ci), first);
            int cf[PMAX], cb[PMAX];
            bool ok = true;
            // (checked build: the split points increase strictly from 0 to L)
#pragma unroll
            for (int k = 0; k < PMAX; ++k)
                if (k < a.P)
                    ok = ok && PPS_CHECK(first[k] >= 0 && first[k] < first[k + 1] && first[k + 1] <= a.L &&
                                             (k + 1 < a.P || first[k + 1] == a.L),
                                         kChkSearchSplit, first[k + 1]);
            if (!ok) {
#pragma unroll
                for (int k = 0; k <= PMAX; ++k) first[k] = 0;
            }
            uint32_t big = 0;
#pragma unroll
            for (int k = 0; k < PMAX; ++k) {
                cf[k] = 0; cb[k] = 0;
                if (k < a.P) {
                    const int64_t sf = t.pre_tf[first[k + 1]] - t.pre_tf[first[k]];
                    const int64_t sb = t.pre_tb[first[k + 1]] - t.pre_tb[first[k]];
                    const int64_t sa = t.pre_act[first[k + 1]] - t.pre_act[first[k]];
                    if ((int64_t)a.peak[k] * sa > a.cap) ok = false;
                    if (sf < 0 || sb < 0 || sf > 0x7FFFFFFF || sb > 0x7FFFFFFF) big = 0x80000000u;
                    cf[k] = (int)sf; cb[k] = (int)sb;
                }
            }
            if (ok && !a.all_mk) {
                // Only the winner is wanted: skip a candidate that provably
                // ends after the best makespan found so far.  Stage k runs its
                // M forwards and M backwards one at a time; its first forward
                // starts after microbatch 0 crossed stages 0..k-1 and their
                // boundaries, and its last backward's gradient still has to
                // cross them back, so every 1F1B makespan (costs >= 0) is at
                // least max_k [ sum_{j<k} (f_j + b_j) + 2k comm + M (f_k + b_k) ].
                // A candidate equal to the best is still evaluated (ties go to
                // the lower index), so the argmin is exact.  A stage sum beyond
                // int32 (big) makes the candidate unselectable either way.
                int64_t pre = 0, lb = 0;
#pragma unroll
                for (int k = 0; k < PMAX; ++k)
                    if (k < a.P) {
                        const int64_t w = (int64_t)cf[k] + cb[k];
                        lb = max(lb, pre + (int64_t)a.M * w);
                        pre += w + 2 * (int64_t)a.comm;
                    }
                const unsigned long long best = *reinterpret_cast<volatile unsigned long long *>(a.key);
                if (lb > (int64_t)(best >> 32)) ok = false;
            }
            if (ok) {
                SState<PMAX> S;
                S.acc = big | (uint32_t)a.comm;
                mk = eval_1f1b<PMAX>(a, S, cf, cb);
                if (S.acc >> 31) mk = -2;
            }
            if (a.all_mk) a.all_mk[ci] = mk;
        }
        unsigned long long key = ~0ull;
        if (live && mk >= 0) key = ((unsigned long long)(uint32_t)mk << 32) | (uint32_t)(ci * a.step);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
            key = other < key ? other : key;
        }
        if (lane == 0 && key != ~0ull) atomicMin(a.key, key);
    }
}

template <int PMAX, bool EXH>
__global__ void k_search_finish(const SearchArgs a, int64_t *best_idx, int32_t *best_mk, int32_t *best_cuts) {
    __shared__ Tables t;
    build_tables(a, t);
    if (threadIdx.x != 0) return;
    const unsigned long long key = *a.key;
    if (key == ~0ull) {
        *best_idx = -1;
        if (best_mk) *best_mk = -1;
        if (best_cuts) for (int k = 0; k + 1 < a.P; ++k) best_cuts[k] = -1;
        return;
    }
    const int64_t ci = (int64_t)(key & 0xFFFFFFFFull);
    const int mk = (int)(key >> 32);
    if (best_cuts) {
        int first[PMAX + 1];
        unrank<PMAX>(a, t, cand_rank<EXH>(a, ci), first);
        for (int k = 1; k < a.P; ++k) best_cuts[k - 1] = first[k];
    }
    if (best_mk) *best_mk = mk;
    *best_idx = a.begin + ci;
}

template <int PMAX, bool EXH>
int run_search(SearchArgs &a, int64_t *best_idx, int32_t *best_mk, int32_t *best_cuts, cudaStream_t st) {
    int dev = 0, sms = 0, per_sm = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    PPS_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    PPS_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_search<PMAX, EXH>, 256, 0));
    if (per_sm < 1) per_sm = 1;
    int64_t want = (a.n + 255) / 256;
    int64_t grid = (int64_t)sms * per_sm;
    if (want < grid) grid = want;
    if (grid < 1) grid = 1;
    // Only the winner wanted from an exhaustive range: first score every
    // kProbe-th split, so that the main pass prunes against a near-best
    // makespan from its start (colex order puts the balanced splits far into
    // the range).  Both passes reduce into the same word; the probe's splits
    // are scored again by the main pass, so the result is unchanged.
    constexpr int64_t kProbe = 1024;
    if (EXH && !a.all_mk && a.n >= 64 * kProbe) {
        SearchArgs pa = a;
        pa.step = kProbe;
        pa.n = (a.n + kProbe - 1) / kProbe;
        const int64_t pgrid = std::min<int64_t>((int64_t)sms * per_sm, (pa.n + 255) / 256);
        k_search<PMAX, EXH><<<(unsigned)pgrid, 256, 0, st>>>(pa);
    }
    if (a.n > 0) k_search<PMAX, EXH><<<(unsigned)grid, 256, 0, st>>>(a);
    k_search_finish<PMAX, EXH><<<1, 64, 0, st>>>(a, best_idx, best_mk, best_cuts);
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}

}  // namespace

}  // namespace pps

namespace pps {
namespace {

int search_entry(const int32_t *layer_tf, const int32_t *layer_tb, const int64_t *layer_act, int L, int P, int M,
                 int32_t comm, int64_t act_cap, uint64_t seed, bool exhaustive, int64_t begin, int64_t n,
                 int64_t *best_idx, int32_t *best_makespan, int32_t *best_cuts, int32_t *all_makespan,
                 cudaStream_t stream) {
    if (!layer_tf || !layer_tb || !layer_act || !best_idx) return PP_ERR_ARG;
    if (P < 1 || M < 1 || L < P || n < 0 || begin < 0 || comm < 0) return PP_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(best_idx) & 7) != 0) return PP_ERR_ARG;
    if (P > PP_MAX_P || L > kMaxL || M > PP_MAX_MV || n >= (int64_t)1 << 32) return PP_ERR_SIZE;
    const uint64_t ncomb = binom_u64(L - 1, P - 1);
    if (ncomb == ~0ull || ncomb == 0) return PP_ERR_SIZE;
    if (exhaustive && (uint64_t)begin + (uint64_t)n > ncomb) return PP_ERR_ARG;
    pp_plan *plan = nullptr;
    int rc = cached_plan(PP_1F1B, P, M, 1, stream, &plan);
    if (rc) return rc;
    if (!plan->reg_ok) return PP_ERR_INTERNAL;
    SearchArgs a;
    a.rw = plan->d_rw; a.seg = plan->d_seg; a.nseg = plan->nseg; a.R = plan->R; a.P = P; a.M = M; a.L = L;
    a.ltf = layer_tf; a.ltb = layer_tb; a.lact = layer_act;
    a.comm = comm; a.cap = act_cap; a.seed = seed; a.begin = begin; a.n = n; a.ncomb = ncomb; a.step = 1;
    for (int k = 0; k < PP_MAX_P; ++k) a.peak[k] = k < P ? plan->h_peak[k] : 0;
    a.all_mk = all_makespan;
    a.key = reinterpret_cast<unsigned long long *>(best_idx);
    PPS_CUDA_TRY(cudaMemsetAsync(best_idx, 0xFF, sizeof(int64_t), stream));
    switch (plan->pmax) {
        case 4: return exhaustive ? run_search<4, true>(a, best_idx, best_makespan, best_cuts, stream)
                                  : run_search<4, false>(a, best_idx, best_makespan, best_cuts, stream);
        case 8: return exhaustive ? run_search<8, true>(a, best_idx, best_makespan, best_cuts, stream)
                                  : run_search<8, false>(a, best_idx, best_makespan, best_cuts, stream);
        case 16: return exhaustive ? run_search<16, true>(a, best_idx, best_makespan, best_cuts, stream)
                                   : run_search<16, false>(a, best_idx, best_makespan, best_cuts, stream);
        default: return PP_ERR_INTERNAL;
    }
}

}  // namespace
}  // namespace pps

extern "C" int pp_sched_partition_search(const int32_t *layer_tf, const int32_t *layer_tb,
                                         const int64_t *layer_act, int L, int P, int M, int32_t comm,
                                         int64_t act_cap, uint64_t seed, int64_t cand_begin,
                                         int64_t n_cand, int64_t *best_idx, int32_t *best_makespan,
                                         int32_t *best_cuts, int32_t *all_makespan, cudaStream_t stream) {
    return pps::search_entry(layer_tf, layer_tb, layer_act, L, P, M, comm, act_cap, seed, false, cand_begin,
                             n_cand, best_idx, best_makespan, best_cuts, all_makespan, stream);
}

extern "C" int pp_sched_partition_search_ranks(const int32_t *layer_tf, const int32_t *layer_tb,
                                               const int64_t *layer_act, int L, int P, int M, int32_t comm,
                                               int64_t act_cap, int64_t rank_begin, int64_t n_ranks,
                                               int64_t *best_rank, int32_t *best_makespan, int32_t *best_cuts,
                                               int32_t *all_makespan, cudaStream_t stream) {
    return pps::search_entry(layer_tf, layer_tb, layer_act, L, P, M, comm, act_cap, 0, true, rank_begin, n_ranks,
                             best_rank, best_makespan, best_cuts, all_makespan, stream);
}
