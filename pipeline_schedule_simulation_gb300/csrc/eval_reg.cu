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
#include <atomic>
#include <type_traits>
#include <utility>

#include "eval_common.cuh"

namespace pps {

#ifndef PPS_REG_NI
#define PPS_REG_NI 1
#endif
// Instances per thread of the table-driven register evaluator.
constexpr int kRegNI = PPS_REG_NI;

// Words of the kernel tables in front of the round words (the loader table,
// padded to 16 bytes); the microbatch-shared kernels skip them.
__host__ __device__ inline int reg_mbz_table_skip(int R, int pmax) { return (R * pmax + 3) & ~3; }

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

// Register state of the NI instances a thread evaluates: per instance and
// device its free tick, the arrival tick of its latest forward result at
// device k+1 (rf) and of its latest backward result at device k-1 (rb), its
// busy ticks, and the comm cF[k] of boundary k|k+1 (a backward result of
// device k crosses boundary k-1, whose comm is cF[k-1]); per device the op
// counter of the per-op output (the same for every instance).
template <int PMAX, int NI>
struct RegState {
    uint32_t fr[NI][PMAX], rf[NI][PMAX], rb[NI][PMAX], busy[NI][PMAX], cF[NI][PMAX];
    int cnt[PMAX];
    uint32_t flag[NI];
};

// Where a thread's instances are: instance i of the thread is x[i].
template <int NI>
struct Lanes {
    int lane;
    int64_t x[NI];
    bool live[NI];
};

// One op on device K for every instance of the thread; its cost for instance
// i is slice[(K*NI + i)*32 + lane].
template <int PMAX, int NI, bool OPS, bool FWD, int K>
__device__ __forceinline__ void reg_op(RegState<PMAX, NI> &S, const uint32_t (&arr)[NI], const int32_t *slice,
                                       const EvalArgs &a, const Lanes<NI> &L) {
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const uint32_t c = (uint32_t)slice[(K * NI + i) * 32 + L.lane];
        const uint32_t st = max(S.fr[i][K], arr[i]);
        const uint32_t en = st + c;
        S.fr[i][K] = en;
        S.busy[i][K] += c;
        S.flag[i] |= st | c;
        if constexpr (FWD) S.rf[i][K] = en + S.cF[i][K];
        else S.rb[i][K] = en + (K > 0 ? S.cF[i][K > 0 ? K - 1 : 0] : 0u);
        if constexpr (OPS) {
            if (L.live[i]) {
                const int64_t off = L.x[i] * a.o_inst + ((int64_t)K * a.O + S.cnt[K]) * a.o_op;
                if (a.op_start) a.op_start[off] = (int)st;
                if (a.op_end) a.op_end[off] = (int)en;
            }
        }
    }
    if constexpr (OPS) ++S.cnt[K];
}

template <int PMAX, int NI, int K>
__device__ __forceinline__ void in_fwd(const RegState<PMAX, NI> &S, uint32_t (&arr)[NI]) {
#pragma unroll
    for (int i = 0; i < NI; ++i) arr[i] = K > 0 ? S.rf[i][K > 0 ? K - 1 : 0] : 0u;
}
template <int PMAX, int NI, int K>
__device__ __forceinline__ void in_bwd(const RegState<PMAX, NI> &S, uint32_t (&arr)[NI]) {
#pragma unroll
    for (int i = 0; i < NI; ++i) arr[i] = K < PMAX - 1 ? S.rb[i][K < PMAX - 1 ? K + 1 : 0] : 0u;
}

// Pattern round bodies.  In the alternating patterns a device's input comes
// from a neighbour that runs the other kind (or nothing) this round, so it is
// unchanged by the round; in all-F (all-B) rounds devices run from the last
// (first) so each reads its input before the neighbour overwrites it.  MASKED
// bodies run only the devices whose bit is set.
template <int PMAX, int NI, bool OPS, bool MASKED, bool EVEN_FWD, int K = 0>
__device__ __forceinline__ void round_alt(RegState<PMAX, NI> &S, uint32_t mask, const int32_t *slice,
                                          const EvalArgs &a, const Lanes<NI> &L) {
    if constexpr (K < PMAX) {
        if (!MASKED || ((mask >> K) & 1u)) {
            uint32_t arr[NI];
            constexpr bool fwd = ((K & 1) == 0) == EVEN_FWD;
            if constexpr (fwd) {
                in_fwd<PMAX, NI, K>(S, arr);
                reg_op<PMAX, NI, OPS, true, K>(S, arr, slice, a, L);
            } else {
                in_bwd<PMAX, NI, K>(S, arr);
                reg_op<PMAX, NI, OPS, false, K>(S, arr, slice, a, L);
            }
        }
        round_alt<PMAX, NI, OPS, MASKED, EVEN_FWD, K + 1>(S, mask, slice, a, L);
    }
}

template <int PMAX, int NI, bool OPS, bool MASKED, int K = PMAX - 1>
__device__ __forceinline__ void round_all_f(RegState<PMAX, NI> &S, uint32_t mask, const int32_t *slice,
                                            const EvalArgs &a, const Lanes<NI> &L) {
    if constexpr (K >= 0) {
        if (!MASKED || ((mask >> K) & 1u)) {
            uint32_t arr[NI];
            in_fwd<PMAX, NI, K>(S, arr);
            reg_op<PMAX, NI, OPS, true, K>(S, arr, slice, a, L);
        }
        round_all_f<PMAX, NI, OPS, MASKED, K - 1>(S, mask, slice, a, L);
    }
}

template <int PMAX, int NI, bool OPS, bool MASKED, int K = 0>
__device__ __forceinline__ void round_all_b(RegState<PMAX, NI> &S, uint32_t mask, const int32_t *slice,
                                            const EvalArgs &a, const Lanes<NI> &L) {
    if constexpr (K < PMAX) {
        if (!MASKED || ((mask >> K) & 1u)) {
            uint32_t arr[NI];
            in_bwd<PMAX, NI, K>(S, arr);
            reg_op<PMAX, NI, OPS, false, K>(S, arr, slice, a, L);
        }
        round_all_b<PMAX, NI, OPS, MASKED, K + 1>(S, mask, slice, a, L);
    }
}

// Any other round: inputs are read as of the start of the round, then each
// device runs its op (or none) by its 2-bit kind.
template <int PMAX, int NI, bool OPS>
__device__ __forceinline__ void round_generic(RegState<PMAX, NI> &S, uint32_t kinds, const int32_t *slice,
                                              const EvalArgs &a, const Lanes<NI> &L) {
    uint32_t inF[PMAX][NI], inB[PMAX][NI];
#pragma unroll
    for (int k = 0; k < PMAX; ++k)
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            inF[k][i] = k > 0 ? S.rf[i][k > 0 ? k - 1 : 0] : 0u;
            inB[k][i] = k < PMAX - 1 ? S.rb[i][k < PMAX - 1 ? k + 1 : 0] : 0u;
        }
    [&]<int... K>(std::integer_sequence<int, K...>) {
        ([&] {
            const uint32_t kind = (kinds >> (2 * K)) & 3u;
            if (kind == kFwd) reg_op<PMAX, NI, OPS, true, K>(S, inF[K], slice, a, L);
            else if (kind == kBwd) reg_op<PMAX, NI, OPS, false, K>(S, inB[K], slice, a, L);
        }(), ...);
    }(std::make_integer_sequence<int, PMAX>{});
}

template <int PMAX, int NI, bool OPS>
__device__ __forceinline__ void run_round(RegState<PMAX, NI> &S, uint64_t w, const int32_t *slice,
                                          const EvalArgs &a, const Lanes<NI> &L) {
    const uint32_t m = rw_mask(w);
    switch (rw_pattern(w)) {
        case kPatAltA: round_alt<PMAX, NI, OPS, false, true>(S, m, slice, a, L); break;
        case kPatAltB: round_alt<PMAX, NI, OPS, false, false>(S, m, slice, a, L); break;
        case kPatAllF: round_all_f<PMAX, NI, OPS, false>(S, m, slice, a, L); break;
        case kPatAllB: round_all_b<PMAX, NI, OPS, false>(S, m, slice, a, L); break;
        case kPatMasked + kPatAltA: round_alt<PMAX, NI, OPS, true, true>(S, m, slice, a, L); break;
        case kPatMasked + kPatAltB: round_alt<PMAX, NI, OPS, true, false>(S, m, slice, a, L); break;
        case kPatMasked + kPatAllF: round_all_f<PMAX, NI, OPS, true>(S, m, slice, a, L); break;
        case kPatMasked + kPatAllB: round_all_b<PMAX, NI, OPS, true>(S, m, slice, a, L); break;
        default: round_generic<PMAX, NI, OPS>(S, rw_kinds(w), slice, a, L); break;
    }
}

// The register evaluator.  A warp covers 32*NI instances (NI per thread).
// LT: the vector loader runs from the per-CTA offset table (NI may be 2);
// otherwise the loader computes addresses from the plan's descriptors (NI 1).
// Dynamic shared memory holds, for LT, the loader table, the round words and
// the segment list (so no global load sits on the warmup / cooldown path),
// then one ring of round slices per warp.
//
// The kernel walks the plan's segments.  Alternating and all-F / all-B
// segments are tight loops over static round bodies (two rounds per iteration
// in the alternating case), so the instances' state stays in the same
// registers across iterations; warmup and cooldown rounds are dispatched one
// at a time by their round word.  Copies run D = kAhead2 rounds ahead, one
// cp.async group per round.  A step waits for its rounds' groups, then issues
// the copies D rounds ahead before it runs their bodies: those copies land in
// the slices of the two rounds before the step, which every lane finished
// reading before the step's warp barrier, so they are in flight while the
// bodies compute.  The table loader reads its entries two rounds before it
// issues them, so no shared-memory load sits on the issue path.
template <int PMAX, int NI, bool VEC, bool OPS, bool LT>
__global__ void __maxnreg__(PMAX == 16 ? 168 : 96) k_eval_reg(const EvalArgs a) {
    // Programmatic dependent launch: the next evaluation on the stream may
    // start its blocks as this grid's blocks retire; it copies the plan's
    // tables (complete before either launch) and waits below for this grid's
    // end before it touches any input or output.  Without the launch
    // attribute both instructions do nothing.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    static_assert(NI == 1 || LT, "two instances per thread need the table loader");
    using RG = Ring<PMAX, NI>;
    constexpr int D = RG::kAhead2;
    extern __shared__ __align__(16) int32_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int lt_words = LT ? a.ktab_words : 0;
    uint32_t *lt = reinterpret_cast<uint32_t *>(smem);
    const uint64_t *rws = a.rw;
    const uint4 *segs = a.seg;
    if constexpr (LT) {
        // the block's copy of the precomputed tables, in flight while the
        // comm values load below
        for (int i = threadIdx.x; i < a.ktab_words / 4; i += blockDim.x)
            cp_async16(smem_addr(smem + 4 * i), a.ktab + i, 16u);
        cp_async_commit();
        const int tw = (a.R * PMAX + 3) & ~3;
        rws = reinterpret_cast<const uint64_t *>(smem + tw);
        segs = reinterpret_cast<const uint4 *>(smem + tw + 2 * ((a.R + 1) & ~1));
    }
    int32_t *ring = smem + lt_words + warp * RG::kWords;
    int64_t task = (int64_t)blockIdx.x * nwarps + warp;
    bool has_task = true;
    if (a.tasks > 0) {
        const int64_t t0 = (int64_t)blockIdx.x * a.tasks / gridDim.x;
        const int64_t t1 = ((int64_t)blockIdx.x + 1) * a.tasks / gridDim.x;
        task = t0 + warp;
        has_task = task < t1;
    }
    const int64_t inst0 = has_task ? a.inst_begin + task * (32 * NI) : a.n;
    Lanes<NI> L;
    L.lane = lane;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        L.x[i] = inst0 + 32 * i + lane;
        L.live[i] = L.x[i] < a.n;
    }

    RegState<PMAX, NI> S;
    uint32_t negc[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        S.flag[i] = 0;
#pragma unroll
        for (int k = 0; k < PMAX; ++k) {
            S.fr[i][k] = 0; S.rf[i][k] = 0; S.rb[i][k] = 0; S.busy[i][k] = 0;
        }
    }
    // the comm values; loaded once the first rounds' cost copies are in
    // flight, so their latency hides behind the copies'
    auto load_comm = [&]() {
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            negc[i] = 0;
#pragma unroll
            for (int k = 0; k < PMAX; ++k) {
                int c = 0;
                if (a.comm && L.live[i] && k < a.P - 1) c = a.comm[L.x[i] * a.c_inst + (int64_t)k * a.c_bnd];
                negc[i] |= (uint32_t)c;
                S.cF[i][k] = (uint32_t)c;
            }
        }
    };
#pragma unroll
    for (int k = 0; k < PMAX; ++k) S.cnt[k] = 0;
    if constexpr (LT) {
        cp_async_wait<0>();
        __syncthreads();
    }
    // the previous grid on the stream has finished and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    copy_peak(a);
    if (inst0 >= a.n) return;  // warp-uniform, after the block barrier

    // loader state: lane copies 16 bytes (4 instances) at instance offset 4g
    // of its row; a row of the warp's 32*NI instances takes 8*NI lanes
    const int g = lane % (8 * NI);
    const int64_t x0 = inst0 + 4 * g;
    const int64_t left = a.n - x0;
    const uint32_t bytes_in = left <= 0 ? 0u : (left >= 4 ? 16u : (uint32_t)left * 4u);
    const int64_t xoff = bytes_in ? x0 : 0;
    const int32_t *fbase = a.cost_f + xoff;
    const int32_t *bbase = a.cost_b + xoff;
    [[maybe_unused]] const int64_t reach = cost_reach(a.n, a.S, a.M, a.s_inst, a.s_stage, a.s_mb);
    const int R = a.R;
    constexpr uint32_t kSliceWords = PMAX * NI * 32;
    // shared address of this lane's first 16-byte chunk in slice 0 (table loader)
    const uint32_t dst_lane = smem_addr(ring) + (uint32_t)(((lane / (8 * NI)) * NI * 32 + 4 * g) * 4);
    // the table loader's entries for the next two rounds it issues; the walk
    // with `full` set (every instance of the warp exists) copies whole 16-byte
    // chunks, the other (the last warp of a ragged batch) partial ones
    constexpr int kRPL = PMAX * NI / 4;  // table entries a lane reads per round
    uint32_t eq0[kRPL], eq1[kRPL];
    auto ent = [&](int q, uint32_t (&e)[kRPL]) {
        const uint32_t *row = lt + min(q, R - 1) * PMAX + lane / (8 * NI);
#pragma unroll
        for (int i = 0; i < kRPL; ++i) e[i] = row[(32 / (8 * NI)) * i];
    };
    if constexpr (LT) { ent(0, eq0); ent(1, eq1); }
    auto issue = [&](int rl, auto full) {
        if (rl < R) {
            if constexpr (LT) {
                if constexpr (decltype(full)::value)
                    load_round_lt_q<PMAX, NI>(eq0, dst_lane + ((uint32_t)rl & (RG::kSlices - 1)) * kSliceWords * 4,
                                              fbase, bbase, xoff, reach);
                else
                    load_round_lt<PMAX, NI>(lt, rl, ring, fbase, bbase, bytes_in, lane, xoff, reach);
            } else {
                LoadDesc<PMAX, VEC> ld;
                fetch_load_desc<PMAX, VEC>(a, rl, lane, ld);
                load_round<PMAX, VEC>(a, rl, ld, ring, inst0, lane);
            }
        }
        cp_async_commit();
        if constexpr (LT && decltype(full)::value) {
#pragma unroll
            for (int i = 0; i < kRPL; ++i) eq0[i] = eq1[i];
            ent(rl + 2, eq1);
        }
    };
    auto slice = [&](int r) { return ring + ((uint32_t)r & (RG::kSlices - 1)) * kSliceWords; };
    auto altA = [&](const int32_t *sl) { round_alt<PMAX, NI, OPS, false, true>(S, 0u, sl, a, L); };
    auto altB = [&](const int32_t *sl) { round_alt<PMAX, NI, OPS, false, false>(S, 0u, sl, a, L); };
    auto allF = [&](const int32_t *sl) { round_all_f<PMAX, NI, OPS, false>(S, 0u, sl, a, L); };
    auto allB = [&](const int32_t *sl) { round_all_b<PMAX, NI, OPS, false>(S, 0u, sl, a, L); };

    auto walk = [&](auto full) {
        // one round: its copies D ahead, wait for it, run `body`
        auto step1 = [&](int r, auto &&body) {
            cp_async_wait<D - 1>();
            __syncwarp();
            issue(r + D, full);
            body(slice(r));
        };
        auto step2 = [&](int r, auto &&body0, auto &&body1) {
            cp_async_wait<D - 2>();
            __syncwarp();
            issue(r + D, full);
            issue(r + D + 1, full);
            body0(slice(r));
            body1(slice(r + 1));
        };
#pragma unroll 1
        for (int q = 0; q < D; ++q) issue(q, full);
        load_comm();
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
                    step1(r, [&](const int32_t *sl) { run_round<PMAX, NI, OPS>(S, w, sl, a, L); });
                    break;
                }
            }
        }
    };
    if (LT && inst0 + 32 * NI <= a.n) walk(std::true_type{});
    else walk(std::false_type{});
    cp_async_wait<0>();
    __syncwarp();  // the ring is free: stage the idle block through it
#pragma unroll
    for (int i = 0; i < NI; ++i)
        write_results_warp<PMAX>(a, inst0 + 32 * i, lane, S.fr[i], S.busy[i], S.flag[i], (negc[i] >> 31) != 0,
                                 ring);
}

// The register evaluator for costs shared by every microbatch (stride_mb ==
// 0, e.g. per-stage costs): an op's cost depends only on its device and
// kind, so there is nothing to load per round.  Each lane writes its
// instance's costs once into four static round slices, one per round pattern
// (alternating A and B, all-F, all-B), in the same [device][lane] layout the
// round bodies read; a round that follows no pattern gets its slice from its
// kind word.  No cost ring, no loader, no waits.
// The body takes the CTA's index within its problem (`bid`), so the fused
// kernel over many problems runs it too.
template <int PMAX, bool OPS>
__device__ __forceinline__ void reg_mbz_body(const EvalArgs &a, int64_t bid) {
    copy_peak(a, bid);
    constexpr int kSl = PMAX * 32;  // words per slice
    extern __shared__ __align__(16) int32_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    // only the round words and segments of the kernel tables: the loader
    // table in front of them serves per-microbatch costs
    const int tw = reg_mbz_table_skip(a.R, PMAX);
    const int words = a.ktab_words - tw;
    for (int i = threadIdx.x; i < words / 4; i += blockDim.x)
        cp_async16(smem_addr(smem + 4 * i), a.ktab + tw / 4 + i, 16u);
    cp_async_commit();
    const uint64_t *rws = reinterpret_cast<const uint64_t *>(smem);
    const uint4 *segs = reinterpret_cast<const uint4 *>(smem + 2 * ((a.R + 1) & ~1));
    int32_t *sl_alt_a = smem + words + warp * 5 * kSl;
    int32_t *sl_alt_b = sl_alt_a + kSl, *sl_f = sl_alt_b + kSl, *sl_b = sl_f + kSl, *sl_gen = sl_b + kSl;
    const int64_t inst0 = a.inst_begin + (bid * nwarps + warp) * 32;
    Lanes<1> L;
    L.lane = lane;
    L.x[0] = inst0 + lane;
    L.live[0] = L.x[0] < a.n;
    RegState<PMAX, 1> S;
    uint32_t negc = 0;
    S.flag[0] = 0;
#pragma unroll
    for (int k = 0; k < PMAX; ++k) {
        int c = 0, f = 0, b = 0;
        if (L.live[0] && k < a.P) {
            if (a.comm && k < a.P - 1) c = a.comm[L.x[0] * a.c_inst + (int64_t)k * a.c_bnd];
            f = a.cost_f[L.x[0] * a.s_inst + (int64_t)k * a.s_stage];
            b = a.cost_b[L.x[0] * a.s_inst + (int64_t)k * a.s_stage];
        }
        negc |= (uint32_t)c;
        S.cF[0][k] = (uint32_t)c;
        S.fr[0][k] = 0; S.rf[0][k] = 0; S.rb[0][k] = 0; S.busy[0][k] = 0;
        S.cnt[k] = 0;
        sl_alt_a[k * 32 + lane] = (k & 1) ? b : f;
        sl_alt_b[k * 32 + lane] = (k & 1) ? f : b;
        sl_f[k * 32 + lane] = f;
        sl_b[k * 32 + lane] = b;
    }
    cp_async_wait<0>();
    __syncthreads();
    if (inst0 >= a.n) return;  // warp-uniform, after the block barrier

    // a lane reads only its own column of a slice, so no warp barrier is needed
    auto round_w = [&](uint64_t w) {
        const int32_t *sl;
        switch (rw_pattern(w)) {
            case kPatAltA: case kPatMasked + kPatAltA: sl = sl_alt_a; break;
            case kPatAltB: case kPatMasked + kPatAltB: sl = sl_alt_b; break;
            case kPatAllF: case kPatMasked + kPatAllF: sl = sl_f; break;
            case kPatAllB: case kPatMasked + kPatAllB: sl = sl_b; break;
            default: {
                const uint32_t kinds = rw_kinds(w);
#pragma unroll
                for (int k = 0; k < PMAX; ++k)
                    sl_gen[k * 32 + lane] = sl_f[(((kinds >> (2 * k)) & 3u) == kBwd ? kSl : 0) + k * 32 + lane];
                sl = sl_gen;
            }
        }
        run_round<PMAX, 1, OPS>(S, w, sl, a, L);
    };
#pragma unroll 1
    for (int si = 0; si < a.nseg; ++si) {
        const uint4 sg = segs[si];
        int r = (int)sg.y;
        const int r1 = (int)sg.z;
        switch (sg.x) {
            case kSegAltA:
            case kSegAltB: {
                bool a_next = sg.x == kSegAltA;
#pragma unroll 1
                for (; r + 1 < r1; r += 2) {
                    if (a_next) {
                        round_alt<PMAX, 1, OPS, false, true>(S, 0u, sl_alt_a, a, L);
                        round_alt<PMAX, 1, OPS, false, false>(S, 0u, sl_alt_b, a, L);
                    } else {
                        round_alt<PMAX, 1, OPS, false, false>(S, 0u, sl_alt_b, a, L);
                        round_alt<PMAX, 1, OPS, false, true>(S, 0u, sl_alt_a, a, L);
                    }
                }
                if (r < r1) {
                    if (a_next) round_alt<PMAX, 1, OPS, false, true>(S, 0u, sl_alt_a, a, L);
                    else round_alt<PMAX, 1, OPS, false, false>(S, 0u, sl_alt_b, a, L);
                }
                break;
            }
            case kSegAllF:
#pragma unroll 1
                for (; r < r1; ++r) round_all_f<PMAX, 1, OPS, false>(S, 0u, sl_f, a, L);
                break;
            case kSegAllB:
#pragma unroll 1
                for (; r < r1; ++r) round_all_b<PMAX, 1, OPS, false>(S, 0u, sl_b, a, L);
                break;
            default:
                round_w(rws[r]);
                break;
        }
    }
    __syncwarp();  // the slices are free: stage the idle block through them
    write_results_warp<PMAX>(a, inst0, lane, S.fr[0], S.busy[0], S.flag[0], (negc >> 31) != 0, sl_alt_a);
}

template <int PMAX, bool OPS>
__global__ void __launch_bounds__(128) k_eval_reg_mbz(const EvalArgs a) {
    reg_mbz_body<PMAX, OPS>(a, blockIdx.x);
}

// Many problems in one launch: CTA c runs CTA c - block_begin of its problem.
template <int PMAX>
__global__ void __launch_bounds__(128) k_eval_reg_mbz_many(const ManyJob *jobs, int njobs) {
    const int j = many_job_of(jobs, njobs, blockIdx.x);
    const EvalArgs &a = jobs[j].a;  // read in place: uniform per CTA, cached
    reg_mbz_body<PMAX, false>(a, (int64_t)blockIdx.x - jobs[j].block_begin);
}

template <int PMAX, bool OPS>
static int launch_reg_mbz(const EvalArgs &a, cudaStream_t st) {
    constexpr int kWarps = 4;
    const size_t smem = (size_t)(a.ktab_words - reg_mbz_table_skip(a.R, PMAX)) * sizeof(uint32_t) +
                        (size_t)kWarps * 5 * PMAX * 32 * sizeof(int32_t);
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    static std::atomic<bool> attr_set[64];  // per device, set once (idempotent)
    if (dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
        PPS_CUDA_TRY(cudaFuncSetAttribute(k_eval_reg_mbz<PMAX, OPS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          160 * 1024));
        attr_set[dev].store(true, std::memory_order_release);
    }
    const int64_t warps = (a.n + 31) / 32;
    const int64_t blocks = (warps + kWarps - 1) / kWarps;
    if (blocks > 0x7FFFFFFF) return PP_ERR_SIZE;
    k_eval_reg_mbz<PMAX, OPS><<<(unsigned)blocks, kWarps * 32, smem, st>>>(a);
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}

// Launch `kern` on `st`, as a programmatic dependent launch when `pdl` (the
// kernel waits for the previous grid before it reads inputs or writes
// outputs; its tables must be complete before the launch).
template <typename Kern>
static cudaError_t launch_pdl(Kern kern, unsigned grid, unsigned block, size_t smem, cudaStream_t st, bool pdl,
                              const EvalArgs &b) {
    if (!pdl) {
        kern<<<grid, block, smem, st>>>(b);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, b);
}

template <int PMAX, int NI, bool VEC, bool OPS, bool LT>
static int launch_reg_t(const EvalArgs &a, int64_t begin, int64_t end, cudaStream_t st, bool pdl = false) {
    // two-instance warps hold twice the ring: use two warps per block so the
    // blocks still spread evenly over the SMs
    constexpr int kWarps = NI == 1 ? 4 : 2;
    if (end <= begin) return PP_OK;
    const auto kern = k_eval_reg<PMAX, NI, VEC, OPS, LT>;
    const size_t lt_bytes = LT ? (size_t)a.ktab_words * sizeof(uint32_t) : 0;
    const size_t ring_bytes = (size_t)Ring<PMAX, NI>::kWords * sizeof(int32_t);
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    if (dev >= 64) return PP_ERR_INTERNAL;
    // per device: the shared memory a block may opt into (set on the kernel)
    // and an SM's total
    static std::atomic<int> smem_optin[64], smem_sm[64];
    if (!smem_optin[dev].load(std::memory_order_acquire)) {
        int optin = 0, per_sm = 0;
        PPS_CUDA_TRY(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
        PPS_CUDA_TRY(cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev));
        PPS_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin));
        smem_sm[dev].store(per_sm, std::memory_order_relaxed);
        smem_optin[dev].store(optin, std::memory_order_release);
    }
    const int64_t warps = (end - begin + 32 * NI - 1) / (32 * NI);
    EvalArgs b = a;
    b.inst_begin = begin;
    b.n = end;
    b.tasks = 0;
    // A batch whose warps all fit on the GPU at once: one block per SM, block
    // i taking warp tasks [i*T/G, (i+1)*T/G), so SMs differ by one warp at
    // most (fixed-size blocks would leave some SMs a whole block more than
    // others).  Asking for more than half an SM's shared memory keeps a
    // second block off every SM.
    if constexpr (NI == 1) {
        const int nsm = sm_count(dev);
        const int64_t grid = warps < nsm ? warps : nsm;
        const int64_t wpb = (warps + grid - 1) / grid;
        if (wpb <= 32) {
            size_t smem = lt_bytes + (size_t)wpb * ring_bytes;
            const size_t half = (size_t)smem_sm[dev].load(std::memory_order_relaxed) / 2;
            if (smem < half) smem = half;
            // whether such a block fits, remembered per device for the last
            // (warps, shared memory) pair asked
            // (key in the high word, blocks per SM in the low word)
            static std::atomic<uint64_t> fit_memo[64];
            const uint64_t key = ((uint64_t)wpb << 16 | (uint64_t)(smem >> 4)) + 1;
            uint64_t memo = fit_memo[dev].load(std::memory_order_relaxed);
            if (memo >> 32 != key) {
                int fit = 0;
                if (smem > (size_t)smem_optin[dev].load(std::memory_order_relaxed) ||
                    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, kern, (int)wpb * 32, smem) != cudaSuccess)
                    fit = 0;
                (void)cudaGetLastError();
                memo = key << 32 | (uint32_t)fit;
                fit_memo[dev].store(memo, std::memory_order_relaxed);
            }
            if ((int)(uint32_t)memo >= 1) {
                b.tasks = warps;
                PPS_CUDA_TRY(launch_pdl(kern, (unsigned)grid, (unsigned)wpb * 32, smem, st, pdl, b));
                return PP_OK;
            }
        }
    }
    // several blocks per SM here: an early-started next grid could pile its
    // blocks onto the SMs that free up first, so these launches keep plain
    // stream order
    const size_t smem = lt_bytes + (size_t)kWarps * ring_bytes;
    const int64_t blocks = (warps + kWarps - 1) / kWarps;
    if (blocks > 0x7FFFFFFF) return PP_ERR_SIZE;
    PPS_CUDA_TRY(launch_pdl(kern, (unsigned)blocks, kWarps * 32, smem, st, false, b));
    return PP_OK;
}

// pdl: the tables are the plan's cached ones (built and synchronized before
// this call), so the kernel may copy them before the previous grid ends.
template <int PMAX, bool OPS>
static int launch_reg_o(const EvalArgs &a, bool vec, bool lt, cudaStream_t st, bool pdl = false) {
    if (lt) return launch_reg_t<PMAX, kRegNI, true, OPS, true>(a, 0, a.n, st, pdl);
    if (vec) return launch_reg_t<PMAX, 1, true, OPS, false>(a, 0, a.n, st, pdl);
    return launch_reg_t<PMAX, 1, false, OPS, false>(a, 0, a.n, st, pdl);
}

// Largest per-CTA table area kept in shared memory (words); bigger plans use
// the in-loop address computation.
constexpr int kMaxLtWords = 8192;

template <int PMAX>
static int launch_reg_p(pp_plan *plan, EvalArgs &a, bool vec, bool ops, cudaStream_t st) {
    // costs shared by every microbatch: no loads per round
    if (a.s_mb == 0 && ktab_words(a.R, PMAX, a.nseg) <= kMaxLtWords &&
        (int64_t)(a.S - 1) * a.s_stage < ((int64_t)1 << 30)) {
        const pp_ktab *t = nullptr;
        const int rc = kernel_tables(plan, a.s_stage, a.s_mb, st, &t);
        if (rc) return rc;
        a.ktab = t->d;
        a.ktab_words = t->words;
        return ops ? launch_reg_mbz<PMAX, true>(a, st) : launch_reg_mbz<PMAX, false>(a, st);
    }
    // the table path needs 16-byte aligned rows and offsets below 2^30
    const bool lt = vec && ktab_words(a.R, PMAX, a.nseg) <= kMaxLtWords &&
                    (int64_t)(a.S - 1) * a.s_stage + (int64_t)(a.M - 1) * a.s_mb < ((int64_t)1 << 30);
    if (lt) {
        const pp_ktab *t = nullptr;
        const int rc = kernel_tables(plan, a.s_stage, a.s_mb, st, &t);
        if (rc) return rc;
        a.ktab = t->d;
        a.ktab_words = t->words;
        // 8-wide plans without per-op output, in batches too small to give
        // every SM eight warps of 32 instances: two lanes per instance, twice
        // the warps (on larger batches the one-lane kernel is as fast or
        // faster and moves fewer, larger rows)
        if constexpr (PMAX == 8) {
            int dev = 0;
            PPS_CUDA_TRY(cudaGetDevice(&dev));
            if (!ops && a.n < (int64_t)sm_count(dev) * 8 * 32) return launch_eval_split8(a, st);
        }
    }
    return ops ? launch_reg_o<PMAX, true>(a, vec, lt, st, true) : launch_reg_o<PMAX, false>(a, vec, lt, st, true);
}

int launch_eval_reg(pp_plan *plan, EvalArgs &a, bool vec, bool ops, cudaStream_t st) {
    switch (plan->pmax) {
        case 4: return launch_reg_p<4>(plan, a, vec, ops, st);
        case 8: return launch_reg_p<8>(plan, a, vec, ops, st);
        case 16: return launch_reg_p<16>(plan, a, vec, ops, st);
        default: return PP_ERR_INTERNAL;
    }
}

// Launch the register evaluator on tables the caller already built (the
// entry point that allocates nothing): the table path when a.ktab is set.
bool reg_table_path(int pmax, const EvalArgs &a, bool vec) {
    return vec && ktab_words(a.R, pmax, a.nseg) <= kMaxLtWords &&
           (int64_t)(a.S - 1) * a.s_stage + (int64_t)(a.M - 1) * a.s_mb < ((int64_t)1 << 30);
}

int launch_eval_reg_tables(int pmax, const EvalArgs &a, bool vec, bool ops, cudaStream_t st) {
    const bool lt = a.ktab != nullptr;
    switch (pmax) {
        case 4: return ops ? launch_reg_o<4, true>(a, vec, lt, st) : launch_reg_o<4, false>(a, vec, lt, st);
        case 8: return ops ? launch_reg_o<8, true>(a, vec, lt, st) : launch_reg_o<8, false>(a, vec, lt, st);
        case 16: return ops ? launch_reg_o<16, true>(a, vec, lt, st) : launch_reg_o<16, false>(a, vec, lt, st);
        default: return PP_ERR_INTERNAL;
    }
}

// The fused register path over many problems takes GPipe / 1F1B plans whose
// costs are the same for every microbatch (stride_mb == 0), without per-op
// output: the conditions of the single-problem microbatch-shared path.
bool reg_mbz_ok(const pp_plan *plan, const EvalArgs &a) {
    if (!plan->reg_ok || a.comm_b || a.op_start || a.op_end || a.s_mb != 0 || a.n <= 0) return false;
    return ktab_words(a.R, plan->pmax, a.nseg) <= kMaxLtWords && (int64_t)(a.S - 1) * a.s_stage < ((int64_t)1 << 30);
}

int64_t reg_mbz_warps(const EvalArgs &a) { return (a.n + 31) / 32; }

int64_t reg_mbz_ctas(const EvalArgs &a, int warps) { return (reg_mbz_warps(a) + warps - 1) / warps; }

size_t reg_mbz_smem(int pmax, const EvalArgs &a, int warps) {
    return (size_t)(a.ktab_words - reg_mbz_table_skip(a.R, pmax)) * sizeof(uint32_t) +
           (size_t)warps * 5 * pmax * 32 * sizeof(int32_t);
}

template <int PMAX>
static int launch_mbz_many_t(int warps, const ManyJob *d_jobs, int njobs, int64_t ctas, size_t smem,
                             cudaStream_t st) {
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    if (dev >= 64) return PP_ERR_INTERNAL;
    static std::atomic<int> optin[64];
    if (!optin[dev].load(std::memory_order_acquire)) {
        int o = 0;
        PPS_CUDA_TRY(cudaDeviceGetAttribute(&o, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
        PPS_CUDA_TRY(cudaFuncSetAttribute(k_eval_reg_mbz_many<PMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, o));
        optin[dev].store(o, std::memory_order_release);
    }
    if (smem > (size_t)optin[dev].load(std::memory_order_relaxed)) return PP_ERR_SIZE;
    k_eval_reg_mbz_many<PMAX><<<(unsigned)ctas, warps * 32, smem, st>>>(d_jobs, njobs);
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}

int launch_reg_mbz_many(int pmax, int warps, const ManyJob *d_jobs, int njobs, int64_t ctas, size_t smem,
                        cudaStream_t st) {
    if (njobs <= 0 || ctas <= 0) return PP_OK;
    if (ctas > 0x7FFFFFFF || warps < 1 || warps > kManyRegWarps) return PP_ERR_SIZE;
    switch (pmax) {
        case 4: return launch_mbz_many_t<4>(warps, d_jobs, njobs, ctas, smem, st);
        case 8: return launch_mbz_many_t<8>(warps, d_jobs, njobs, ctas, smem, st);
        case 16: return launch_mbz_many_t<16>(warps, d_jobs, njobs, ctas, smem, st);
        default: return PP_ERR_INTERNAL;
    }
}

}  // namespace pps

namespace pps {

int eval_check(pp_policy_t policy, int P, int M, int v, const int32_t *cost_f, const int32_t *cost_b,
               int64_t stride_inst, int64_t stride_stage, int64_t stride_mb, int64_t comm_stride_inst,
               int64_t comm_stride_bnd, int64_t n_instances) {
    const int rc = check_shape((int)policy, P, M, v);
    if (rc) return rc;
    if (n_instances < 0) return PP_ERR_ARG;
    if (n_instances > 0 && (!cost_f || !cost_b)) return PP_ERR_ARG;
    if (stride_inst < 0 || stride_stage < 0 || stride_mb < 0 || comm_stride_inst < 0 || comm_stride_bnd < 0)
        return PP_ERR_ARG;
    return PP_OK;
}

EvalArgs eval_args(const pp_plan *plan, const int32_t *cost_f, const int32_t *cost_b, int64_t stride_inst,
                   int64_t stride_stage, int64_t stride_mb, const int32_t *comm, const int32_t *comm_b,
                   int64_t comm_stride_inst, int64_t comm_stride_bnd, int64_t n_instances, int32_t *makespan,
                   int32_t *idle, int64_t *bub_num, int64_t *bub_den, int32_t *peak, int32_t *op_start,
                   int32_t *op_end, int64_t op_stride_inst, int64_t op_stride_op, int8_t *status) {
    EvalArgs a{};
    a.peak_src = plan->d_peak; a.peak_dst = peak;
    a.desc = plan->d_desc; a.desc2 = plan->d_desc2; a.rw = plan->d_rw;
    a.seg = plan->d_seg; a.nseg = plan->nseg;
    a.ktab = nullptr; a.ktab_words = 0;
    a.R = plan->R; a.P = plan->P; a.M = plan->M; a.v = plan->v; a.S = plan->S; a.O = plan->O;
    a.nslots = plan->nslots;
    a.cost_f = cost_f; a.cost_b = cost_b;
    a.s_inst = stride_inst; a.s_stage = stride_stage; a.s_mb = stride_mb;
    a.comm = comm; a.comm_b = comm_b; a.c_inst = comm_stride_inst; a.c_bnd = comm_stride_bnd;
    a.n = n_instances;
    a.inst_begin = 0;
    a.makespan = makespan; a.idle = idle; a.bub_num = bub_num; a.bub_den = bub_den; a.status = status;
    a.op_start = op_start; a.op_end = op_end; a.o_inst = op_stride_inst; a.o_op = op_stride_op;
    return a;
}

namespace {

int eval_impl(pp_policy_t policy, int P, int M, int v, const int32_t *cost_f, const int32_t *cost_b,
              int64_t stride_inst, int64_t stride_stage, int64_t stride_mb, const int32_t *comm,
              const int32_t *comm_b, int64_t comm_stride_inst, int64_t comm_stride_bnd, int64_t n_instances,
              int32_t *makespan, int32_t *idle, int64_t *bub_num, int64_t *bub_den, int32_t *peak,
              int32_t *op_start, int32_t *op_end, int64_t op_stride_inst, int64_t op_stride_op, int8_t *status,
              cudaStream_t stream) {
    int rc = eval_check(policy, P, M, v, cost_f, cost_b, stride_inst, stride_stage, stride_mb, comm_stride_inst,
                        comm_stride_bnd, n_instances);
    if (rc) return rc;
    if ((op_start || op_end) && (op_stride_inst < 0 || op_stride_op < 0)) return PP_ERR_ARG;
    pp_plan *plan = nullptr;
    rc = cached_plan((int)policy, P, M, v, stream, &plan);
    if (rc) return rc;
    if (n_instances == 0) {
        // no evaluation kernel to carry the peak
        if (peak)
            PPS_CUDA_TRY(cudaMemcpyAsync(peak, plan->d_peak, P * sizeof(int32_t), cudaMemcpyDeviceToDevice, stream));
        return PP_OK;
    }
    EvalArgs a = eval_args(plan, cost_f, cost_b, stride_inst, stride_stage, stride_mb, comm, comm_b,
                           comm_stride_inst, comm_stride_bnd, n_instances, makespan, idle, bub_num, bub_den, peak,
                           op_start, op_end, op_stride_inst, op_stride_op, status);
    const bool vec = stride_inst == 1 && (reinterpret_cast<uintptr_t>(cost_f) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(cost_b) & 15) == 0 && stride_stage % 4 == 0 &&
                     stride_mb % 4 == 0 &&
                     (int64_t)(plan->S - 1) * stride_stage + (int64_t)(M - 1) * stride_mb < ((int64_t)1 << 31);
    const bool ops = op_start || op_end;
    if (comm_b) {
        // a separate backward latency: the lane evaluator takes it for every policy
        rc = plan_value_slots(plan, stream);
        if (rc) return rc;
        a.desc2 = plan->d_desc2;
        a.nslots = plan->nslots;
        if (!lane_path(plan, a)) return PP_ERR_SIZE;
        return launch_eval_lane(plan, a, vec, ops, stream);
    }
    if (plan->reg_ok) return launch_eval_reg(plan, a, vec, ops, stream);
    if (lane_path(plan, a)) return launch_eval_lane(plan, a, vec, ops, stream);
    return launch_eval_slot(plan, a, vec, ops, stream);
}

}  // namespace
}  // namespace pps

extern "C" int pp_sched_eval(pp_policy_t policy, int P, int M, int v, const int32_t *cost_f,
                             const int32_t *cost_b, int64_t stride_inst, int64_t stride_stage,
                             int64_t stride_mb, const int32_t *comm, int64_t comm_stride_inst,
                             int64_t comm_stride_bnd, int64_t n_instances, int32_t *makespan,
                             int32_t *idle, int64_t *bub_num, int64_t *bub_den, int32_t *peak,
                             int32_t *op_start, int32_t *op_end, int64_t op_stride_inst,
                             int64_t op_stride_op, int8_t *status, cudaStream_t stream) {
    return pps::eval_impl(policy, P, M, v, cost_f, cost_b, stride_inst, stride_stage, stride_mb, comm, nullptr,
                          comm_stride_inst, comm_stride_bnd, n_instances, makespan, idle, bub_num, bub_den, peak,
                          op_start, op_end, op_stride_inst, op_stride_op, status, stream);
}

extern "C" int pp_sched_eval_fb(pp_policy_t policy, int P, int M, int v, const int32_t *cost_f,
                                const int32_t *cost_b, int64_t stride_inst, int64_t stride_stage,
                                int64_t stride_mb, const int32_t *comm_f, const int32_t *comm_b,
                                int64_t comm_stride_inst, int64_t comm_stride_bnd, int64_t n_instances,
                                int32_t *makespan, int32_t *idle, int64_t *bub_num, int64_t *bub_den,
                                int32_t *peak, int32_t *op_start, int32_t *op_end, int64_t op_stride_inst,
                                int64_t op_stride_op, int8_t *status, cudaStream_t stream) {
    return pps::eval_impl(policy, P, M, v, cost_f, cost_b, stride_inst, stride_stage, stride_mb, comm_f, comm_b,
                          comm_stride_inst, comm_stride_bnd, n_instances, makespan, idle, bub_num, bub_den, peak,
                          op_start, op_end, op_stride_inst, op_stride_op, status, stream);
}
