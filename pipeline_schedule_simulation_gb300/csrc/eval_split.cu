// eval_split.cu -- the register evaluator with two lanes per instance.
//
// The same round-by-round max-plus recurrence as k_eval_reg ("2. 1F1B" §2.3,
// §4.3; M040 §04), for GPipe and 1F1B plans with 8-wide rounds, but every
// instance is split over two lanes of a warp: lane j (j < 16) runs devices
// 0..3 of instance j and lane j + 16 devices 4..7.  A warp therefore holds 16
// instances and a batch fills twice as many warps, which is what the
// HBM-bound hot path lacks at tens of thousands of instances: each warp keeps
// its own rounds of cost copies in flight, so more warps means more bytes in
// flight.  The price is one shuffle per round: at the end of every round the
// lower lane passes its device 3's forward arrival to device 4 and the upper
// lane its device 4's backward arrival to device 3, so every input is still
// the value as of the start of the round (the register evaluator's rule).
//
// Costs are staged by cp.async six rounds ahead into a per-warp ring of round
// slices laid out [device mod 4][half][instance], conflict-free for the
// compute; one 16-byte copy per lane and round (4 lanes cover the 64 bytes of
// a device's row for the warp's 16 instances), driven by the same per-stride
// loader table, round words and segments as k_eval_reg.
#include <atomic>

#include "eval_common.cuh"

namespace pps {

template <int PMAX>
struct SplitGeom {
    static constexpr int kH = PMAX / 2;                 // devices per lane
    static constexpr int kIPW = 16;                     // instances per warp
    static constexpr int kSlices = 8;
    static constexpr int kAhead2 = kSlices - 2;         // rounds copied ahead
    static constexpr int kSliceWords = PMAX * kIPW;     // [PMAX/2][2][16]
    static constexpr int kRingWords = kSlices * kSliceWords;
    static constexpr int kWarps = 4;
    static_assert(PMAX == 8, "the loader maps 4 lanes to each of 8 device rows");
};

template <int H>
struct SplitState {
    uint32_t fr[H], rf[H], rb[H], busy[H], cF[H];
    uint32_t cL;           // comm of the boundary below this lane's first device (upper half)
    uint32_t rf_in, rb_in;  // the other half's boundary arrivals (0 where there is none)
    uint32_t flag;
};

template <int H, bool FWD, int I>
__device__ __forceinline__ void split_op(SplitState<H> &S, uint32_t arr, const int32_t *sl) {
    const uint32_t c = (uint32_t)sl[I * 32];
    const uint32_t st = max(S.fr[I], arr);
    const uint32_t en = st + c;
    S.fr[I] = en;
    S.busy[I] += c;
    S.flag |= st | c;
    if constexpr (FWD) S.rf[I] = en + S.cF[I];
    else S.rb[I] = en + (I > 0 ? S.cF[I > 0 ? I - 1 : 0] : S.cL);
}

template <int H, int I>
__device__ __forceinline__ uint32_t split_in_f(const SplitState<H> &S) {
    return I > 0 ? S.rf[I > 0 ? I - 1 : 0] : S.rf_in;
}
template <int H, int I>
__device__ __forceinline__ uint32_t split_in_b(const SplitState<H> &S) {
    return I < H - 1 ? S.rb[I < H - 1 ? I + 1 : 0] : S.rb_in;
}

// Alternating round (devices of one parity F, the other B); the device index
// parity is the same in both halves since H is even.
template <int H, bool MASKED, bool EVEN_FWD, int I = 0>
__device__ __forceinline__ void split_alt(SplitState<H> &S, uint32_t mask, const int32_t *sl) {
    if constexpr (I < H) {
        if (!MASKED || ((mask >> I) & 1u)) {
            constexpr bool fwd = ((I & 1) == 0) == EVEN_FWD;
            if constexpr (fwd) split_op<H, true, I>(S, split_in_f<H, I>(S), sl);
            else split_op<H, false, I>(S, split_in_b<H, I>(S), sl);
        }
        split_alt<H, MASKED, EVEN_FWD, I + 1>(S, mask, sl);
    }
}

template <int H, bool MASKED, int I = H - 1>
__device__ __forceinline__ void split_all_f(SplitState<H> &S, uint32_t mask, const int32_t *sl) {
    if constexpr (I >= 0) {
        if (!MASKED || ((mask >> I) & 1u)) split_op<H, true, I>(S, split_in_f<H, I>(S), sl);
        split_all_f<H, MASKED, I - 1>(S, mask, sl);
    }
}

template <int H, bool MASKED, int I = 0>
__device__ __forceinline__ void split_all_b(SplitState<H> &S, uint32_t mask, const int32_t *sl) {
    if constexpr (I < H) {
        if (!MASKED || ((mask >> I) & 1u)) split_op<H, false, I>(S, split_in_b<H, I>(S), sl);
        split_all_b<H, MASKED, I + 1>(S, mask, sl);
    }
}

template <int H>
__device__ __forceinline__ void split_generic(SplitState<H> &S, uint32_t kinds, const int32_t *sl) {
    uint32_t inF[H], inB[H];
#pragma unroll
    for (int i = 0; i < H; ++i) {
        inF[i] = i > 0 ? S.rf[i > 0 ? i - 1 : 0] : S.rf_in;
        inB[i] = i < H - 1 ? S.rb[i < H - 1 ? i + 1 : 0] : S.rb_in;
    }
    [&]<int... I>(std::integer_sequence<int, I...>) {
        ([&] {
            const uint32_t kind = (kinds >> (2 * I)) & 3u;
            if (kind == kFwd) split_op<H, true, I>(S, inF[I], sl);
            else if (kind == kBwd) split_op<H, false, I>(S, inB[I], sl);
        }(), ...);
    }(std::make_integer_sequence<int, H>{});
}

// kinds and mask of this lane's devices
template <int H>
__device__ __forceinline__ void split_round(SplitState<H> &S, uint64_t w, int h, const int32_t *sl) {
    const uint32_t m = (rw_mask(w) >> (h * H)) & ((1u << H) - 1u);
    switch (rw_pattern(w)) {
        case kPatAltA: split_alt<H, false, true>(S, m, sl); break;
        case kPatAltB: split_alt<H, false, false>(S, m, sl); break;
        case kPatAllF: split_all_f<H, false>(S, m, sl); break;
        case kPatAllB: split_all_b<H, false>(S, m, sl); break;
        case kPatMasked + kPatAltA: split_alt<H, true, true>(S, m, sl); break;
        case kPatMasked + kPatAltB: split_alt<H, true, false>(S, m, sl); break;
        case kPatMasked + kPatAllF: split_all_f<H, true>(S, m, sl); break;
        case kPatMasked + kPatAllB: split_all_b<H, true>(S, m, sl); break;
        default: split_generic<H>(S, rw_kinds(w) >> (2 * h * H), sl); break;
    }
}

template <int PMAX>
__global__ void __launch_bounds__(128) k_eval_split(const EvalArgs a) {
    copy_peak(a);
    using G = SplitGeom<PMAX>;
    constexpr int H = G::kH, D = G::kAhead2;
    extern __shared__ __align__(16) int32_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int h = lane >> 4, j = lane & 15;
    // the block's copy of the loader table, round words and segments
    for (int i = threadIdx.x; i < a.ktab_words / 4; i += blockDim.x)
        cp_async16(smem_addr(smem + 4 * i), a.ktab + i, 16u);
    cp_async_commit();
    const uint32_t *lt = reinterpret_cast<const uint32_t *>(smem);
    const int tw = (a.R * PMAX + 3) & ~3;
    const uint64_t *rws = reinterpret_cast<const uint64_t *>(smem + tw);
    const uint4 *segs = reinterpret_cast<const uint4 *>(smem + tw + 2 * ((a.R + 1) & ~1));
    int32_t *ring = smem + a.ktab_words + warp * G::kRingWords;
    const int64_t inst0 = ((int64_t)blockIdx.x * G::kWarps + warp) * G::kIPW;
    const int64_t x = inst0 + j;
    const bool live = x < a.n;

    SplitState<H> S;
    uint32_t negc = 0;
#pragma unroll
    for (int i = 0; i < H; ++i) {
        const int gk = h * H + i;
        uint32_t c = 0;
        if (a.comm && live && gk < a.P - 1) c = (uint32_t)a.comm[x * a.c_inst + (int64_t)gk * a.c_bnd];
        negc |= c;
        S.cF[i] = c;
        S.fr[i] = 0; S.rf[i] = 0; S.rb[i] = 0; S.busy[i] = 0;
    }
    S.cL = 0;
    if (a.comm && live && h == 1 && H - 1 < a.P - 1) S.cL = (uint32_t)a.comm[x * a.c_inst + (int64_t)(H - 1) * a.c_bnd];
    negc |= S.cL;
    S.rf_in = 0; S.rb_in = 0; S.flag = 0;
    cp_async_wait<0>();
    __syncthreads();
    if (inst0 >= a.n) return;  // warp-uniform, after the block barrier

    // loader: lane copies 16 bytes (4 instances) of device row d = lane / 4
    const int d = lane >> 2, q = lane & 3;
    const int64_t x4 = inst0 + 4 * q;
    const int64_t left = a.n - x4;
    const uint32_t bytes_in = left <= 0 ? 0u : (left >= 4 ? 16u : (uint32_t)left * 4u);
    const int64_t xoff = bytes_in ? x4 : 0;
    const int32_t *fbase = a.cost_f + xoff;
    const int32_t *bbase = a.cost_b + xoff;
    [[maybe_unused]] const int64_t reach = cost_reach(a.n, a.S, a.M, a.s_inst, a.s_stage, a.s_mb);
    const int dst_word = ((d % H) * 2 + d / H) * G::kIPW + 4 * q;
    const int R = a.R;
    auto issue = [&](int rl) {
        if (rl < R) {
            const uint32_t e = lt[rl * PMAX + d];
            const int32_t *src = (e & 1u) ? bbase : fbase;
            uint32_t nb = 0;
            if (e != kLtIdle && PPS_CHECK(xoff + (e >> 1) + bytes_in / 4 <= reach, kChkCostRead, xoff + (e >> 1))) {
                src += e >> 1;
                nb = bytes_in;
            }
            cp_async16(smem_addr(ring + (rl % G::kSlices) * G::kSliceWords + dst_word), src, nb);
        }
        cp_async_commit();
    };
    // this lane's costs in a slice: device i at word (i*2 + h)*16 + j
    auto slice = [&](int r) { return ring + (r % G::kSlices) * G::kSliceWords + h * G::kIPW + j; };
    auto exchange = [&]() {
        const uint32_t send = h ? S.rb[0] : S.rf[H - 1];
        const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, send, 16);
        S.rf_in = h ? recv : 0u;
        S.rb_in = h ? 0u : recv;
    };
    auto step1 = [&](int r, auto &&body) {
        issue(r + D);
        cp_async_wait<D>();
        __syncwarp();
        body(slice(r));
        exchange();
    };
    auto step2 = [&](int r, auto &&body0, auto &&body1) {
        issue(r + D);
        issue(r + D + 1);
        cp_async_wait<D>();
        __syncwarp();
        body0(slice(r));
        exchange();
        body1(slice(r + 1));
        exchange();
    };
    auto altA = [&](const int32_t *sl) { split_alt<H, false, true>(S, 0u, sl); };
    auto altB = [&](const int32_t *sl) { split_alt<H, false, false>(S, 0u, sl); };
    auto allF = [&](const int32_t *sl) { split_all_f<H, false>(S, 0u, sl); };
    auto allB = [&](const int32_t *sl) { split_all_b<H, false>(S, 0u, sl); };

#pragma unroll 1
    for (int qd = 0; qd < D; ++qd) issue(qd);
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
                step1(r, [&](const int32_t *sl) { split_round<H>(S, w, h, sl); });
                break;
            }
        }
    }
    cp_async_wait<0>();

    // per-instance reductions over both lanes (as write_results_u)
    uint32_t mk = 0;
#pragma unroll
    for (int i = 0; i < H; ++i) mk = max(mk, S.fr[i]);
    mk = max(mk, __shfl_xor_sync(0xFFFFFFFFu, mk, 16));
    uint32_t flag = S.flag | mk;
    flag |= __shfl_xor_sync(0xFFFFFFFFu, flag, 16);
    negc |= __shfl_xor_sync(0xFFFFFFFFu, negc, 16);
    int64_t num = 0;
#pragma unroll
    for (int i = 0; i < H; ++i) {
        const int gk = h * H + i;
        if (gk < a.P) {
            const int idle = (int)(mk - S.busy[i]);
            num += idle;
            if (live && a.idle) a.idle[x * a.P + gk] = idle;
        }
    }
    num += __shfl_xor_sync(0xFFFFFFFFu, num, 16);
    if (!live || h) return;
    if (a.makespan) a.makespan[x] = (int)mk;
    if (a.bub_num) a.bub_num[x] = num;
    if (a.bub_den) a.bub_den[x] = (int64_t)a.P * (int)mk;
    if (a.status) {
        int8_t st = PP_ST_OK;
        if (negc >> 31) st = PP_ST_NEG_COST;
        else if (flag >> 31) st = any_negative_cost(a, x) ? PP_ST_NEG_COST : PP_ST_OVERFLOW;
        a.status[x] = st;
    }
}

// Launch on tables the caller resolved (a.ktab set, PMAX 8, no per-op output).
int launch_eval_split8(const EvalArgs &a, cudaStream_t st) {
    using G = SplitGeom<8>;
    const size_t smem = (size_t)a.ktab_words * sizeof(uint32_t) + (size_t)G::kWarps * G::kRingWords * sizeof(int32_t);
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    static std::atomic<bool> attr_set[64];  // per device, set once (idempotent)
    if (dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
        PPS_CUDA_TRY(cudaFuncSetAttribute(k_eval_split<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024));
        attr_set[dev].store(true, std::memory_order_release);
    }
    const int64_t warps = (a.n + G::kIPW - 1) / G::kIPW;
    const int64_t blocks = (warps + G::kWarps - 1) / G::kWarps;
    if (blocks > 0x7FFFFFFF) return PP_ERR_SIZE;
    k_eval_split<8><<<(unsigned)blocks, G::kWarps * 32, smem, st>>>(a);
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}

}  // namespace pps
