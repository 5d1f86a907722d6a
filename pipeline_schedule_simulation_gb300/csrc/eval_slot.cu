// eval_slot.cu -- the generic evaluator (any policy; used for interleaved 1F1B).
//
// Same round-by-round max-plus recurrence as the register evaluator, but an
// op's input is found through the plan's value slots instead of a fixed
// register: with v > 1 chunks per device several results of one kind can be
// in flight between two devices ("2. 1F1B" §6.1; M040 §06: a device holds
// virtual stages k, k+P, ...).  The plan colours each in-flight result (from
// its producer's round to its consumer's round) onto one of at most 64 slots;
// each warp keeps the slots and the instance's comm table in shared memory as
// [slot][lane], so every access is conflict-free.
#include <atomic>

#include "eval_common.cuh"

namespace pps {

template <int PMAX, bool VEC, bool OPS>
__global__ void __launch_bounds__(128) k_eval_slot(const EvalArgs a) {
    copy_peak(a);
    using RG = Ring<PMAX>;
    extern __shared__ __align__(16) int32_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per_warp = RG::kWords + (a.nslots + a.S) * 32;
    int32_t *ring = smem + warp * per_warp;
    int32_t *val = ring + RG::kWords;           // [nslots][32]
    int32_t *ctab = val + a.nslots * 32;        // [S][32], entry b = comm of boundary b
    const int64_t inst0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + warp) * 32;
    if (inst0 >= a.n) return;  // warp-uniform
    const int64_t x = inst0 + lane;
    const bool live = x < a.n;

    uint32_t neg = 0;
    for (int b = 0; b < a.S; ++b) {
        int c = 0;
        if (a.comm && live && b < a.S - 1) c = a.comm[x * a.c_inst + (int64_t)b * a.c_bnd];
        neg |= (uint32_t)c;
        ctab[b * 32 + lane] = c;
    }
    int fr[PMAX], busy[PMAX], cnt[PMAX];
#pragma unroll
    for (int k = 0; k < PMAX; ++k) { fr[k] = 0; busy[k] = 0; cnt[k] = 0; }
    uint32_t accE = 0, accC = 0;

    // Descriptors are loaded one round before they are used (the loader's for
    // round r+kAhead+1, the compute's for round r+1), so no global load sits
    // on the critical path of a round.
    const int R = a.R;
    LoadDesc<PMAX, VEC> ld;
#pragma unroll 1
    for (int q = 0; q < RG::kAhead; ++q) {
        if (q < R) {
            fetch_load_desc<PMAX, VEC>(a, q, lane, ld);
            load_round<PMAX, VEC>(a, q, ld, ring, inst0, lane);
        }
        cp_async_commit();
    }
    if (RG::kAhead < R) fetch_load_desc<PMAX, VEC>(a, RG::kAhead, lane, ld);
    uint32_t dn[PMAX], d2n[PMAX];
    load_desc<PMAX>(a.desc, dn);
    load_desc<PMAX>(a.desc2, d2n);
#pragma unroll 1
    for (int r = 0; r < R; ++r) {
        if (r + RG::kAhead < R) {
            load_round<PMAX, VEC>(a, r + RG::kAhead, ld, ring, inst0, lane);
            if (r + RG::kAhead + 1 < R) fetch_load_desc<PMAX, VEC>(a, r + RG::kAhead + 1, lane, ld);
        }
        cp_async_commit();
        uint32_t d[PMAX], d2[PMAX];
#pragma unroll
        for (int k = 0; k < PMAX; ++k) { d[k] = dn[k]; d2[k] = d2n[k]; }
        if (r + 1 < R) {
            load_desc<PMAX>(a.desc + (int64_t)(r + 1) * PMAX, dn);
            load_desc<PMAX>(a.desc2 + (int64_t)(r + 1) * PMAX, d2n);
        }
        cp_async_wait<RG::kAhead>();
        __syncwarp();
        const int32_t *slice = ring + (r % RG::kSlices) * (PMAX * 32);
        // All reads of the round happen before its writes: a slot is reused only
        // after the round that consumed it, so reads and writes of one round
        // never alias; reading first keeps that independent of device order.
        int arr[PMAX];
#pragma unroll
        for (int k = 0; k < PMAX; ++k) {
            arr[k] = 0;
            const uint32_t rs = d2_rslot(d2[k]);
            if (desc_kind(d[k]) != kIdle && rs != kNoSlot &&
                PPS_CHECK(rs < (uint32_t)a.nslots, kChkSlotIndex, rs) &&
                PPS_CHECK(d2_cbnd(d2[k]) < (uint32_t)a.S, kChkSlotIndex, d2_cbnd(d2[k])))
                arr[k] = wrap_add(val[rs * 32 + lane], ctab[d2_cbnd(d2[k]) * 32 + lane]);
        }
#pragma unroll
        for (int k = 0; k < PMAX; ++k) {
            if (desc_kind(d[k]) == kIdle) continue;
            const int c = slice[k * 32 + lane];
            const int st = max(fr[k], arr[k]);
            const int en = wrap_add(st, c);
            fr[k] = en;
            busy[k] = wrap_add(busy[k], c);
            accE |= (uint32_t)en | (uint32_t)arr[k];
            accC |= (uint32_t)c;
            const uint32_t ws = d2_wslot(d2[k]);
            if (ws != kNoSlot && PPS_CHECK(ws < (uint32_t)a.nslots, kChkSlotIndex, ws)) val[ws * 32 + lane] = en;
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
static int launch_slot_t(const EvalArgs &a, cudaStream_t st) {
    constexpr int kWarps = 2;
    const size_t per_warp = (size_t)(Ring<PMAX>::kWords + (a.nslots + a.S) * 32) * sizeof(int32_t);
    const size_t smem = kWarps * per_warp;
    // opt in to > 48 KB once per instantiation and device (idempotent)
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    static std::atomic<bool> attr_set[64];
    if (dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
        PPS_CUDA_TRY(cudaFuncSetAttribute(k_eval_slot<PMAX, VEC, OPS>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
        if (dev < 64) attr_set[dev].store(true, std::memory_order_release);
    }
    const int64_t warps = (a.n + 31) / 32;
    const int64_t blocks = (warps + kWarps - 1) / kWarps;
    if (blocks > 0x7FFFFFFF) return PP_ERR_SIZE;
    k_eval_slot<PMAX, VEC, OPS><<<(unsigned)blocks, kWarps * 32, smem, st>>>(a);
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}

template <int PMAX>
static int launch_slot_p(const EvalArgs &a, bool vec, bool ops, cudaStream_t st) {
    if (vec) return ops ? launch_slot_t<PMAX, true, true>(a, st) : launch_slot_t<PMAX, true, false>(a, st);
    return ops ? launch_slot_t<PMAX, false, true>(a, st) : launch_slot_t<PMAX, false, false>(a, st);
}

int launch_eval_slot(const pp_plan *plan, const EvalArgs &a, bool vec, bool ops, cudaStream_t st) {
    if (!plan->d_desc2) return PP_ERR_INTERNAL;
    switch (plan->pmax) {
        case 4: return launch_slot_p<4>(a, vec, ops, st);
        case 8: return launch_slot_p<8>(a, vec, ops, st);
        case 16: return launch_slot_p<16>(a, vec, ops, st);
        default: return PP_ERR_INTERNAL;
    }
}

}  // namespace pps
