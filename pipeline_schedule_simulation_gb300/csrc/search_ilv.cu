// search_ilv.cu -- the partition search over interleaved layouts
// (pp_sched_partition_search_interleaved).
//
// "Pipeline scheduling" (M040) §06: one device can hold several virtual
// stages (segments 0..3 in order, device A holding 0 and 2, B holding 1 and
// 3); §05: split by measured computation and activation.  A candidate cuts the
// L layers into S = P*v contiguous non-empty ranges (a seeded draw of a colex
// rank, as the 1F1B search); range s is virtual stage s, chunk s / P of device
// s mod P.  It is rejected when a device's held activation bytes -- the
// ledger of "2. 1F1B" §4.1 weighted by the bytes of each op's chunk -- peak
// above the cap, and otherwise scored by its interleaved 1F1B makespan.
//
// The candidates of a call are processed in chunks of up to kChunk: one
// kernel draws each candidate's split, checks the byte ledger (from the
// shape's table of dominant held-count vectors) and, when only the winner is
// wanted, a makespan lower bound against the best of the chunks already
// scored; the candidates left are packed into a scratch cost table laid out
// [S][column] (the evaluator's instance-minor layout, costs the same for every
// microbatch); the host reads how many there are and the interleaved evaluator
// scores them; a third kernel maps the results back to the candidates and
// reduces (makespan, candidate) with one 64-bit atomicMin per warp into the
// caller's best_idx word.  The scratch table is allocated on a device's first
// call and kept (grown when a call needs more).
#include <algorithm>
#include <deque>
#include <mutex>
#include <vector>

#include <atomic>

#include "eval_common.cuh"
#include "search_common.cuh"

namespace pps {
namespace {

constexpr int kIlvMaxL = 256;
constexpr int kChunk = 1 << 18;

struct IlvArgs {
    const int32_t *ltf, *ltb;
    const int64_t *lact;
    int L, P, v, S, M, O;
    int64_t cap;
    uint64_t seed;
    int64_t begin;
    uint64_t ncomb;        // C(L-1, S-1)
    const uint32_t *ops;   // plan: [P][O] packed ops (kind bit 31, chunk bits 24..30)
    const uint16_t *lvec;  // held-count vectors that can be a device's ledger maximum, [..][v]
    const int *loff;       // device d's vectors are lvec rows loff[d] .. loff[d+1]-1
    int32_t *cf, *cb;      // scratch [S][cn]
    int8_t *flag;          // scratch [cn]: kIlvScored, kIlvOverCap, kIlvBig or kIlvBound
    int *slot;             // scratch [cn]: the candidate's column in cf / cb, -1 if not scored
    int *count;            // columns handed out in this chunk
    const unsigned long long *key;  // the call's reduction word (best so far)
    int32_t comm;
    bool prune;            // only the winner is wanted: skip candidates by the makespan bound
    int cn;                // stride of the scratch tables
};

// Dynamic shared memory: prefix sums of the layer costs and bytes, then
// C(n, i) for n < L, i < S.
struct IlvTables {
    int64_t *pre_tf, *pre_tb, *pre_act;
    uint64_t *C;  // [L][S]
};

__device__ IlvTables ilv_tables(const IlvArgs &a, unsigned char *smem) {
    IlvTables t;
    t.pre_tf = reinterpret_cast<int64_t *>(smem);
    t.pre_tb = t.pre_tf + (a.L + 1);
    t.pre_act = t.pre_tb + (a.L + 1);
    t.C = reinterpret_cast<uint64_t *>(t.pre_act + (a.L + 1));
    for (int e = threadIdx.x; e < a.L * a.S; e += blockDim.x) t.C[e] = binom_u64(e / a.S, e % a.S);
    if (threadIdx.x == 0) {
        int64_t f = 0, b = 0, c = 0;
        t.pre_tf[0] = t.pre_tb[0] = t.pre_act[0] = 0;
        for (int l = 0; l < a.L; ++l) {
            f += a.ltf[l]; b += a.ltb[l]; c += a.lact[l];
            t.pre_tf[l + 1] = f; t.pre_tb[l + 1] = b; t.pre_act[l + 1] = c;
        }
    }
    __syncthreads();
    return t;
}

size_t ilv_smem(int L, int S) { return (size_t)3 * (L + 1) * sizeof(int64_t) + (size_t)L * S * sizeof(uint64_t); }

// Colex unranking of r into S-1 cut positions; first[s] = first layer of
// range s (first[0] = 0, first[S] = L).
__device__ void ilv_unrank(const IlvArgs &a, const IlvTables &t, uint64_t r, int *first) {
    int hi = a.L - 2;
    for (int i = a.S - 1; i >= 1; --i) {
        int c = hi;
        while (c >= i && t.C[c * a.S + i] > r) --c;
        r -= t.C[c * a.S + i];
        first[i] = c + 1;
        hi = c - 1;
    }
    first[0] = 0;
    first[a.S] = a.L;
}

// Flags of a chunk candidate: 0 scored, 1 over the byte cap, 2 a stage sum
// out of int32, 3 skipped by the makespan bound (only when the winner alone
// is wanted).  Only flag-0 candidates are written to the scratch table, packed
// in the order a warp-aggregated counter hands out columns; slot[i] is chunk
// candidate i's column.
constexpr int8_t kIlvScored = 0, kIlvOverCap = 1, kIlvBig = 2, kIlvBound = 3;

__global__ void __launch_bounds__(256) k_ilv_cands(const IlvArgs a, int64_t chunk0, int nchunk) {
    extern __shared__ __align__(16) unsigned char ilv_sm[];
    const IlvTables t = ilv_tables(a, ilv_sm);
    const int lane = threadIdx.x & 31;
    for (int base = blockIdx.x * blockDim.x; base < nchunk; base += gridDim.x * blockDim.x) {
        const int i = base + threadIdx.x;
        const bool live = i < nchunk;
        int first[PP_MAX_S + 1];
        int8_t fl = kIlvBig;
        if (live) {
            int64_t act[PP_MAX_S];
            const uint64_t r = splitmix64(a.seed + (uint64_t)(a.begin + chunk0 + i)) % a.ncomb;
            ilv_unrank(a, t, r, first);
            fl = kIlvScored;
            // (checked build: the split points increase strictly from 0 to L)
            for (int s = 0; s < a.S; ++s)
                if (!PPS_CHECK(first[s] >= 0 && first[s] < first[s + 1] && first[s + 1] <= a.L &&
                                   (s + 1 < a.S || first[s + 1] == a.L),
                               kChkSearchSplit, first[s + 1])) {
                    for (int q = 0; q <= a.S; ++q) first[q] = 0;
                    fl = kIlvBig;
                    break;
                }
            for (int s = 0; s < a.S; ++s) {
                const int64_t sf = t.pre_tf[first[s + 1]] - t.pre_tf[first[s]];
                const int64_t sb = t.pre_tb[first[s + 1]] - t.pre_tb[first[s]];
                act[s] = t.pre_act[first[s + 1]] - t.pre_act[first[s]];
                if (sf < 0 || sb < 0 || sf > 0x7FFFFFFF || sb > 0x7FFFFFFF) fl = kIlvBig;
            }
            // held bytes per device: + the chunk's bytes at F, - at B, running
            // max.  With every range's bytes >= 0 the maximum over the order is
            // the largest dot product of the bytes with the device's held-count
            // vectors that no other vector of its order dominates (the plan's
            // ledger table, a few per device); otherwise walk the order.
            bool nonneg = a.lvec != nullptr;
            for (int s = 0; s < a.S; ++s) nonneg = nonneg && act[s] >= 0;
            for (int d = 0; d < a.P && fl == kIlvScored && nonneg; ++d) {
                int64_t top = 0;
                for (int q = a.loff[d]; q < a.loff[d + 1]; ++q) {
                    int64_t held = 0;
                    for (int c = 0; c < a.v; ++c) held += (int64_t)a.lvec[q * a.v + c] * act[c * a.P + d];
                    top = max(top, held);
                }
                if (top > a.cap) fl = kIlvOverCap;
            }
            for (int d = 0; d < a.P && fl == kIlvScored && !nonneg; ++d) {
                int64_t held = 0, top = 0;
                const uint32_t *row = a.ops + (int64_t)d * a.O;
                for (int j = 0; j < a.O; ++j) {
                    const uint32_t op = __ldg(row + j);
                    const int64_t b = act[((op >> 24) & 0x7Fu) * a.P + d];
                    held += (op >> 31) ? -b : b;
                    top = max(top, held);
                }
                if (top > a.cap) fl = kIlvOverCap;
            }
            if (fl == kIlvScored && a.prune) {
                // Only the winner is wanted: with M a multiple of P, device d
                // starts with microbatch 0's forward of virtual stage d (after
                // the stages before it and their boundaries), ends with the
                // backward of virtual stage d for microbatch M-1 (whose gradient
                // still crosses them back) and runs its 2Mv ops one at a time,
                // so the makespan is at least
                //   max_d [sum_{s<d} (f_s + b_s) + 2 d comm + M sum_chunks (f + b)].
                // A candidate above the best makespan of the chunks already
                // scored cannot win (ties are still scored).
                int64_t lb = 0, pre = 0;
                for (int d = 0; d < a.P; ++d) {
                    int64_t busy = 0;
                    for (int c = 0; c < a.v; ++c) {
                        const int s = c * a.P + d;
                        busy += (t.pre_tf[first[s + 1]] - t.pre_tf[first[s]]) +
                                (t.pre_tb[first[s + 1]] - t.pre_tb[first[s]]);
                    }
                    lb = max(lb, pre + 2 * (int64_t)d * a.comm + (int64_t)a.M * busy);
                    pre += (t.pre_tf[first[d + 1]] - t.pre_tf[first[d]]) + (t.pre_tb[first[d + 1]] - t.pre_tb[first[d]]);
                }
                const unsigned long long best = *reinterpret_cast<volatile const unsigned long long *>(a.key);
                if (lb > (int64_t)(best >> 32)) fl = kIlvBound;
            }
        }
        // columns for the candidates to score, one atomic per warp
        const bool keep = live && fl == kIlvScored;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, keep);
        int col0 = 0;
        if (lane == 0 && m) col0 = atomicAdd(a.count, __popc(m));
        col0 = __shfl_sync(0xFFFFFFFFu, col0, 0);
        if (!live) continue;
        int col = -1;
        if (keep) {
            col = col0 + __popc(m & ((1u << lane) - 1u));
            for (int s = 0; s < a.S; ++s) {
                a.cf[(int64_t)s * a.cn + col] = (int32_t)(t.pre_tf[first[s + 1]] - t.pre_tf[first[s]]);
                a.cb[(int64_t)s * a.cn + col] = (int32_t)(t.pre_tb[first[s + 1]] - t.pre_tb[first[s]]);
            }
        }
        a.flag[i] = fl;
        a.slot[i] = col;
    }
}

__global__ void __launch_bounds__(256) k_ilv_select(const int32_t *mk, const int8_t *status, const int8_t *flag,
                                                    const int *slot, int nchunk, int64_t chunk0, int32_t *all_mk,
                                                    unsigned long long *key) {
    const int lane = threadIdx.x & 31;
    for (int base = blockIdx.x * blockDim.x; base < nchunk; base += gridDim.x * blockDim.x) {
        const int i = base + threadIdx.x;
        int m = -1;
        if (i < nchunk) {
            const int8_t f = flag[i];
            if (f == kIlvOverCap || f == kIlvBound) m = -1;
            else if (f == kIlvBig) m = -2;
            else m = status[slot[i]] != PP_ST_OK ? -2 : mk[slot[i]];
            if (all_mk) all_mk[chunk0 + i] = m;
        }
        unsigned long long k = ~0ull;
        if (i < nchunk && m >= 0) k = ((unsigned long long)(uint32_t)m << 32) | (uint32_t)(chunk0 + i);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, k, o);
            k = other < k ? other : k;
        }
        if (lane == 0 && k != ~0ull) atomicMin(key, k);
    }
}

__global__ void k_ilv_finish(const IlvArgs a, const unsigned long long *key, int64_t *best_idx, int32_t *best_mk,
                             int32_t *best_cuts) {
    extern __shared__ __align__(16) unsigned char ilv_sm[];
    const IlvTables t = ilv_tables(a, ilv_sm);
    if (threadIdx.x != 0) return;
    const unsigned long long k = *key;
    if (k == ~0ull) {
        *best_idx = -1;
        if (best_mk) *best_mk = -1;
        if (best_cuts) for (int s = 0; s + 1 < a.S; ++s) best_cuts[s] = -1;
        return;
    }
    const int64_t ci = (int64_t)(k & 0xFFFFFFFFull);
    if (best_cuts) {
        int first[PP_MAX_S + 1];
        ilv_unrank(a, t, splitmix64(a.seed + (uint64_t)(a.begin + ci)) % a.ncomb, first);
        for (int s = 1; s < a.S; ++s) best_cuts[s - 1] = first[s];
    }
    if (best_mk) *best_mk = (int)(k >> 32);
    *best_idx = a.begin + ci;
}

// Per-device scratch: cost tables [S][cn] x 2, makespan, status, flag, comm.
struct IlvScratch {
    void *p = nullptr;
    size_t bytes = 0;
};
std::mutex g_ilv_mu;
IlvScratch g_ilv[64];

int ilv_scratch(size_t need, void **out) {
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return PP_ERR_SIZE;
    IlvScratch &s = g_ilv[dev];
    if (s.bytes < need) {
        if (s.p) PPS_CUDA_TRY(cudaFree(s.p));
        s.p = nullptr;
        s.bytes = 0;
        PPS_CUDA_TRY(cudaMalloc(&s.p, need));
        s.bytes = need;
    }
    *out = s.p;
    return PP_OK;
}

// Per shape and device: the ledger table of the plan's order.  For device d
// it holds the held-count vectors h (h[c] = forwards minus backwards of chunk
// c so far, the empty prefix included) that no other vector of the order
// dominates in every component; for non-negative bytes the ledger's maximum
// is the largest dot product of the bytes with one of them.  Built once from
// the plan (a copy to the host and back) and kept; guarded by g_ilv_mu.
struct LedgerTab {
    int dev, P, M, v;
    uint16_t *d_vec = nullptr;
    int *d_off = nullptr;
};
std::deque<LedgerTab> g_ledger;

int ledger_tab(const pp_plan *plan, int dev, const LedgerTab **out) {
    for (const LedgerTab &t : g_ledger)
        if (t.dev == dev && t.P == plan->P && t.M == plan->M && t.v == plan->v) { *out = &t; return PP_OK; }
    const int P = plan->P, v = plan->v, O = plan->O;
    std::vector<uint32_t> ops((size_t)P * O);
    PPS_CUDA_TRY(cudaMemcpy(ops.data(), plan->d_ops, ops.size() * sizeof(uint32_t), cudaMemcpyDeviceToHost));
    std::vector<uint16_t> vec;
    std::vector<int> off(1, 0);
    for (int d = 0; d < P; ++d) {
        std::vector<std::vector<int>> seen(1, std::vector<int>(v, 0));
        std::vector<int> h(v, 0);
        for (int j = 0; j < O; ++j) {
            const uint32_t op = ops[(size_t)d * O + j];
            h[PP_OP_CHUNK(op)] += PP_OP_KIND(op) ? -1 : 1;
            seen.push_back(h);
        }
        std::sort(seen.begin(), seen.end());
        seen.erase(std::unique(seen.begin(), seen.end()), seen.end());
        for (size_t x = 0; x < seen.size(); ++x) {
            bool dominated = false;
            for (size_t y = 0; y < seen.size() && !dominated; ++y) {
                if (y == x) continue;
                bool ge = true;
                for (int c = 0; c < v && ge; ++c) ge = seen[y][c] >= seen[x][c];
                dominated = ge;  // distinct vectors: >= everywhere means > somewhere
            }
            if (dominated) continue;
            for (int c = 0; c < v; ++c) {
                if (seen[x][c] < 0 || seen[x][c] > 0xFFFF) return PP_ERR_INTERNAL;
                vec.push_back((uint16_t)seen[x][c]);
            }
        }
        off.push_back((int)(vec.size() / v));
    }
    LedgerTab t{dev, P, plan->M, v};
    PPS_CUDA_TRY(cudaMalloc(&t.d_vec, vec.size() * sizeof(uint16_t)));
    PPS_CUDA_TRY(cudaMalloc(&t.d_off, off.size() * sizeof(int)));
    PPS_CUDA_TRY(cudaMemcpy(t.d_vec, vec.data(), vec.size() * sizeof(uint16_t), cudaMemcpyHostToDevice));
    PPS_CUDA_TRY(cudaMemcpy(t.d_off, off.data(), off.size() * sizeof(int), cudaMemcpyHostToDevice));
    g_ledger.push_back(t);
    *out = &g_ledger.back();
    return PP_OK;
}

}  // namespace
}  // namespace pps

extern "C" int pp_sched_partition_search_interleaved(const int32_t *layer_tf, const int32_t *layer_tb,
                                                     const int64_t *layer_act, int L, int P, int v, int M,
                                                     int32_t comm, int64_t act_cap, uint64_t seed,
                                                     int64_t cand_begin, int64_t n_cand, int64_t *best_idx,
                                                     int32_t *best_makespan, int32_t *best_cuts,
                                                     int32_t *all_makespan, cudaStream_t stream) {
    using namespace pps;
    if (!layer_tf || !layer_tb || !layer_act || !best_idx) return PP_ERR_ARG;
    if (P < 1 || v < 2 || M < 1 || n_cand < 0 || cand_begin < 0 || comm < 0) return PP_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(best_idx) & 7) != 0) return PP_ERR_ARG;
    const int S = P * v;
    if (P > PP_MAX_P || S > PP_MAX_S || L > kIlvMaxL || (int64_t)M * v > PP_MAX_MV || n_cand >= (int64_t)1 << 32)
        return PP_ERR_SIZE;
    if (L < S) return PP_ERR_ARG;
    if (M % P != 0) return PP_ERR_DIVISIBILITY;
    const uint64_t ncomb = binom_u64(L - 1, S - 1);
    if (ncomb == ~0ull || ncomb == 0) return PP_ERR_SIZE;
    pp_plan *plan = nullptr;
    int rc = cached_plan(PP_INTERLEAVED_1F1B, P, M, v, stream, &plan);
    if (rc) return rc;

    std::lock_guard<std::mutex> lk(g_ilv_mu);
    const int cn = (int)std::min<int64_t>(kChunk, std::max<int64_t>(32, (n_cand + 31) / 32 * 32));
    const size_t cost_bytes = (size_t)S * cn * sizeof(int32_t);
    const size_t need = 2 * cost_bytes + (size_t)cn * (2 * sizeof(int32_t) + 2) + 512;
    void *scratch = nullptr;
    rc = ilv_scratch(need, &scratch);
    if (rc) return rc;
    unsigned char *base = static_cast<unsigned char *>(scratch);
    int32_t *cf = reinterpret_cast<int32_t *>(base);
    int32_t *cb = reinterpret_cast<int32_t *>(base + cost_bytes);
    int32_t *mk = reinterpret_cast<int32_t *>(base + 2 * cost_bytes);
    int32_t *dcomm = mk + cn;  // one word, broadcast to every instance and boundary
    int8_t *st = reinterpret_cast<int8_t *>(dcomm + 4);
    int8_t *flag = st + cn;
    int *slot = reinterpret_cast<int *>((reinterpret_cast<uintptr_t>(flag + cn) + 255) & ~(uintptr_t)255);
    int *count = slot + cn;

    IlvArgs a;
    a.ltf = layer_tf; a.ltb = layer_tb; a.lact = layer_act;
    a.L = L; a.P = P; a.v = v; a.S = S; a.M = M; a.O = plan->O;
    a.cap = act_cap; a.seed = seed; a.begin = cand_begin; a.ncomb = ncomb;
    a.ops = plan->d_ops; a.cf = cf; a.cb = cb; a.flag = flag; a.cn = cn;
    a.slot = slot; a.count = count; a.comm = comm; a.prune = all_makespan == nullptr;
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    const LedgerTab *lt = nullptr;
    rc = ledger_tab(plan, dev, &lt);
    if (rc) return rc;
    a.lvec = lt->d_vec; a.loff = lt->d_off;
    const size_t smem = ilv_smem(L, S);
    static std::atomic<bool> attr_set[64];  // per device, set once (idempotent)
    if (dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
        PPS_CUDA_TRY(cudaFuncSetAttribute(k_ilv_cands, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
        PPS_CUDA_TRY(cudaFuncSetAttribute(k_ilv_finish, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
        attr_set[dev].store(true, std::memory_order_release);
    }
    unsigned long long *key = reinterpret_cast<unsigned long long *>(best_idx);
    a.key = key;
    PPS_CUDA_TRY(cudaMemsetAsync(best_idx, 0xFF, sizeof(int64_t), stream));
    PPS_CUDA_TRY(cudaMemcpyAsync(dcomm, &comm, sizeof(int32_t), cudaMemcpyHostToDevice, stream));

    EvalArgs e{};
    e.desc = plan->d_desc; e.desc2 = plan->d_desc2; e.rw = plan->d_rw; e.seg = plan->d_seg; e.nseg = plan->nseg;
    e.R = plan->R; e.P = P; e.M = M; e.v = v; e.S = S; e.O = plan->O; e.nslots = plan->nslots;
    e.cost_f = cf; e.cost_b = cb; e.s_inst = 1; e.s_stage = cn; e.s_mb = 0;
    e.comm = dcomm; e.c_inst = 0; e.c_bnd = 0;
    e.makespan = mk; e.status = st;
    for (int64_t c0 = 0; c0 < n_cand; c0 += cn) {
        const int nc = (int)std::min<int64_t>(cn, n_cand - c0);
        const unsigned blocks = (unsigned)((nc + 255) / 256);
        // a grid-stride loop over the chunk: a few CTAs per SM, each building
        // its binomial and prefix tables once for many candidates
        const unsigned cand_blocks = std::min<unsigned>(blocks, (unsigned)sm_count(dev) * 4u);
        PPS_CUDA_TRY(cudaMemsetAsync(count, 0, sizeof(int), stream));
        k_ilv_cands<<<cand_blocks, 256, smem, stream>>>(a, c0, nc);
        PPS_CUDA_TRY(cudaGetLastError());
        // only the packed candidates that passed the cap (and the bound) are scored
        int scored = 0;
        PPS_CUDA_TRY(cudaMemcpyAsync(&scored, count, sizeof(int), cudaMemcpyDeviceToHost, stream));
        PPS_CUDA_TRY(cudaStreamSynchronize(stream));
        if (scored > 0) {
            e.n = scored;
            rc = lane_path(plan, e) ? launch_eval_lane(plan, e, true, false, stream)
                                    : launch_eval_slot(plan, e, true, false, stream);
            if (rc) return rc;
        }
        k_ilv_select<<<blocks, 256, 0, stream>>>(mk, st, flag, slot, nc, c0, all_makespan, key);
        PPS_CUDA_TRY(cudaGetLastError());
    }
    k_ilv_finish<<<1, 64, smem, stream>>>(a, key, best_idx, best_makespan, best_cuts);
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}
