// plan.cu -- the schedule plan, built on the GPU once per (policy, P, M, v).
//
// Steps (all kernels below):
//   1. k_order: one thread per (device k, position j) writes the op from the
//      policy's rules, and the inverse map (kind, virtual stage, microbatch) ->
//      position.
//   2. k_rounds: each op's wavefront round, i.e. its start tick when every op
//      takes one tick and comm is 0: round = max(previous op on the device,
//      the op it depends on) + 1.  Rounds are a topological order of the
//      dependency graph, so evaluating ops round by round is valid for any
//      costs.  One lane per device walks its order; a lane advances while the
//      op it depends on already has its round.  Each pass either advances some
//      lane or proves the order cyclic (deadlock), so the loop is bounded.
//   3. k_desc: scatter ops into the per-round table [round][device].
//   4. k_peak: the held-activation ledger per device ("2. 1F1B" §4.1 table:
//      +1 at each F, -1 at each B, peak = running maximum).
//   5. k_latest (GPipe/1F1B): checks that every input an op reads is the latest
//      result of its kind on the neighbouring device at the start of its round,
//      which lets the fast evaluator keep one register per (device, kind).
//   6. k_slots (interleaved, or when 5 fails): greedy interval colouring of
//      the in-flight results onto value slots for the generic evaluator.
#include <algorithm>
#include <cstdio>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>
#include <vector>

#include "internal.cuh"

namespace pps {

namespace {

constexpr uint32_t kOpB = 0x80000000u;  // PP_OP kind bit

// The op at position j of device k, as a PP_OP-packed word.  Rules:
//  GPipe: "Pipeline scheduling" (M040) §02 -- all F, then B from the last
//    microbatch back to the first (GPipe FIFO: B from the first to the last).
//  1F1B: "2. 1F1B" §2.3 and §3.2 -- P-k forwards (at most M), then B,F pairs
//    with the oldest outstanding backward first, then the remaining B.
//  Interleaved: device k holds chunks c (virtual stage c*P+k); warmup
//    2(P-k-1)+(v-1)P forwards, then F,B pairs, then the remaining B; forward j
//    runs chunk (j mod Pv)/P of microbatch (j/(Pv))*P + j mod P and backward j
//    runs chunk v-1-(j mod Pv)/P of the same microbatch.
__device__ uint32_t op_at(int policy, int P, int M, int v, int k, int j) {
    auto F = [](uint32_t c, uint32_t i) { return (c << 24) | i; };
    auto B = [](uint32_t c, uint32_t i) { return kOpB | (c << 24) | i; };
    if (policy == PP_GPIPE) {
        return j < M ? F(0, j) : B(0, 2 * M - 1 - j);
    }
    if (policy == PP_GPIPE_FIFO) {
        return j < M ? F(0, j) : B(0, j - M);
    }
    if (policy == PP_1F1B) {
        int w = min(P - k, M);
        if (j < w) return F(0, j);
        int t = j - w;
        if (t < 2 * (M - w)) return (t & 1) ? F(0, w + (t >> 1)) : B(0, t >> 1);
        return B(0, M - w + (t - 2 * (M - w)));
    }
    // interleaved
    int total = M * v;
    int w = min(2 * (P - k - 1) + (v - 1) * P, total);
    int grp = P * v;
    auto fwd = [&](int x) { return F((x % grp) / P, (x / grp) * P + x % P); };
    auto bwd = [&](int x) { return B(v - 1 - (x % grp) / P, (x / grp) * P + x % P); };
    if (j < w) return fwd(j);
    int t = j - w;
    if (t < 2 * (total - w)) return (t & 1) ? bwd(t >> 1) : fwd(w + (t >> 1));
    return bwd(total - w + (t - 2 * (total - w)));
}

__device__ inline int op_kind(uint32_t op) { return op >> 31; }            // 0 F, 1 B
__device__ inline int op_chunk(uint32_t op) { return (op >> 24) & 0x7F; }
__device__ inline int op_mb(uint32_t op) { return op & 0xFFFFFF; }
__device__ inline int64_t pos_key(int kind, int s, int mb, int S, int M) {
    return ((int64_t)kind * S + s) * M + mb;
}

// Word e of the register evaluator's tables for one stride pair (see k_ktab).
__device__ uint32_t ktab_word(const uint32_t *desc, const uint64_t *rw, const uint4 *seg, int R, int P, int pmax,
                              int s_stage, int s_mb, int e) {
    const int tw = (R * pmax + 3) & ~3;
    const int rw_words = 2 * ((R + 1) & ~1);
    uint32_t v = 0;
    if (e < R * pmax) {
        const uint32_t d = desc[e];
        const uint32_t kind = desc_kind(d);
        v = 0xFFFFFFFFu;
        if (kind != kIdle) {
            const int st = (int)desc_chunk(d) * P + (e % pmax);
            const uint32_t off = (uint32_t)(st * s_stage + (int)desc_mb(d) * s_mb);
            v = (off << 1) | (kind == kBwd ? 1u : 0u);
        }
    } else if (e >= tw && e < tw + rw_words) {
        const int q = e - tw;
        if (q / 2 < R) v = (q & 1) ? (uint32_t)(rw[q / 2] >> 32) : (uint32_t)rw[q / 2];
    } else if (e >= tw + rw_words) {
        const int q = e - tw - rw_words;
        const uint4 sg = seg[q / 4];
        const int c = q % 4;
        v = c == 0 ? sg.x : (c == 1 ? sg.y : (c == 2 ? sg.z : sg.w));
    }
    return v;
}

// One shape of a batched plan build (device-side record).
struct BuildJob {
    int policy, P, M, v, pmax, R;
    uint32_t *ops;
    int32_t *pos;      // inverse of ops; reused as slot_of in the value-slot step
    int32_t *round;
    int32_t *info;     // 8 words, as in the single-shape kernels
    int32_t *peak;
    uint32_t *desc;
    uint64_t *rw;
    uint4 *seg;
    uint32_t *desc2;
    int32_t *slot_of;
    uint8_t *lslot;
};

// ---------------------------------------------------------------------------
// Kernel bodies.  Each step is a device function over one shape's tables; the
// single-shape kernels (k_*) and the batched kernels over many shapes (kb_*,
// one BuildJob per shape, blockIdx.y or the thread index picks the shape)
// are thin wrappers around them.
// ---------------------------------------------------------------------------

__device__ void order_one(int policy, int P, int M, int v, uint32_t *ops, int32_t *pos, int64_t t) {
    const int O = 2 * M * v, S = P * v;
    const int k = (int)(t / O), j = (int)(t % O);
    const uint32_t op = op_at(policy, P, M, v, k, j);
    ops[t] = op;
    pos[pos_key(op_kind(op), op_chunk(op) * P + k, op_mb(op), S, M)] = j;
}

// info[0] = rounds, info[1] = 1 on deadlock.  Run by one warp; P <= 32; pub
// is 32 ints of the warp's shared memory.
__device__ void rounds_warp(const uint32_t *ops, const int32_t *pos, int P, int M, int v, int32_t *round,
                            int32_t *info, int *pub) {
    const int O = 2 * M * v, S = P * v;
    const int k = threadIdx.x & 31;
    const bool active = k < P;
    int cur = 0, rprev = -1;
    pub[k] = active ? 0 : O;
    __syncwarp();
    const int64_t limit = (int64_t)P * O + 2;
    bool dead = false;
    for (int64_t it = 0; it < limit; ++it) {
        bool moved = false;
        while (active && cur < O) {
            uint32_t op = ops[k * O + cur];
            int kd = op_kind(op), s = op_chunk(op) * P + k, mb = op_mb(op);
            int ddev = -1, dj = 0;
            if (kd == 0 && s > 0) { ddev = (s - 1) % P; dj = pos[pos_key(0, s - 1, mb, S, M)]; }
            if (kd == 1 && s < S - 1) { ddev = (s + 1) % P; dj = pos[pos_key(1, s + 1, mb, S, M)]; }
            if (kd == 1 && pos[pos_key(0, s, mb, S, M)] >= cur) break;  // its own F not yet run
            int rd = -1;
            if (ddev >= 0) {
                int avail = (ddev == k) ? cur : pub[ddev];
                if (dj >= avail) break;
                rd = round[ddev * O + dj];
            }
            int r = max(rprev + 1, rd + 1);
            round[k * O + cur] = r;
            rprev = r;
            ++cur;
            moved = true;
        }
        __syncwarp();
        if (active) pub[k] = cur;
        __syncwarp();
        bool any = __any_sync(0xffffffffu, moved);
        bool all = __all_sync(0xffffffffu, !active || cur == O);
        if (all) break;
        if (!any) { dead = true; break; }
    }
    int rmax = rprev;
    for (int o = 16; o > 0; o >>= 1) rmax = max(rmax, __shfl_xor_sync(0xffffffffu, rmax, o));
    if (k == 0) {
        info[0] = rmax + 1;
        info[1] = dead ? 1 : 0;
    }
}

__device__ void desc_one(const uint32_t *ops, const int32_t *round, int P, int M, int v, int pmax, uint32_t *desc,
                         int64_t t) {
    const int O = 2 * M * v;
    const int k = (int)(t / O);
    const uint32_t op = ops[t];
    desc[(int64_t)round[t] * pmax + k] =
        desc_pack(op_kind(op) ? kBwd : kFwd, (uint32_t)op_chunk(op), (uint32_t)op_mb(op));
}

// Round r: pack the devices' kinds and classify the round.
__device__ void rwords_one(const uint32_t *desc, int P, int pmax, uint64_t *rw, int r) {
    uint32_t kinds = 0, mask = 0;
    bool allF = true, allB = true, altA = true, altB = true;
    for (int k = 0; k < pmax; ++k) {
        uint32_t kd = desc_kind(desc[(int64_t)r * pmax + k]);
        kinds |= kd << (2 * k);
        if (kd == kIdle) continue;
        mask |= 1u << k;
        allF &= kd == kFwd;
        allB &= kd == kBwd;
        altA &= kd == ((k & 1) ? kBwd : kFwd);
        altB &= kd == ((k & 1) ? kFwd : kBwd);
    }
    uint32_t pat = kPatGeneric;
    if (mask) {
        if (allF) pat = kPatAllF;
        else if (allB) pat = kPatAllB;
        else if (altA) pat = kPatAltA;
        else if (altB) pat = kPatAltB;
        if (pat != kPatGeneric && (P != pmax || mask != (1u << pmax) - 1u)) pat += kPatMasked;
    }
    rw[r] = (uint64_t)kinds | ((uint64_t)pat << 32) | ((uint64_t)mask << 48);
}

// Cut the rounds into segments (one thread).  info[6] = segment count.
__device__ void segments_one(const uint64_t *rw, int R, uint4 *seg, int32_t *info) {
    int n = 0, r = 0;
    while (r < R) {
        const uint32_t pat = rw_pattern(rw[r]);
        const int r0 = r;
        uint32_t type = kSegRound;
        if (pat == kPatAltA || pat == kPatAltB) {
            uint32_t expect = pat;
            while (r < R && rw_pattern(rw[r]) == expect) {
                ++r;
                expect = expect == kPatAltA ? kPatAltB : kPatAltA;
            }
            type = pat == kPatAltA ? kSegAltA : kSegAltB;
        } else if (pat == kPatAllF || pat == kPatAllB) {
            while (r < R && rw_pattern(rw[r]) == pat) ++r;
            type = pat == kPatAllF ? kSegAllF : kSegAllB;
        } else {
            ++r;
        }
        seg[n++] = make_uint4(type, (uint32_t)r0, (uint32_t)r, 0u);
    }
    info[6] = n;
}

// The held-activation ledger of device k ("2. 1F1B" §4.1 table).
__device__ void peak_one(const uint32_t *ops, int O, int32_t *peak, int k) {
    int held = 0, pk = 0;
    for (int j = 0; j < O; ++j) {
        held += op_kind(ops[k * O + j]) ? -1 : 1;
        pk = max(pk, held);
    }
    peak[k] = pk;
}

// v == 1 only.  info[2] |= 1 if the input of op t is not the latest result of
// its kind on the producing device at the start of the consumer's round.
__device__ void latest_one(const uint32_t *ops, const int32_t *pos, const int32_t *round, int P, int M,
                           int32_t *info, int64_t t) {
    const int O = 2 * M, S = P;
    const int k = (int)(t / O), j = (int)(t % O);
    const uint32_t op = ops[t];
    const int kd = op_kind(op), mb = op_mb(op);
    int cdev;
    if (kd == 0 && k < P - 1) cdev = k + 1;
    else if (kd == 1 && k > 0) cdev = k - 1;
    else return;  // no consumer on another device
    const int rc = round[cdev * O + pos[pos_key(kd, cdev, mb, S, M)]];
    for (int q = j + 1; q < O; ++q) {
        if (op_kind(ops[k * O + q]) == kd) {
            if (round[k * O + q] < rc) atomicOr(&info[2], 1);
            break;
        }
    }
}

// Greedy value-slot assignment (one thread).  info[3] = slots used, info[4] = 1
// if more than kMaxValueSlots would be needed, info[5] = 1 if a read slot was
// never assigned.
__device__ void slots_one(const uint32_t *desc, int R, int P, int M, int v, int pmax, int32_t *slot_of,
                          uint32_t *desc2, int32_t *info) {
    const int S = P * v;
    uint64_t used = 0;
    int nmax = 0;
    for (int r = 0; r < R; ++r) {
        uint64_t freed = 0;
        for (int k = 0; k < pmax; ++k) {
            uint32_t d = desc[(int64_t)r * pmax + k];
            uint32_t kind = desc_kind(d);
            if (kind == kIdle) { desc2[(int64_t)r * pmax + k] = d2_pack(kNoSlot, kNoSlot, kNoSlot); continue; }
            int s = (int)desc_chunk(d) * P + k, mb = (int)desc_mb(d);
            uint32_t rs = kNoSlot, cb = kNoSlot, ws = kNoSlot;
            if (kind == kFwd && s > 0) { rs = (uint32_t)slot_of[pos_key(0, s - 1, mb, S, M)]; cb = s - 1; }
            if (kind == kBwd && s < S - 1) { rs = (uint32_t)slot_of[pos_key(1, s + 1, mb, S, M)]; cb = s; }
            if (rs != kNoSlot) {
                if (rs >= (uint32_t)kMaxValueSlots) { info[5] = 1; return; }  // never assigned
                freed |= 1ull << rs;
            }
            bool produces = (kind == kFwd && s < S - 1) || (kind == kBwd && s > 0);
            if (produces) {
                if (used == ~0ull) { info[4] = 1; return; }
                int b = __ffsll((long long)~used) - 1;
                used |= 1ull << b;
                nmax = max(nmax, b + 1);
                ws = (uint32_t)b;
                slot_of[pos_key(kind == kBwd ? 1 : 0, s, mb, S, M)] = b;
            }
            desc2[(int64_t)r * pmax + k] = d2_pack(rs, ws, cb);
        }
        used &= ~freed;
    }
    info[3] = nmax;
}

// Per-consumer value slots for the lane evaluator.  Every in-flight result
// has one consumer op, on device (k+1) mod P for a forward and (k-1) mod P
// for a backward.  The lane evaluator keeps a result in its consumer
// device's column, so results with different consumers never share a cell
// and each consumer device colours only its own inputs; that needs far fewer
// rows than the plan-wide colouring of slots_one.  One warp, lane kc colours
// the inputs of device kc in round order, mapping each in-flight result
// from its plan-wide slot (unique while it is in flight) to a local one, and
// frees a local slot at the end of the round that consumes it.  Writes
// lrd[r][k] (local slot read by op (r,k)) for k = kc, lwr[r][k] (local slot
// op (r,k) writes) for producers whose consumer is kc; 0xFF where none.
// info[7] = local slots used (the maximum over devices), -1 on exhaustion.
// loc is the warp's [32][kMaxValueSlots] bytes of shared memory.
__device__ void cslots_warp(const uint32_t *desc, const uint32_t *desc2, int R, int P, int pmax, uint8_t *lrd,
                            uint8_t *lwr, int32_t *info, uint8_t (*loc)[kMaxValueSlots]) {
    const int kc = threadIdx.x & 31;
    uint64_t used = 0;
    int nmax = 0;
    bool bad = false;
    if (kc < P) {
        for (int r = 0; r < R && !bad; ++r) {
            uint64_t freed = 0;
            const int64_t row = (int64_t)r * pmax;
            uint8_t rd = 0xFF;
            if (desc_kind(desc[row + kc]) != kIdle) {
                const uint32_t rs = d2_rslot(desc2[row + kc]);
                if (rs != kNoSlot) {
                    rd = loc[kc][rs];
                    freed |= 1ull << rd;
                }
            }
            lrd[row + kc] = rd;
            for (int k = 0; k < P; ++k) {
                const uint32_t kind = desc_kind(desc[row + k]);
                if (kind == kIdle) continue;
                const uint32_t ws = d2_wslot(desc2[row + k]);
                if (ws == kNoSlot) continue;
                const int cons = kind == kFwd ? (k + 1) % P : (k + P - 1) % P;
                if (cons != kc) continue;
                if (used == ~0ull) { bad = true; break; }
                const int b = __ffsll((long long)~used) - 1;
                used |= 1ull << b;
                nmax = max(nmax, b + 1);
                loc[kc][ws] = (uint8_t)b;
                lwr[row + k] = (uint8_t)b;
            }
            used &= ~freed;
        }
    }
    const unsigned any_bad = __ballot_sync(0xFFFFFFFFu, bad);
#pragma unroll
    for (int m = 16; m; m >>= 1) nmax = max(nmax, __shfl_xor_sync(0xFFFFFFFFu, nmax, m));
    if ((threadIdx.x & 31) == 0) info[7] = any_bad ? -1 : nmax;
}

// ---- single-shape kernels ----

__global__ void k_order(int policy, int P, int M, int v, uint32_t *ops, int32_t *pos) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t < (int64_t)P * 2 * M * v) order_one(policy, P, M, v, ops, pos, t);
}

__global__ void k_rounds(const uint32_t *ops, const int32_t *pos, int P, int M, int v, int32_t *round,
                         int32_t *info) {
    __shared__ int pub[32];
    rounds_warp(ops, pos, P, M, v, round, info, pub);
}

__global__ void k_desc(const uint32_t *ops, const int32_t *round, int P, int M, int v, int pmax, uint32_t *desc) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t < (int64_t)P * 2 * M * v) desc_one(ops, round, P, M, v, pmax, desc, t);
}

__global__ void k_rwords(const uint32_t *desc, int R, int P, int pmax, uint64_t *rw) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r < R) rwords_one(desc, P, pmax, rw, r);
}

__global__ void k_segments(const uint64_t *rw, int R, uint4 *seg, int32_t *info) {
    if (threadIdx.x == 0 && blockIdx.x == 0) segments_one(rw, R, seg, info);
}

__global__ void k_peak(const uint32_t *ops, int P, int O, int32_t *peak) {
    if ((int)threadIdx.x < P) peak_one(ops, O, peak, threadIdx.x);
}

__global__ void k_latest(const uint32_t *ops, const int32_t *pos, const int32_t *round, int P, int M,
                         int32_t *info) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t < (int64_t)P * 2 * M) latest_one(ops, pos, round, P, M, info, t);
}

__global__ void k_slots(const uint32_t *desc, int R, int P, int M, int v, int pmax, int32_t *slot_of,
                        uint32_t *desc2, int32_t *info) {
    if (threadIdx.x == 0 && blockIdx.x == 0) slots_one(desc, R, P, M, v, pmax, slot_of, desc2, info);
}

__global__ void k_cslots(const uint32_t *desc, const uint32_t *desc2, int R, int P, int pmax, uint8_t *lrd,
                         uint8_t *lwr, int32_t *info) {
    __shared__ uint8_t loc[32][kMaxValueSlots];
    cslots_warp(desc, desc2, R, P, pmax, lrd, lwr, info, loc);
}

// Fill the register evaluator's tables for one stride pair: loader table
// entries (element offset of the op's cost row, shifted left by one, bit 0 set
// for a backward op; all ones for an idle slot), then the round words, then
// the segments.
__global__ void k_ktab(const uint32_t *desc, const uint64_t *rw, const uint4 *seg, int R, int P, int pmax,
                       int nseg, int s_stage, int s_mb, uint32_t *out) {
    const int total = ktab_words(R, pmax, nseg);
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x)
        out[e] = ktab_word(desc, rw, seg, R, P, pmax, s_stage, s_mb, e);
}

// ---- batched kernels: one BuildJob per shape ----

// Element t of shape j's [P][O] tables, for t in the grid's stride over them.
#define PPS_JOB_LOOP(n)                                                                          \
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, n_ = (n); t < n_;           \
         t += (int64_t)gridDim.x * blockDim.x)

__global__ void kb_order(const BuildJob *jobs) {
    const BuildJob &b = jobs[blockIdx.y];
    PPS_JOB_LOOP((int64_t)b.P * 2 * b.M * b.v) order_one(b.policy, b.P, b.M, b.v, b.ops, b.pos, t);
}

__global__ void kb_rounds(const BuildJob *jobs) {
    __shared__ int pub[32];
    const BuildJob &b = jobs[blockIdx.x];
    rounds_warp(b.ops, b.pos, b.P, b.M, b.v, b.round, b.info, pub);
}

// desc, the ledger peak and (v == 1) the latest-result check, all from the
// op order and the rounds.
__global__ void kb_desc(const BuildJob *jobs) {
    const BuildJob &b = jobs[blockIdx.y];
    const int O = 2 * b.M * b.v;
    PPS_JOB_LOOP((int64_t)b.P * O) {
        desc_one(b.ops, b.round, b.P, b.M, b.v, b.pmax, b.desc, t);
        if (b.v == 1) latest_one(b.ops, b.pos, b.round, b.P, b.M, b.info, t);
    }
    if (blockIdx.x == 0 && (int)threadIdx.x < b.P) peak_one(b.ops, O, b.peak, threadIdx.x);
}

__global__ void kb_rwords(const BuildJob *jobs) {
    const BuildJob &b = jobs[blockIdx.y];
    PPS_JOB_LOOP(b.R) rwords_one(b.desc, b.P, b.pmax, b.rw, (int)t);
}

__global__ void kb_segments(const BuildJob *jobs, int njobs) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j < njobs) segments_one(jobs[j].rw, jobs[j].R, jobs[j].seg, jobs[j].info);
}

__global__ void kb_slots(const BuildJob *jobs, int njobs) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= njobs) return;
    const BuildJob &b = jobs[j];
    slots_one(b.desc, b.R, b.P, b.M, b.v, b.pmax, b.slot_of, b.desc2, b.info);
}

__global__ void kb_cslots(const BuildJob *jobs) {
    __shared__ uint8_t loc[32][kMaxValueSlots];
    const BuildJob &b = jobs[blockIdx.x];
    if (b.info[4] || b.info[5]) return;  // the plan-wide colouring failed: desc2 is incomplete
    const int64_t cells = (int64_t)b.R * b.pmax;
    cslots_warp(b.desc, b.desc2, b.R, b.P, b.pmax, b.lslot, b.lslot + cells, b.info, loc);
}

__global__ void kb_ktab(const TableJob *jobs) {
    const TableJob &b = jobs[blockIdx.y];
    PPS_JOB_LOOP(b.words) b.out[t] = ktab_word(b.desc, b.rw, b.seg, b.R, b.P, b.pmax, b.s_stage, b.s_mb, (int)t);
}
#undef PPS_JOB_LOOP

struct DevBuf {
    void *p = nullptr;
    ~DevBuf() { if (p) cudaFree(p); }
    template <class T> T *as() { return static_cast<T *>(p); }
};

}  // namespace

int cuda_status(cudaError_t e) {
    (void)cudaGetLastError();
    (void)e;
    return PP_ERR_CUDA;
}

int check_shape(int policy, int P, int M, int v) {
    if (policy != PP_GPIPE && policy != PP_1F1B && policy != PP_INTERLEAVED_1F1B && policy != PP_GPIPE_FIFO)
        return PP_ERR_ARG;
    if (P < 1 || M < 1 || v < 1) return PP_ERR_ARG;
    if (policy != PP_INTERLEAVED_1F1B && v != 1) return PP_ERR_ARG;
    if (policy == PP_INTERLEAVED_1F1B && v < 2) return PP_ERR_ARG;
    if (P > PP_MAX_P || (int64_t)P * v > PP_MAX_S || (int64_t)M * v > PP_MAX_MV) return PP_ERR_SIZE;
    if (policy == PP_INTERLEAVED_1F1B && M % P != 0) return PP_ERR_DIVISIBILITY;
    return PP_OK;
}

// Value slots of a plan: the plan-wide colouring (k_slots, for the generic
// slot evaluator) and the per-consumer one (k_cslots, for the lane
// evaluator).  Allocates *desc2 [R][pmax] and *lslot [2][R][pmax]; returns
// PP_ERR_SIZE when more than kMaxValueSlots results would be in flight.
static int build_slots(const uint32_t *desc, int R, int P, int M, int v, int pmax, cudaStream_t st,
                       uint32_t **desc2_out, uint8_t **lslot_out, int *nslots, int *nlslots) {
    const int64_t npos = 2LL * P * v * M;
    const int64_t cells = (int64_t)R * pmax;
    DevBuf desc2, slot_of, info, lslot;
    int32_t h_info[8];
    PPS_CUDA_TRY(cudaMalloc(&info.p, 8 * sizeof(int32_t)));
    PPS_CUDA_TRY(cudaMemsetAsync(info.p, 0, 8 * sizeof(int32_t), st));
    PPS_CUDA_TRY(cudaMalloc(&desc2.p, cells * sizeof(uint32_t)));
    PPS_CUDA_TRY(cudaMalloc(&slot_of.p, npos * sizeof(int32_t)));
    PPS_CUDA_TRY(cudaMemsetAsync(slot_of.p, 0xFF, npos * sizeof(int32_t), st));
    k_slots<<<1, 32, 0, st>>>(desc, R, P, M, v, pmax, slot_of.as<int32_t>(), desc2.as<uint32_t>(),
                              info.as<int32_t>());
    PPS_CUDA_TRY(cudaGetLastError());
    PPS_CUDA_TRY(cudaMemcpyAsync(h_info, info.p, sizeof(h_info), cudaMemcpyDeviceToHost, st));
    PPS_CUDA_TRY(cudaStreamSynchronize(st));
    if (h_info[5]) return PP_ERR_INTERNAL;
    if (h_info[4]) return PP_ERR_SIZE;
    // per-consumer slots of the lane evaluator: lrd then lwr, [R][pmax] bytes each
    PPS_CUDA_TRY(cudaMalloc(&lslot.p, 2 * cells));
    PPS_CUDA_TRY(cudaMemsetAsync(lslot.p, 0xFF, 2 * cells, st));
    k_cslots<<<1, 32, 0, st>>>(desc, desc2.as<uint32_t>(), R, P, pmax, lslot.as<uint8_t>(),
                               lslot.as<uint8_t>() + cells, info.as<int32_t>());
    PPS_CUDA_TRY(cudaGetLastError());
    PPS_CUDA_TRY(cudaMemcpyAsync(h_info, info.p, sizeof(h_info), cudaMemcpyDeviceToHost, st));
    PPS_CUDA_TRY(cudaStreamSynchronize(st));
    if (h_info[7] < 0) return PP_ERR_INTERNAL;
    *nslots = h_info[3];
    *nlslots = h_info[7];
    *desc2_out = desc2.as<uint32_t>(); desc2.p = nullptr;
    *lslot_out = lslot.as<uint8_t>(); lslot.p = nullptr;
    return PP_OK;
}

namespace {

int64_t pad4(int64_t w) { return (w + 3) & ~(int64_t)3; }

// A device allocation in 32-bit words, freed on scope exit unless handed over.
struct Arena {
    pp_arena *a = nullptr;
    ~Arena() {
        if (a) {
            if (a->base) cudaFree(a->base);
            delete a;
        }
    }
    int alloc(int64_t words) {
        a = new pp_arena;
        const cudaError_t e = cudaMalloc(&a->base, (size_t)std::max<int64_t>(words, 4) * sizeof(uint32_t));
        if (e != cudaSuccess) {
            a->base = nullptr;
            return cuda_status(e);
        }
        return PP_OK;
    }
    uint32_t *w() const { return static_cast<uint32_t *>(a->base); }
};

// Upload jobs[0..n) to d (device) and run launch(first, count) over chunks of
// at most 65,535 shapes (a grid dimension's limit).
template <class T, class F>
int for_chunks(const std::vector<T> &jobs, T *d, cudaStream_t st, F launch) {
    PPS_CUDA_TRY(cudaMemcpyAsync(d, jobs.data(), jobs.size() * sizeof(T), cudaMemcpyHostToDevice, st));
    const int n = (int)jobs.size();
    for (int j0 = 0; j0 < n; j0 += 65535) launch(d + j0, std::min(65535, n - j0));
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}

// Blocks along x for a grid-stride loop over at most `elems` elements per shape.
unsigned grid_x(int64_t elems) {
    return (unsigned)std::min<int64_t>(1024, std::max<int64_t>(1, (elems + 255) / 256));
}

// The build's temporary words (inverse op positions, info words, job records):
// one grow-only buffer per device, kept for the process, so a build neither
// allocates nor frees it again (a free would synchronize the device).  Builds
// hold g_build_mu while they use it.
std::mutex g_build_mu;
struct TempBuf {
    void *p = nullptr;
    size_t bytes = 0;
};
TempBuf g_temp[64];

int temp_words(int64_t words, uint32_t **out) {
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return PP_ERR_INTERNAL;
    TempBuf &t = g_temp[dev];
    const size_t need = (size_t)std::max<int64_t>(words, 4) * sizeof(uint32_t);
    if (t.bytes < need) {
        if (t.p) PPS_CUDA_TRY(cudaFree(t.p));
        t.p = nullptr;
        t.bytes = 0;
        const size_t grow = std::max(need, (size_t)1 << 20);
        PPS_CUDA_TRY(cudaMalloc(&t.p, grow));
        t.bytes = grow;
    }
    *out = static_cast<uint32_t *>(t.p);
    return PP_OK;
}

void arena_ref(pp_arena *a) {
    if (a) a->refs.fetch_add(1);
}

void arena_release(pp_arena *a) {
    if (a && a->refs.fetch_sub(1) == 1) {
        cudaFree(a->base);
        delete a;
    }
}

}  // namespace

int build_plans(const PlanShape *shapes, int n, cudaStream_t st, pp_plan **out) {
    if (n <= 0) return PP_OK;
    for (int i = 0; i < n; ++i) {
        out[i] = nullptr;
        const int rc = check_shape(shapes[i].policy, shapes[i].P, shapes[i].M, shapes[i].v);
        if (rc) return rc;
    }
    int device = 0;
    PPS_CUDA_TRY(cudaGetDevice(&device));
    std::vector<BuildJob> jobs(n);

    // Step 1: op order and rounds.  Persistent: ops, rounds, peaks (all peaks
    // together, copied out at once); temporary: pos, info (together), the
    // job records.
    int64_t wA = 0, wT = 0, max_ops = 0, npeak = 0;
    std::vector<int64_t> offA(n), offT(n);
    for (int i = 0; i < n; ++i) {
        const PlanShape &sh = shapes[i];
        const int64_t nops = (int64_t)sh.P * 2 * sh.M * sh.v;
        offA[i] = wA;
        wA += 2 * pad4(nops);
        offT[i] = wT;
        wT += pad4(nops);  // pos: 2*S*M entries = P*O
        max_ops = std::max(max_ops, nops);
        npeak += sh.P;
    }
    const int64_t peak_at = wA, info_at = wT;
    wA += pad4(npeak);
    wT += 8LL * n;
    const int64_t jobs_at = pad4(wT);
    wT = jobs_at + pad4((int64_t)n * (int64_t)sizeof(BuildJob) / 4 + 1);
    std::lock_guard<std::mutex> build_lock(g_build_mu);
    Arena A, B, C;
    uint32_t *Tw = nullptr;
    int rc = A.alloc(wA);
    if (!rc) rc = temp_words(wT, &Tw);
    if (rc) return rc;
    BuildJob *d_jobs = reinterpret_cast<BuildJob *>(Tw + jobs_at);
    int64_t pk = 0;
    for (int i = 0; i < n; ++i) {
        const PlanShape &sh = shapes[i];
        const int64_t nops = (int64_t)sh.P * 2 * sh.M * sh.v;
        BuildJob &b = jobs[i];
        b = BuildJob{};
        b.policy = sh.policy; b.P = sh.P; b.M = sh.M; b.v = sh.v; b.pmax = pmax_for(sh.P);
        b.ops = A.w() + offA[i];
        b.round = reinterpret_cast<int32_t *>(A.w() + offA[i] + pad4(nops));
        b.peak = reinterpret_cast<int32_t *>(A.w() + peak_at + pk);
        pk += sh.P;
        b.pos = reinterpret_cast<int32_t *>(Tw + offT[i]);
        b.info = reinterpret_cast<int32_t *>(Tw + info_at) + 8LL * i;
    }
    PPS_CUDA_TRY(cudaMemsetAsync(Tw + info_at, 0, 8LL * n * sizeof(int32_t), st));
    rc = for_chunks(jobs, d_jobs, st, [&](BuildJob *d, int c) {
        kb_order<<<dim3(grid_x(max_ops), c), 256, 0, st>>>(d);
        kb_rounds<<<c, 32, 0, st>>>(d);
    });
    if (rc) return rc;
    std::vector<int32_t> h_info(8LL * n);
    PPS_CUDA_TRY(cudaMemcpyAsync(h_info.data(), Tw + info_at, h_info.size() * sizeof(int32_t),
                                 cudaMemcpyDeviceToHost, st));
    PPS_CUDA_TRY(cudaStreamSynchronize(st));

    // Step 2: per-round tables, peaks, the latest-result check, segments.
    int64_t wB = 0, max_R = 0;
    std::vector<int64_t> offB(n);
    for (int i = 0; i < n; ++i) {
        if (h_info[8 * i + 1]) return PP_ERR_DEADLOCK;
        const int R = h_info[8 * i];
        if (R < 1) return PP_ERR_INTERNAL;
        jobs[i].R = R;
        offB[i] = wB;
        // desc [R][pmax]; round words [R + 1] (one spare word so the table can
        // be copied in 16-byte pieces); segments [R]
        wB += pad4((int64_t)R * jobs[i].pmax) + pad4(2LL * (R + 1)) + 4LL * R;
        max_R = std::max<int64_t>(max_R, R);
    }
    rc = B.alloc(wB);
    if (rc) return rc;
    PPS_CUDA_TRY(cudaMemsetAsync(B.w(), 0, (size_t)std::max<int64_t>(wB, 4) * sizeof(uint32_t), st));
    for (int i = 0; i < n; ++i) {
        BuildJob &b = jobs[i];
        uint32_t *base = B.w() + offB[i];
        const int64_t dw = pad4((int64_t)b.R * b.pmax);
        b.desc = base;
        b.rw = reinterpret_cast<uint64_t *>(base + dw);
        b.seg = reinterpret_cast<uint4 *>(base + dw + pad4(2LL * (b.R + 1)));
    }
    rc = for_chunks(jobs, d_jobs, st, [&](BuildJob *d, int c) {
        kb_desc<<<dim3(grid_x(max_ops), c), 256, 0, st>>>(d);
        kb_rwords<<<dim3(grid_x(max_R), c), 256, 0, st>>>(d);
        kb_segments<<<(c + 127) / 128, 128, 0, st>>>(d, c);
    });
    if (rc) return rc;
    std::vector<int32_t> h_peak(npeak);
    PPS_CUDA_TRY(cudaMemcpyAsync(h_info.data(), Tw + info_at, h_info.size() * sizeof(int32_t),
                                 cudaMemcpyDeviceToHost, st));
    PPS_CUDA_TRY(cudaMemcpyAsync(h_peak.data(), A.w() + peak_at, npeak * sizeof(int32_t), cudaMemcpyDeviceToHost,
                                 st));
    PPS_CUDA_TRY(cudaStreamSynchronize(st));

    // Step 3: value slots of the plans without the register path.
    std::vector<BuildJob> sjobs;
    std::vector<int> sidx;
    int64_t wC = 0, max_pos = 0;
    std::vector<int64_t> offC(n, -1);
    for (int i = 0; i < n; ++i) {
        const bool reg_ok = jobs[i].v == 1 && h_info[8 * i + 2] == 0;
        if (reg_ok) continue;
        const int64_t cells = (int64_t)jobs[i].R * jobs[i].pmax;
        offC[i] = wC;
        wC += pad4(cells) + pad4((2 * cells + 3) / 4);
        sidx.push_back(i);
    }
    if (!sidx.empty()) {
        rc = C.alloc(wC);
        if (rc) return rc;
        PPS_CUDA_TRY(cudaMemsetAsync(C.w(), 0xFF, (size_t)std::max<int64_t>(wC, 4) * sizeof(uint32_t), st));
        PPS_CUDA_TRY(cudaMemsetAsync(Tw, 0xFF, (size_t)info_at * sizeof(uint32_t), st));  // slot_of := -1
        for (int i : sidx) {
            BuildJob b = jobs[i];
            const int64_t cells = (int64_t)b.R * b.pmax;
            b.desc2 = C.w() + offC[i];
            b.lslot = reinterpret_cast<uint8_t *>(C.w() + offC[i] + pad4(cells));
            b.slot_of = b.pos;
            jobs[i].desc2 = b.desc2;
            jobs[i].lslot = b.lslot;
            sjobs.push_back(b);
            max_pos = std::max<int64_t>(max_pos, 2LL * b.P * b.v * b.M);
        }
        rc = for_chunks(sjobs, d_jobs, st, [&](BuildJob *d, int c) {
            kb_slots<<<(c + 127) / 128, 128, 0, st>>>(d, c);
            kb_cslots<<<c, 32, 0, st>>>(d);
        });
        if (rc) return rc;
        PPS_CUDA_TRY(cudaMemcpyAsync(h_info.data(), Tw + info_at, h_info.size() * sizeof(int32_t),
                                     cudaMemcpyDeviceToHost, st));
        PPS_CUDA_TRY(cudaStreamSynchronize(st));
        for (int i : sidx) {
            const int32_t *f = &h_info[8 * i];
            if (f[5]) return PP_ERR_INTERNAL;
            if (f[4]) return PP_ERR_SIZE;
            if (f[7] < 0) return PP_ERR_INTERNAL;
        }
    }
    (void)max_pos;

    // The plans: each references the arenas its tables live in.
    pk = 0;
    for (int i = 0; i < n; ++i) {
        const BuildJob &b = jobs[i];
        const int32_t *f = &h_info[8 * i];
        pp_plan *p = new pp_plan();
        p->policy = b.policy; p->P = b.P; p->M = b.M; p->v = b.v; p->S = b.P * b.v; p->O = 2 * b.M * b.v;
        p->R = b.R; p->pmax = b.pmax; p->device = device;
        p->reg_ok = b.v == 1 && f[2] == 0;
        p->nseg = f[6];
        p->nslots = p->reg_ok ? 0 : f[3];
        p->nlslots = p->reg_ok ? 0 : f[7];
        p->d_ops = b.ops; p->d_round = b.round; p->d_peak = b.peak;
        p->d_desc = b.desc; p->d_rw = b.rw; p->d_seg = b.seg;
        p->d_desc2 = p->reg_ok ? nullptr : b.desc2;
        p->d_lslot = p->reg_ok ? nullptr : b.lslot;
        p->slots_in_arena = !p->reg_ok;
        for (int k = 0; k < b.P; ++k) p->h_peak[k] = h_peak[pk + k];
        pk += b.P;
        p->arena[0] = A.a; p->arena[1] = B.a; p->arena[2] = p->reg_ok ? nullptr : C.a;
        for (pp_arena *x : p->arena) arena_ref(x);
        out[i] = p;
    }
    A.a = nullptr;  // now owned by the plans
    B.a = nullptr;
    if (!sidx.empty()) C.a = nullptr;
    return PP_OK;
}

static int build_plan(int policy, int P, int M, int v, cudaStream_t st, pp_plan **out) {
    const PlanShape sh{policy, P, M, v};
    return build_plans(&sh, 1, st, out);
}

int plan_value_slots(pp_plan *plan, cudaStream_t stream) {
    std::lock_guard<std::mutex> lk(plan->ktab_mu);
    if (plan->d_lslot) return PP_OK;
    uint32_t *desc2 = nullptr;
    uint8_t *lslot = nullptr;
    int nslots = 0, nlslots = 0;
    const int rc = build_slots(plan->d_desc, plan->R, plan->P, plan->M, plan->v, plan->pmax, stream, &desc2, &lslot,
                               &nslots, &nlslots);
    if (rc) return rc;
    plan->d_desc2 = desc2;
    plan->d_lslot = lslot;
    plan->nslots = nslots;
    plan->nlslots = nlslots;
    return PP_OK;
}

int kernel_tables(pp_plan *plan, int64_t s_stage, int64_t s_mb, cudaStream_t stream, const pp_ktab **out) {
    std::lock_guard<std::mutex> lk(plan->ktab_mu);
    for (const pp_ktab &t : plan->ktabs)
        if (t.s_stage == s_stage && t.s_mb == s_mb) { *out = &t; return PP_OK; }
    pp_ktab t;
    t.s_stage = s_stage;
    t.s_mb = s_mb;
    t.words = ktab_words(plan->R, plan->pmax, plan->nseg);
    PPS_CUDA_TRY(cudaMalloc(&t.d, (size_t)t.words * sizeof(uint32_t)));
    const int blocks = (t.words + 255) / 256;
    k_ktab<<<blocks, 256, 0, stream>>>(plan->d_desc, plan->d_rw, plan->d_seg, plan->R, plan->P, plan->pmax,
                                       plan->nseg, (int)s_stage, (int)s_mb, reinterpret_cast<uint32_t *>(t.d));
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        cudaFree(t.d);
        return cuda_status(e);
    }
    plan->ktabs.push_back(t);
    *out = &plan->ktabs.back();
    return PP_OK;
}

int plan_into(int policy, int P, int M, uint32_t *region, int64_t region_words, cudaStream_t st,
              ScratchPlan *sp) {
    if (policy != PP_GPIPE && policy != PP_1F1B) return PP_ERR_ARG;
    int rc = check_shape(policy, P, M, 1);
    if (rc) return rc;
    const int O = 2 * M, pmax = pmax_for(P);
    const int64_t nops = (int64_t)P * O, npos = 2LL * P * M;
    auto pad4 = [](int64_t w) { return (w + 3) & ~(int64_t)3; };
    int64_t off = 0;
    auto take = [&](int64_t w) {
        uint32_t *p = region + off;
        off += pad4(w);
        return p;
    };
    if (pad4(8) + pad4(P) + 2 * pad4(nops) + pad4(npos) > region_words) return PP_ERR_SIZE;
    int32_t *info = reinterpret_cast<int32_t *>(take(8));
    int32_t *peak = reinterpret_cast<int32_t *>(take(P));
    uint32_t *ops = take(nops);
    int32_t *round = reinterpret_cast<int32_t *>(take(nops));
    int32_t *pos = reinterpret_cast<int32_t *>(take(npos));
    PPS_CUDA_TRY(cudaMemsetAsync(info, 0, 8 * sizeof(int32_t), st));
    const int tpb = 256;
    const unsigned nblk = (unsigned)((nops + tpb - 1) / tpb);
    k_order<<<nblk, tpb, 0, st>>>(policy, P, M, 1, ops, pos);
    k_rounds<<<1, 32, 0, st>>>(ops, pos, P, M, 1, round, info);
    PPS_CUDA_TRY(cudaGetLastError());
    int32_t h_info[8];
    PPS_CUDA_TRY(cudaMemcpyAsync(h_info, info, sizeof(h_info), cudaMemcpyDeviceToHost, st));
    PPS_CUDA_TRY(cudaStreamSynchronize(st));
    if (h_info[1]) return PP_ERR_DEADLOCK;
    const int R = h_info[0];
    if (R < 1) return PP_ERR_INTERNAL;
    if (off + pad4((int64_t)R * pmax) + pad4(2LL * (R + 1)) + pad4(4LL * R) > region_words) return PP_ERR_SIZE;
    uint32_t *desc = take((int64_t)R * pmax);
    uint64_t *rw = reinterpret_cast<uint64_t *>(take(2LL * (R + 1)));
    uint4 *seg = reinterpret_cast<uint4 *>(take(4LL * R));
    PPS_CUDA_TRY(cudaMemsetAsync(desc, 0, (int64_t)R * pmax * sizeof(uint32_t), st));
    PPS_CUDA_TRY(cudaMemsetAsync(rw, 0, (int64_t)(R + 1) * sizeof(uint64_t), st));
    k_desc<<<nblk, tpb, 0, st>>>(ops, round, P, M, 1, pmax, desc);
    k_peak<<<1, 32, 0, st>>>(ops, P, O, peak);
    k_rwords<<<(R + 255) / 256, 256, 0, st>>>(desc, R, P, pmax, rw);
    k_segments<<<1, 32, 0, st>>>(rw, R, seg, info);
    k_latest<<<nblk, tpb, 0, st>>>(ops, pos, round, P, M, info);
    PPS_CUDA_TRY(cudaGetLastError());
    PPS_CUDA_TRY(cudaMemcpyAsync(h_info, info, sizeof(h_info), cudaMemcpyDeviceToHost, st));
    PPS_CUDA_TRY(cudaStreamSynchronize(st));
    if (h_info[2]) return PP_ERR_INTERNAL;  // the register evaluator would not apply
    sp->region = region; sp->region_words = region_words; sp->used_words = off;
    sp->policy = policy; sp->P = P; sp->M = M; sp->R = R; sp->pmax = pmax; sp->nseg = h_info[6];
    sp->desc = desc; sp->rw = rw; sp->seg = seg; sp->peak = peak;
    sp->ktab = nullptr; sp->ktab_words = 0;
    return PP_OK;
}

// The kernel tables go right after the plan's tables (at used_words, which is
// not advanced), so a later call for another stride pair replaces them in place.
int ktab_into(ScratchPlan *sp, int64_t s_stage, int64_t s_mb, cudaStream_t st) {
    const int words = ktab_words(sp->R, sp->pmax, sp->nseg);
    if (sp->used_words + words > sp->region_words) return PP_ERR_SIZE;
    uint32_t *out = sp->region + sp->used_words;
    k_ktab<<<(words + 255) / 256, 256, 0, st>>>(sp->desc, sp->rw, sp->seg, sp->R, sp->P, sp->pmax, sp->nseg,
                                                (int)s_stage, (int)s_mb, out);
    PPS_CUDA_TRY(cudaGetLastError());
    sp->ktab = out;
    sp->ktab_words = words;
    return PP_OK;
}

namespace {
std::mutex g_cache_mu;
std::map<std::tuple<int, int, int, int, int>, pp_plan *> g_cache;
}  // namespace

int cached_plans(const PlanShape *shapes, int n, cudaStream_t stream, pp_plan **out) {
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(g_cache_mu);
    std::vector<PlanShape> need;
    std::map<std::tuple<int, int, int, int, int>, int> queued;
    for (int i = 0; i < n; ++i) {
        const PlanShape &sh = shapes[i];
        const auto key = std::make_tuple(dev, sh.policy, sh.P, sh.M, sh.v);
        const auto it = g_cache.find(key);
        out[i] = it != g_cache.end() ? it->second : nullptr;
        if (!out[i] && queued.emplace(key, (int)need.size()).second) need.push_back(sh);
    }
    if (need.empty()) return PP_OK;
    std::vector<pp_plan *> built(need.size(), nullptr);
    const int rc = build_plans(need.data(), (int)need.size(), stream, built.data());
    if (rc) return rc;
    for (size_t q = 0; q < need.size(); ++q)
        g_cache[std::make_tuple(dev, need[q].policy, need[q].P, need[q].M, need[q].v)] = built[q];
    for (int i = 0; i < n; ++i)
        if (!out[i]) out[i] = built[queued[std::make_tuple(dev, shapes[i].policy, shapes[i].P, shapes[i].M,
                                                           shapes[i].v)]];
    return PP_OK;
}

int cached_plan(int policy, int P, int M, int v, cudaStream_t stream, pp_plan **out) {
    const PlanShape sh{policy, P, M, v};
    return cached_plans(&sh, 1, stream, out);
}

int build_tables(TableReq *reqs, int n, cudaStream_t st) {
    struct Q {
        pp_plan *plan;
        int64_t s_stage, s_mb;
        int lane, nblocks;
        int64_t off, words;
    };
    std::vector<Q> q;
    std::vector<int> which(n, -1);
    std::map<std::tuple<pp_plan *, int64_t, int64_t, int>, int> seen;
    int64_t total = 0, max_reg = 0, max_lane = 0;
    for (int i = 0; i < n; ++i) {
        TableReq &r = reqs[i];
        r.out = nullptr;
        {
            std::lock_guard<std::mutex> lk(r.plan->ktab_mu);
            for (const pp_ktab &t : r.lane ? r.plan->ltabs : r.plan->ktabs)
                if (t.s_stage == r.s_stage && t.s_mb == r.s_mb && t.variant == r.lane) { r.out = &t; break; }
        }
        if (r.out) continue;
        const auto key = std::make_tuple(r.plan, r.s_stage, r.s_mb, r.lane);
        const auto it = seen.find(key);
        if (it != seen.end()) { which[i] = it->second; continue; }
        Q e{r.plan, r.s_stage, r.s_mb, r.lane, 0, total, 0};
        if (r.lane) {
            e.words = lane_table_words(r.plan->pmax, r.plan->R, lane_word_entries(r.plan->nlslots, r.plan->v, r.s_mb, 1),
                                       &e.nblocks);
            if (e.words < 0) return PP_ERR_INTERNAL;
            max_lane = std::max(max_lane, e.words);
        } else {
            e.words = ktab_words(r.plan->R, r.plan->pmax, r.plan->nseg);
            max_reg = std::max(max_reg, e.words);
        }
        total += pad4(e.words);
        which[i] = (int)q.size();
        seen.emplace(key, (int)q.size());
        q.push_back(e);
    }
    if (q.empty()) return PP_OK;
    // the job records go after the tables, in the same allocation
    const int64_t jobs_at = total;
    Arena A;
    int rc = A.alloc(jobs_at + pad4((int64_t)q.size() * (int64_t)sizeof(TableJob) / 4 + 1));
    if (rc) return rc;
    TableJob *d_jobs = reinterpret_cast<TableJob *>(A.w() + jobs_at);
    // every job record, grouped by kind and table width, in one upload
    std::vector<TableJob> jobs;
    std::vector<std::pair<int, int>> groups;  // (kind, pmax) of each run of records
    std::vector<size_t> first;
    for (int kind = 0; kind < 2; ++kind) {
        for (int pmax : {4, 8, 16}) {
            const size_t f0 = jobs.size();
            for (const Q &e : q) {
                if (e.lane != kind || e.plan->pmax != pmax) continue;
                const pp_plan *p = e.plan;
                TableJob j{};
                j.desc = p->d_desc; j.rw = p->d_rw; j.seg = p->d_seg; j.lslot = p->d_lslot;
                j.R = p->R; j.P = p->P; j.v = p->v; j.pmax = p->pmax; j.nseg = p->nseg;
                j.nslots = p->nlslots; j.nblocks = e.nblocks;
                j.s_stage = (int)e.s_stage; j.s_mb = (int)e.s_mb;
                j.word = e.lane && lane_word_entries(p->nlslots, p->v, e.s_mb, 1);
                j.words = e.words; j.out = A.w() + e.off;
                jobs.push_back(j);
            }
            if (jobs.size() > f0) {
                groups.emplace_back(kind, pmax);
                first.push_back(f0);
            }
        }
    }
    first.push_back(jobs.size());
    PPS_CUDA_TRY(cudaMemcpyAsync(d_jobs, jobs.data(), jobs.size() * sizeof(TableJob), cudaMemcpyHostToDevice, st));
    for (size_t gi = 0; gi < groups.size() && !rc; ++gi) {
        const int kind = groups[gi].first, pmax = groups[gi].second;
        for (size_t j0 = first[gi]; j0 < first[gi + 1] && !rc; j0 += 65535) {
            const int c = (int)std::min<size_t>(65535, first[gi + 1] - j0);
            if (kind == 0) kb_ktab<<<dim3(grid_x(max_reg), c), 256, 0, st>>>(d_jobs + j0);
            else rc = launch_ltab_batch(pmax, d_jobs + j0, c, max_lane, st);
        }
    }
    if (!rc) PPS_CUDA_TRY(cudaGetLastError());
    if (rc) return rc;
    std::vector<const pp_ktab *> made(q.size());
    for (size_t x = 0; x < q.size(); ++x) {
        const Q &e = q[x];
        pp_ktab t;
        t.s_stage = e.s_stage;
        t.s_mb = e.s_mb;
        t.d = reinterpret_cast<uint4 *>(A.w() + e.off);
        t.words = (int)e.words;
        t.variant = e.lane;
        t.arena = A.a;
        arena_ref(A.a);
        std::lock_guard<std::mutex> lk(e.plan->ktab_mu);
        std::deque<pp_ktab> &d = e.lane ? e.plan->ltabs : e.plan->ktabs;
        d.push_back(t);
        made[x] = &d.back();
    }
    A.a = nullptr;  // now owned by the tables
    for (int i = 0; i < n; ++i)
        if (!reqs[i].out) reqs[i].out = made[which[i]];
    return PP_OK;
}

}  // namespace pps

extern "C" {

int pp_sched_plan(pp_policy_t policy, int P, int M, int v, pp_plan_t **plan, cudaStream_t stream) {
    if (!plan) return PP_ERR_ARG;
    *plan = nullptr;
    return pps::build_plan((int)policy, P, M, v, stream, plan);
}

int pp_sched_plan_info(const pp_plan_t *p, int32_t *info) {
    if (!p || !info) return PP_ERR_ARG;
    info[0] = p->R; info[1] = p->O; info[2] = p->nslots; info[3] = p->reg_ok;
    info[4] = p->P; info[5] = p->M; info[6] = p->v; info[7] = p->policy;
    return PP_OK;
}

int pp_sched_plan_ops(const pp_plan_t *p, uint32_t *host_ops, int32_t *host_peak, int32_t *host_round) {
    if (!p) return PP_ERR_ARG;
    int cur = 0;
    PPS_CUDA_TRY(cudaGetDevice(&cur));
    if (cur != p->device) PPS_CUDA_TRY(cudaSetDevice(p->device));
    const size_t n = (size_t)p->P * p->O;
    int rc = PP_OK;
    if (host_ops && cudaMemcpy(host_ops, p->d_ops, n * sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        rc = PP_ERR_CUDA;
    if (!rc && host_round && cudaMemcpy(host_round, p->d_round, n * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        rc = PP_ERR_CUDA;
    if (host_peak) for (int k = 0; k < p->P; ++k) host_peak[k] = p->h_peak[k];
    if (cur != p->device) cudaSetDevice(cur);
    if (rc) (void)cudaGetLastError();
    return rc;
}

void pp_sched_plan_destroy(pp_plan_t *p) {
    if (!p) return;
    if (!p->slots_in_arena) {
        if (p->d_desc2) cudaFree(p->d_desc2);
        if (p->d_lslot) cudaFree(p->d_lslot);
    }
    for (pp_ktab &t : p->ktabs) t.arena ? pps::arena_release(t.arena) : (void)cudaFree(t.d);
    for (pp_ktab &t : p->ltabs) t.arena ? pps::arena_release(t.arena) : (void)cudaFree(t.d);
    for (pp_arena *a : p->arena) pps::arena_release(a);
    delete p;
}

void pp_sched_cache_clear(void) {
    std::lock_guard<std::mutex> lk(pps::g_cache_mu);
    for (auto &kv : pps::g_cache) pp_sched_plan_destroy(kv.second);
    pps::g_cache.clear();
}

const char *pp_sched_status_str(int code) {
    switch (code) {
        case PP_OK: return "ok";
        case PP_ERR_ARG: return "invalid argument";
        case PP_ERR_DIVISIBILITY: return "interleaved schedule needs M divisible by P";
        case PP_ERR_SIZE: return "shape beyond the library's limits";
        case PP_ERR_CUDA: return "CUDA runtime error";
        case PP_ERR_DEADLOCK: return "schedule order deadlocks";
        case PP_ERR_INTERNAL: return "internal consistency check failed";
        default: return "unknown status";
    }
}

}  // extern "C"
