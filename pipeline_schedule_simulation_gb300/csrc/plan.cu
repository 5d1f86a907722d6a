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

__global__ void k_order(int policy, int P, int M, int v, uint32_t *ops, int32_t *pos) {
    const int O = 2 * M * v, S = P * v;
    int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)P * O) return;
    int k = (int)(t / O), j = (int)(t % O);
    uint32_t op = op_at(policy, P, M, v, k, j);
    ops[t] = op;
    pos[pos_key(op_kind(op), op_chunk(op) * P + k, op_mb(op), S, M)] = j;
}

// info[0] = rounds, info[1] = 1 on deadlock.  Launched as one warp; P <= 32.
__global__ void k_rounds(const uint32_t *ops, const int32_t *pos, int P, int M, int v,
                         int32_t *round, int32_t *info) {
    __shared__ int pub[32];
    const int O = 2 * M * v, S = P * v;
    const int k = threadIdx.x;
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

__global__ void k_desc(const uint32_t *ops, const int32_t *round, int P, int M, int v, int pmax,
                       uint32_t *desc) {
    const int O = 2 * M * v;
    int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)P * O) return;
    int k = (int)(t / O);
    uint32_t op = ops[t];
    desc[(int64_t)round[t] * pmax + k] =
        desc_pack(op_kind(op) ? kBwd : kFwd, (uint32_t)op_chunk(op), (uint32_t)op_mb(op));
}

// One thread per round: pack the devices' kinds and classify the round.
__global__ void k_rwords(const uint32_t *desc, int R, int P, int pmax, uint64_t *rw) {
    int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= R) return;
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

// One thread: cut the rounds into segments.  info[6] = segment count.
__global__ void k_segments(const uint64_t *rw, int R, uint4 *seg, int32_t *info) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
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

__global__ void k_peak(const uint32_t *ops, int P, int O, int32_t *peak) {
    int k = threadIdx.x;
    if (k >= P) return;
    int held = 0, pk = 0;
    for (int j = 0; j < O; ++j) {
        held += op_kind(ops[k * O + j]) ? -1 : 1;
        pk = max(pk, held);
    }
    peak[k] = pk;
}

// v == 1 only.  info[2] |= 1 if some input is not the latest result of its kind
// on the producing device at the start of the consumer's round.
__global__ void k_latest(const uint32_t *ops, const int32_t *pos, const int32_t *round, int P,
                         int M, int32_t *info) {
    const int O = 2 * M, S = P;
    int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)P * O) return;
    int k = (int)(t / O), j = (int)(t % O);
    uint32_t op = ops[t];
    int kd = op_kind(op), mb = op_mb(op);
    int cdev;
    if (kd == 0 && k < P - 1) cdev = k + 1;
    else if (kd == 1 && k > 0) cdev = k - 1;
    else return;  // no consumer on another device
    int rc = round[cdev * O + pos[pos_key(kd, cdev, mb, S, M)]];
    for (int q = j + 1; q < O; ++q) {
        if (op_kind(ops[k * O + q]) == kd) {
            if (round[k * O + q] < rc) atomicOr(&info[2], 1);
            break;
        }
    }
}

// Greedy value-slot assignment, one thread.  info[3] = slots used, info[4] = 1
// if more than kMaxValueSlots would be needed.
__global__ void k_slots(const uint32_t *desc, int R, int P, int M, int v, int pmax,
                        int32_t *slot_of, uint32_t *desc2, int32_t *info) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
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
// rows than the plan-wide colouring of k_slots.  One warp, lane kc colours
// the inputs of device kc in round order, mapping each in-flight result
// from its plan-wide slot (unique while it is in flight) to a local one, and
// frees a local slot at the end of the round that consumes it.  Writes
// lrd[r][k] (local slot read by op (r,k)) for k = kc, lwr[r][k] (local slot
// op (r,k) writes) for producers whose consumer is kc; 0xFF where none.
// info[7] = local slots used (the maximum over devices), -1 on exhaustion.
__global__ void k_cslots(const uint32_t *desc, const uint32_t *desc2, int R, int P, int pmax, uint8_t *lrd,
                         uint8_t *lwr, int32_t *info) {
    __shared__ uint8_t loc[32][kMaxValueSlots];
    const int kc = threadIdx.x;
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
    if (threadIdx.x == 0) info[7] = any_bad ? -1 : nmax;
}

// Fill the register evaluator's tables for one stride pair: loader table
// entries (element offset of the op's cost row, shifted left by one, bit 0 set
// for a backward op; all ones for an idle slot), then the round words, then
// the segments.
__global__ void k_ktab(const uint32_t *desc, const uint64_t *rw, const uint4 *seg, int R, int P, int pmax,
                       int nseg, int s_stage, int s_mb, uint32_t *out) {
    const int tw = (R * pmax + 3) & ~3;
    const int rw_words = 2 * ((R + 1) & ~1);
    const int total = tw + rw_words + 4 * nseg;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
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
        out[e] = v;
    }
}

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

static int build_plan(int policy, int P, int M, int v, cudaStream_t st, pp_plan **out) {
    int rc = check_shape(policy, P, M, v);
    if (rc) return rc;
    const int S = P * v, O = 2 * M * v, pmax = pmax_for(P);
    const int64_t nops = (int64_t)P * O, npos = 2LL * S * M;
    DevBuf ops, pos, round, info, peak, desc, desc2, rw, seg, lslot;
    PPS_CUDA_TRY(cudaMalloc(&ops.p, nops * sizeof(uint32_t)));
    PPS_CUDA_TRY(cudaMalloc(&pos.p, npos * sizeof(int32_t)));
    PPS_CUDA_TRY(cudaMalloc(&round.p, nops * sizeof(int32_t)));
    PPS_CUDA_TRY(cudaMalloc(&info.p, 8 * sizeof(int32_t)));
    PPS_CUDA_TRY(cudaMalloc(&peak.p, P * sizeof(int32_t)));
    PPS_CUDA_TRY(cudaMemsetAsync(info.p, 0, 8 * sizeof(int32_t), st));
    const int tpb = 256;
    const unsigned nblk = (unsigned)((nops + tpb - 1) / tpb);
    k_order<<<nblk, tpb, 0, st>>>(policy, P, M, v, ops.as<uint32_t>(), pos.as<int32_t>());
    k_rounds<<<1, 32, 0, st>>>(ops.as<uint32_t>(), pos.as<int32_t>(), P, M, v, round.as<int32_t>(),
                               info.as<int32_t>());
    PPS_CUDA_TRY(cudaGetLastError());
    int32_t h_info[8];
    PPS_CUDA_TRY(cudaMemcpyAsync(h_info, info.p, sizeof(h_info), cudaMemcpyDeviceToHost, st));
    PPS_CUDA_TRY(cudaStreamSynchronize(st));
    if (h_info[1]) return PP_ERR_DEADLOCK;
    const int R = h_info[0];
    if (R < 1) return PP_ERR_INTERNAL;
    PPS_CUDA_TRY(cudaMalloc(&desc.p, (int64_t)R * pmax * sizeof(uint32_t)));
    PPS_CUDA_TRY(cudaMemsetAsync(desc.p, 0, (int64_t)R * pmax * sizeof(uint32_t), st));
    k_desc<<<nblk, tpb, 0, st>>>(ops.as<uint32_t>(), round.as<int32_t>(), P, M, v, pmax,
                                 desc.as<uint32_t>());
    k_peak<<<1, 32, 0, st>>>(ops.as<uint32_t>(), P, O, peak.as<int32_t>());
    // one spare word so the table can be copied in 16-byte pieces
    PPS_CUDA_TRY(cudaMalloc(&rw.p, (int64_t)(R + 1) * sizeof(uint64_t)));
    PPS_CUDA_TRY(cudaMemsetAsync(rw.p, 0, (int64_t)(R + 1) * sizeof(uint64_t), st));
    k_rwords<<<(R + 255) / 256, 256, 0, st>>>(desc.as<uint32_t>(), R, P, pmax, rw.as<uint64_t>());
    PPS_CUDA_TRY(cudaMalloc(&seg.p, (int64_t)R * sizeof(uint4)));
    k_segments<<<1, 32, 0, st>>>(rw.as<uint64_t>(), R, seg.as<uint4>(), info.as<int32_t>());
    int reg_ok = 0;
    if (v == 1) {
        k_latest<<<nblk, tpb, 0, st>>>(ops.as<uint32_t>(), pos.as<int32_t>(), round.as<int32_t>(), P, M,
                                       info.as<int32_t>());
        PPS_CUDA_TRY(cudaGetLastError());
        PPS_CUDA_TRY(cudaMemcpyAsync(h_info, info.p, sizeof(h_info), cudaMemcpyDeviceToHost, st));
        PPS_CUDA_TRY(cudaStreamSynchronize(st));
        reg_ok = h_info[2] == 0;
    }
    int nslots = 0, nlslots = 0;
    if (!reg_ok) {
        rc = build_slots(desc.as<uint32_t>(), R, P, M, v, pmax, st, reinterpret_cast<uint32_t **>(&desc2.p),
                         reinterpret_cast<uint8_t **>(&lslot.p), &nslots, &nlslots);
        if (rc) return rc;
    }
    pp_plan *p = new pp_plan();
    p->policy = policy; p->P = P; p->M = M; p->v = v; p->S = S; p->O = O;
    p->R = R; p->pmax = pmax; p->nslots = nslots; p->nlslots = nlslots; p->reg_ok = reg_ok;
    PPS_CUDA_TRY(cudaGetDevice(&p->device));
    if (cudaMemcpyAsync(p->h_peak, peak.p, P * sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        delete p;
        return cuda_status(cudaErrorUnknown);
    }
    p->d_ops = ops.as<uint32_t>(); ops.p = nullptr;
    p->d_round = round.as<int32_t>(); round.p = nullptr;
    p->d_desc = desc.as<uint32_t>(); desc.p = nullptr;
    p->d_desc2 = desc2.as<uint32_t>(); desc2.p = nullptr;
    p->d_lslot = lslot.as<uint8_t>(); lslot.p = nullptr;
    p->d_rw = rw.as<uint64_t>(); rw.p = nullptr;
    p->d_seg = seg.as<uint4>(); seg.p = nullptr;
    p->nseg = h_info[6];
    p->d_peak = peak.as<int32_t>(); peak.p = nullptr;
    *out = p;
    return PP_OK;
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

int cached_plan(int policy, int P, int M, int v, cudaStream_t stream, pp_plan **out) {
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    auto key = std::make_tuple(dev, policy, P, M, v);
    std::lock_guard<std::mutex> lk(g_cache_mu);
    auto it = g_cache.find(key);
    if (it != g_cache.end()) { *out = it->second; return PP_OK; }
    pp_plan *p = nullptr;
    int rc = build_plan(policy, P, M, v, stream, &p);
    if (rc) return rc;
    g_cache[key] = p;
    *out = p;
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
    cudaFree(p->d_ops);
    cudaFree(p->d_round);
    cudaFree(p->d_desc);
    if (p->d_desc2) cudaFree(p->d_desc2);
    if (p->d_lslot) cudaFree(p->d_lslot);
    cudaFree(p->d_rw);
    cudaFree(p->d_seg);
    for (pp_ktab &t : p->ktabs) cudaFree(t.d);
    for (pp_ktab &t : p->ltabs) cudaFree(t.d);
    cudaFree(p->d_peak);
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
