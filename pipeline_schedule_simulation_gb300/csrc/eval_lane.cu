// eval_lane.cu -- the lane-per-device evaluator (interleaved 1F1B).
//
// Interleaved 1F1B ("2. 1F1B" §6.1; "Pipeline scheduling" (M040) §06: device
// k holds the virtual stages k, k+P, ...) can keep several results of one
// kind in flight between two devices, so an op finds its input through the
// plan's value slots rather than a fixed register.  Its cost tables are small
// (a few MB), so the evaluation is bound by instruction issue and latency,
// not by HBM.  This kernel therefore gives every (instance, device) pair its
// own lane: a warp holds 32/PMAX instances, lane = device * (32/PMAX) +
// instance, and in each wavefront round every lane runs at most one op.
// Ops of one round are independent, so all lanes of a round run in parallel
// and one __syncwarp per round publishes the round's results.
//
// Per warp, in shared memory, every row is 32 words per instance set (see
// k_eval_lane) with column = lane:
//   ring   kSlices rows  cost of this lane's op, filled kAhead rounds ahead
//   val    nslots rows + a zero row + a scratch row: an op's end tick is
//          written into its consumer device's column of its value slot;
//          slots are coloured per consumer device (k_cslots), so nslots is
//          the most inputs one device has in flight, not the plan's total
//   ctab   2v rows + a zero row: the comm latency on the input edge of this
//          lane's ops, row 2c for a forward of chunk c (boundary s-1|s) and
//          row 2c+1 for a backward (boundary s|s+1; the backward latency when
//          it is given separately)
// An op without an input reads the zero rows, an op without a consumer
// writes the scratch row, and an idle slot runs as a zero-cost op, so the
// round body has no branch.
//
// The per-(round, device) table (built once per plan and stride pair by
// k_ltab) is streamed through the CTA in blocks of kBR rounds, double
// buffered with cp.async and published with one __syncthreads per block.
// Entry (round r, device k), one uint4 read by the device's lanes at once:
//   x  byte offset of the input slot cell (row * row bytes + column)
//   y  byte offset of the comm cell
//   z  byte offset of the output slot cell; bit 31 set when the op is not idle
//   w  loader entry of round r + kAhead: byte offset of the op's cost row
//      | 1 for a backward op, or kLtIdle; shifted by kAhead rounds so the
//      loader never needs the next block
// With costs shared by all microbatches (stride_mb == 0) there is no loader,
// and the entry is one word, so a block holds four times the rounds and a
// round reads a quarter of the bytes:
//   bits 0..14   byte offset of the output slot cell (as z, without bit 31)
//   bit 15       the op is not idle
//   bits 16..22  the op's {cost, comm} row (2 * chunk + kind; 2v: the zero row)
//   bits 23..31  the input slot row's byte offset / 128 (the lane's own
//                column is added by the lane)
// which holds while (nslots + 2) * row bytes <= 2^15 and 2v + 1 <= 127
// (lane_word_entries); past that, such costs run through the cost ring.
#include <algorithm>
#include <climits>

#include <atomic>

#include "eval_common.cuh"

namespace pps {

template <int PMAX>
struct LaneGeom {
    static constexpr int kIPW = 32 / PMAX;              // instances per warp
    static constexpr int kSlices = 8;                   // cost ring rows
    static constexpr int kAhead = kSlices - 2;          // rounds loaded ahead
    static constexpr int kBR = 512 / PMAX;              // rounds per table block
    static constexpr int kBlockWords = 4 * kBR * PMAX;  // one uint4 per entry
    static constexpr int kBRw = 4 * kBR;                // rounds per block of one-word entries
    static constexpr int kHeadWords = (kAhead * PMAX + 3) & ~3;
    static constexpr int kCopy = kIPW < 4 ? kIPW : 4;   // instances per loader copy (vector path)
    static_assert(kBR > kAhead, "a table block must outlast the loader's lead");
    static_assert(kSlices == 8 && kBR % kSlices == 0, "the round loop is unrolled by the ring size");
};

constexpr uint32_t kLaneActive = 0x80000000u;

// Loader entry of (round r, device k): the byte offset of the op's cost row
// (element offsets stay below 2^30, checked on the host), bit 0 set for a
// backward op; kLtIdle for an idle slot or a round past the end.
__device__ __forceinline__ uint32_t lane_lt(const uint32_t *desc, int R, int P, int pmax, int r, int k,
                                            int s_stage, int s_mb) {
    if (r >= R) return kLtIdle;
    const uint32_t d = desc[(int64_t)r * pmax + k];
    const uint32_t kind = desc_kind(d);
    if (kind == kIdle) return kLtIdle;
    const int s = (int)desc_chunk(d) * P + k;
    const uint32_t off = (uint32_t)(s * s_stage + (int)desc_mb(d) * s_mb);
    return (off << 2) | (kind == kBwd ? 1u : 0u);
}

// Table of the lane evaluator for one stride pair: head (loader entries of
// rounds 0 .. kAhead-1), then ceil(R / kBR) blocks laid out as described at
// the top of the file (`word`: one-word entries, ceil(R / kBRw) blocks, the
// head unused).  Word e of that table:
template <int PMAX>
__device__ uint32_t ltab_word(const uint32_t *desc, const uint8_t *lrd, const uint8_t *lwr, int R, int P, int v,
                              int nslots, int s_stage, int s_mb, uint32_t row_bytes, bool word, int64_t e) {
    using G = LaneGeom<PMAX>;
    uint32_t w = kLtIdle;
    if (word) {
        // one word per entry; the head (loader entries) is not read
        if (e < G::kHeadWords) return kLtIdle;
        const int64_t e2 = e - G::kHeadWords;
        const int b = (int)(e2 / G::kBlockWords);
        const int o = (int)(e2 % G::kBlockWords);
        const int q = o / PMAX, k = o % PMAX, r = b * G::kBRw + q;
        const uint32_t col = (uint32_t)(k * G::kIPW * 4);
        uint32_t rd = (uint32_t)nslots * row_bytes;              // zero row
        uint32_t wr = (uint32_t)(nslots + 1) * row_bytes + col;  // scratch row
        uint32_t cmr = (uint32_t)(2 * v), act = 0;               // zero comm row
        if (r < R) {
            const uint32_t d = desc[(int64_t)r * PMAX + k];
            const uint32_t kind = desc_kind(d);
            if (kind != kIdle) {
                act = 1u << 15;
                const uint32_t rs = lrd[(int64_t)r * PMAX + k], ws = lwr[(int64_t)r * PMAX + k];
                cmr = 2u * desc_chunk(d) + (kind == kBwd ? 1u : 0u);
                if (rs != kNoSlot) rd = rs * row_bytes;
                if (ws != kNoSlot) {
                    const int kc = kind == kFwd ? (k + 1) % P : (k + P - 1) % P;
                    wr = ws * row_bytes + (uint32_t)(kc * G::kIPW * 4);
                }
            }
        }
        return wr | act | ((rd | cmr) << 16);
    }
    if (e < G::kHeadWords) {
        const int q = (int)e;
        if (q < G::kAhead * PMAX) w = lane_lt(desc, R, P, PMAX, q / PMAX, q % PMAX, s_stage, s_mb);
    } else {
        const int64_t e2 = e - G::kHeadWords;
        const int b = (int)(e2 / G::kBlockWords);
        const int o = (int)(e2 % G::kBlockWords);
        const int idx = o >> 2, q = idx / PMAX, k = idx % PMAX, r = b * G::kBR + q;
        if ((o & 3) == 3) {
            w = lane_lt(desc, R, P, PMAX, r + G::kAhead, k, s_stage, s_mb);
        } else {
            const uint32_t col = (uint32_t)(k * G::kIPW * 4);
            uint32_t rd = (uint32_t)nslots * row_bytes + col;           // zero row
            uint32_t wr = (uint32_t)(nslots + 1) * row_bytes + col;     // scratch row
            uint32_t cm = (uint32_t)(2 * v) * row_bytes + col, act = 0;  // zero comm row
            if (r < R) {
                const uint32_t d = desc[(int64_t)r * PMAX + k];
                const uint32_t kind = desc_kind(d);
                if (kind != kIdle) {
                    act = kLaneActive;
                    const uint32_t rs = lrd[(int64_t)r * PMAX + k], ws = lwr[(int64_t)r * PMAX + k];
                    // the op's (chunk, kind) row: its input edge's comm (0 where
                    // there is no edge) and, with costs shared by all
                    // microbatches, its cost
                    cm = (2u * desc_chunk(d) + (kind == kBwd ? 1u : 0u)) * row_bytes + col;
                    if (rs != kNoSlot) rd = rs * row_bytes + col;
                    if (ws != kNoSlot) {
                        const int kc = kind == kFwd ? (k + 1) % P : (k + P - 1) % P;
                        wr = ws * row_bytes + (uint32_t)(kc * G::kIPW * 4);
                    }
                }
            }
            w = (o & 3) == 0 ? rd : ((o & 3) == 1 ? cm : (wr | act));
        }
    }
    return w;
}

template <int PMAX>
__global__ void k_ltab(const uint32_t *desc, const uint8_t *lrd, const uint8_t *lwr, int R, int P, int v, int nslots,
                       int s_stage, int s_mb, int nblocks, uint32_t row_bytes, bool word, uint32_t *out) {
    using G = LaneGeom<PMAX>;
    const int64_t total = G::kHeadWords + (int64_t)nblocks * G::kBlockWords;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x)
        out[e] = ltab_word<PMAX>(desc, lrd, lwr, R, P, v, nslots, s_stage, s_mb, row_bytes, word, e);
}

// Many tables with one instance set per lane, one TableJob per table (blockIdx.y).
template <int PMAX>
__global__ void kb_ltab(const TableJob *jobs) {
    const TableJob &b = jobs[blockIdx.y];
    const int64_t cells = (int64_t)b.R * PMAX;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < b.words;
         e += (int64_t)gridDim.x * blockDim.x)
        b.out[e] = ltab_word<PMAX>(b.desc, b.lslot, b.lslot + cells, b.R, b.P, b.v, b.nslots, b.s_stage, b.s_mb,
                                   128u, b.word != 0, e);
}

// This lane's share of a round's cost copies.  Vector path: a device row of
// the warp holds NI * 32/PMAX consecutive instances per set, copied in
// pieces of kCopy instances (16 or 8 bytes) by the device's first lanes, one
// piece each.  Scalar path: every lane copies its own word of each set.  Set
// i lands in the ring row at column 32*i + lane (layout [device][instance]).
// Everything but the row offset is fixed per lane, so a round costs a select,
// an add and one predicated cp.async per copy.
template <int PMAX, int NI, bool VEC>
struct LaneLoader {
    static constexpr int kN = VEC ? 1 : NI;  // copies per lane and round
    const char *fb, *bb;   // this lane's first source element in cost_f / cost_b
    int64_t step[kN];      // byte distance from copy 0's source to copy i's (0 if it copies nothing)
    uint32_t bytes[kN];    // bytes of a non-idle op's copy (0 past the last instance)
    uint32_t doff[kN];     // byte offset of the copy in the ring row
    uint32_t on;           // this lane issues copies
    int64_t e0, reach;     // element offset of fb / bb and the elements the strides reach (checked build)

    __device__ __forceinline__ LaneLoader(const EvalArgs &a, int lane, int j, int k, int64_t inst0) {
        using G = LaneGeom<PMAX>;
        reach = cost_reach(a.n, a.S, a.M, a.s_inst, a.s_stage, a.s_mb);
        if constexpr (VEC) {
            constexpr int kPerSet = G::kIPW / G::kCopy;
            const int set = j / kPerSet, piece = j % kPerSet;
            on = j < NI * kPerSet;
            const int64_t xi = inst0 + set * G::kIPW + piece * G::kCopy;
            const int64_t left = a.n - xi;
            e0 = on && left > 0 ? xi : 0;
            fb = reinterpret_cast<const char *>(a.cost_f + e0);
            bb = reinterpret_cast<const char *>(a.cost_b + e0);
            bytes[0] = !on || left <= 0 ? 0u : (uint32_t)(left < G::kCopy ? left : G::kCopy) * 4u;
            step[0] = 0;
            doff[0] = (uint32_t)(set * 32 + k * G::kIPW + piece * G::kCopy) * 4u;
        } else {
            const int64_t x0 = inst0 + j;
            e0 = x0 < a.n ? x0 * a.s_inst : 0;
            fb = reinterpret_cast<const char *>(a.cost_f + e0);
            bb = reinterpret_cast<const char *>(a.cost_b + e0);
            on = 1;
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const bool in = x0 + i * G::kIPW < a.n;
                bytes[i] = in ? 4u : 0u;
                step[i] = in ? (int64_t)i * G::kIPW * a.s_inst * 4 : 0;
                doff[i] = (uint32_t)(32 * i + lane) * 4u;
            }
        }
    }

    // lt: the loader entry of the round; row: shared address of the ring row
    __device__ __forceinline__ void issue(uint32_t lt, uint32_t row) const {
        using G = LaneGeom<PMAX>;
        const bool idle = lt == kLtIdle;
        const char *src = ((lt & 1u) ? bb : fb) + (idle ? 0u : (lt & ~3u));
#pragma unroll
        for (int i = 0; i < kN; ++i) {
            const char *s = src + step[i];
            uint32_t nb = idle ? 0u : bytes[i];
            if (nb && !PPS_CHECK(e0 + (int64_t)((lt & ~3u) + step[i] + nb) / 4 <= reach, kChkCostRead,
                                 e0 + (int64_t)((lt & ~3u) + step[i]) / 4))
                nb = 0;
            const uint32_t d = row + doff[i];
            if constexpr (VEC && G::kCopy == 4)
                asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %3, 0;\n"
                             " @p cp.async.cg.shared.global [%0], [%1], 16, %2;\n}\n" ::"r"(d), "l"(s), "r"(nb),
                             "r"(on) : "memory");
            else if constexpr (VEC)
                asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %3, 0;\n"
                             " @p cp.async.ca.shared.global [%0], [%1], 8, %2;\n}\n" ::"r"(d), "l"(s), "r"(nb),
                             "r"(on) : "memory");
            else
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(d), "l"(s), "r"(nb) : "memory");
        }
    }
};

// Shared-memory accesses by 32-bit shared-window address.
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;\n" ::"r"(addr), "r"(v) : "memory");
}

// Copy table block `b` into `dst` (all threads of the CTA; joins the caller's
// next commit group).
template <int PMAX>
__device__ __forceinline__ void lane_copy_block(const uint4 *blocks, int b, uint32_t *dst) {
    using G = LaneGeom<PMAX>;
    const uint4 *src = blocks + (int64_t)b * (G::kBlockWords / 4);
    for (int i = threadIdx.x; i < G::kBlockWords / 4; i += blockDim.x) cp_async16(smem_addr(dst + 4 * i), src + i, 16);
}

// NI instance sets per lane: a warp holds NI * 32/PMAX instances; every row
// of the warp's shared memory is 32*NI words, set i in words 32i .. 32i+31,
// so the second set of a row sits at a fixed +128 bytes.
// MBZ: the costs are the same for every microbatch (stride_mb == 0), so each
// lane keeps its (chunk, kind) costs next to the comm in shared memory -- the
// ctab rows hold {cost, comm} pairs -- and the cost ring and its loader go.
// The body takes the CTA's index within its problem (`bid`), so the fused
// kernel over many problems runs it too.
template <int PMAX, int NI, bool VEC, bool OPS, bool MBZ>
__device__ __forceinline__ void lane_body(const EvalArgs &a, const uint4 *tab, int nblocks, int64_t bid) {
    // Programmatic dependent launch (the one-CTA-per-SM launch): the next
    // grid may place its CTAs as this one's retire; a CTA copies its first
    // table block (the plan's, complete before the launch) and waits for the
    // previous grid before it reads an input or writes an output.  Without
    // the launch attribute both instructions do nothing.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    using G = LaneGeom<PMAX>;
    constexpr int kRow = 32 * NI;  // words per row
    constexpr int kRingRows = MBZ ? 0 : G::kSlices;
    constexpr int kCw = MBZ ? 2 : 1;  // words per ctab cell
    extern __shared__ __align__(16) uint32_t lsm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int j = lane % G::kIPW, k = lane / G::kIPW;
    const int rows = kRingRows + a.nslots + 2 + (2 * a.v + 1) * kCw;
    uint32_t *ring = lsm + 2 * G::kBlockWords + warp * rows * kRow;
    uint32_t *val = ring + kRingRows * kRow;
    uint32_t *ctab = val + (a.nslots + 2) * kRow;
    // a.tasks > 0 (one CTA per SM): CTA b takes warp tasks [b*T/G, (b+1)*T/G),
    // so SMs differ by one warp at most; a CTA's spare warp runs on
    // instances past the batch (it still takes part in the CTA's barriers)
    int64_t wtask = bid * nwarps + warp;
    bool has_task = true;
    if (a.tasks > 0) {
        const int64_t t0 = bid * a.tasks / gridDim.x, t1 = (bid + 1) * a.tasks / gridDim.x;
        wtask = t0 + warp;
        has_task = wtask < t1;
    }
    const int64_t inst0 = has_task ? wtask * (G::kIPW * NI) : a.n;
    const int64_t x0 = inst0 + j;  // set i holds instance x0 + i * kIPW
    const uint4 *blocks = tab + G::kHeadWords / 4;
    const int R = a.R;

    // every warp stays to the end: the table blocks are shared by the CTA
    lane_copy_block<PMAX>(blocks, 0, lsm);
    cp_async_commit();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    copy_peak(a, bid);
    const uint32_t *head = reinterpret_cast<const uint32_t *>(tab);
    const LaneLoader<PMAX, NI, VEC> ld(a, lane, j, k, inst0);
    const uint32_t ring_s = smem_addr(ring);
    if constexpr (!MBZ) {
#pragma unroll 1
        for (int q = 0; q < G::kAhead; ++q) {
            ld.issue(__ldg(head + q * PMAX + k), ring_s + q * kRow * 4);
            cp_async_commit();
        }
    }
    // The comm rows (and, MBZ, the cost of each row): a lane's rows are read
    // kFill at a time, every load of a group issued before the first store,
    // so the fill waits for about 2v*NI/kFill memory latencies, not 2v*NI.
    constexpr int kFill = 8;
    uint32_t ncomm[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int64_t x = x0 + i * G::kIPW;
        const bool xin = x < a.n && k < a.P;
        ncomm[i] = 0;
#pragma unroll 1
        for (int cr0 = 0; cr0 < 2 * a.v; cr0 += kFill) {
            int32_t c[kFill], cost[kFill];
#pragma unroll
            for (int u = 0; u < kFill; ++u) {
                const int cr = cr0 + u;
                const int s = (cr >> 1) * a.P + k;
                const int bnd = (cr & 1) ? s : s - 1;
                const int32_t *src = (cr & 1) && a.comm_b ? a.comm_b : a.comm;
                c[u] = src && xin && cr < 2 * a.v && bnd >= 0 && bnd < a.S - 1
                           ? src[x * a.c_inst + (int64_t)bnd * a.c_bnd] : 0;
                if constexpr (MBZ)
                    cost[u] = xin && cr < 2 * a.v
                                  ? ((cr & 1) ? a.cost_b : a.cost_f)[x * a.s_inst + (int64_t)s * a.s_stage] : 0;
            }
#pragma unroll
            for (int u = 0; u < kFill; ++u) {
                const int cr = cr0 + u;
                if (cr >= 2 * a.v) break;
                ncomm[i] |= (uint32_t)c[u];
                if constexpr (MBZ) {
                    ctab[(cr * kRow + 32 * i + lane) * 2] = (uint32_t)cost[u];
                    ctab[(cr * kRow + 32 * i + lane) * 2 + 1] = (uint32_t)c[u];
                } else {
                    ctab[cr * kRow + 32 * i + lane] = (uint32_t)c[u];
                }
            }
        }
        if constexpr (MBZ) {
            ctab[(2 * a.v * kRow + 32 * i + lane) * 2] = 0;
            ctab[(2 * a.v * kRow + 32 * i + lane) * 2 + 1] = 0;
        } else {
            ctab[2 * a.v * kRow + 32 * i + lane] = 0;
        }
        val[a.nslots * kRow + 32 * i + lane] = 0;
    }
    // the first table block (with MBZ nothing else is in flight)
    if constexpr (MBZ) cp_async_wait<0>();
    else cp_async_wait<G::kAhead>();
    __syncthreads();

    const uint32_t val_s = smem_addr(val + j), cost_s = smem_addr(ring + lane);
    // ctab cell of this lane's instance j: word offsets in the table entries
    // count 4 bytes per cell, MBZ cells are 8 bytes
    const uint32_t ctab_s = smem_addr(ctab + j * kCw);
    // one-word entries (MBZ) leave out the lane's own column of the input
    // slot and comm rows
    const uint32_t colk = (uint32_t)(k * G::kIPW * 4);
    const uint32_t valk_s = val_s + colk, ctabk_s = ctab_s + colk * kCw;
    uint32_t fr[NI], busy[NI], flag[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) { fr[i] = 0; busy[i] = 0; flag[i] = 0; }
    int cnt = 0;
#pragma unroll 1
    for (int b = 0; b < nblocks; ++b) {
        if (b + 1 < nblocks) lane_copy_block<PMAX>(blocks, b + 1, lsm + ((b + 1) & 1) * G::kBlockWords);
        if constexpr (MBZ) cp_async_commit();  // otherwise the copy joins the next round's group
        constexpr int kEb = MBZ ? 4 : 16;  // bytes per entry
        constexpr int kBr = MBZ ? G::kBRw : G::kBR;
        const uint32_t ent_s = smem_addr(lsm + (b & 1) * G::kBlockWords) + k * kEb;
        const int n_r = min(R - b * kBr, kBr);
        // One round: the loader runs kAhead rounds ahead into ring row nxt,
        // the op reads its cost from row cur (rows are round mod kSlices; a
        // block starts at a multiple of kSlices).  The next round's entry is
        // read one round early; past the block's last round that read lands
        // in the other table buffer or the first warp's ring (still inside
        // the CTA's shared memory) and is discarded.
        uint4 nx = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (MBZ) nx.x = lds32(ent_s);
        else nx = lds128(ent_s);
        auto round = [&](int q, int cur, int nxt) {
            const uint4 e = nx;
            if constexpr (MBZ) nx.x = lds32(ent_s + (q + 1) * PMAX * kEb);
            else nx = lds128(ent_s + (q + 1) * PMAX * kEb);
            if constexpr (!MBZ) {
                ld.issue(e.w, ring_s + nxt * kRow * 4);
                cp_async_commit();
                cp_async_wait<G::kAhead>();
            }
            __syncwarp();
            // shared addresses of the input slot cell, the {cost, comm} or
            // comm cell and the output slot cell; whether the op is not idle
            // (checked build: the entry's offsets inside the warp's value
            // rows and comm rows; row bytes = 128*NI)
            uint32_t vr, cr, vw, act;
            bool okr, okw, okc;
            if constexpr (MBZ) {
                const uint32_t hi = e.x >> 16, xo = hi & 0xFF80u, co = hi & 0x7Fu, wo = e.x & 0x7FFFu;
                vr = valk_s + xo;
                cr = ctabk_s + co * (256u * NI);
                vw = val_s + wo;
                act = e.x & 0x8000u;
                okr = PPS_CHECK(xo + colk < (uint32_t)(a.nslots + 2) * 128u * NI, kChkLaneSlotRead, xo);
                okw = PPS_CHECK(wo < (uint32_t)(a.nslots + 2) * 128u * NI, kChkLaneSlotWrite, wo);
                okc = PPS_CHECK(co < (uint32_t)(2 * a.v + 1), kChkLaneComm, co);
            } else {
                vr = val_s + e.x;
                cr = ctab_s + e.y * kCw;
                vw = val_s + (e.z & ~kLaneActive);
                act = e.z & kLaneActive;
                okr = PPS_CHECK(e.x < (uint32_t)(a.nslots + 2) * 128u * NI, kChkLaneSlotRead, e.x);
                okw = PPS_CHECK((e.z & ~kLaneActive) < (uint32_t)(a.nslots + 2) * 128u * NI, kChkLaneSlotWrite,
                                e.z & ~kLaneActive);
                okc = PPS_CHECK(e.y < (uint32_t)(2 * a.v + 1) * 128u * NI, kChkLaneComm, e.y);
            }
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                uint32_t c = 0, cm = 0;
                if constexpr (MBZ) {
                    if (okc) {
                        const uint2 cc = lds64(cr + 256 * i);
                        c = cc.x;
                        cm = cc.y;
                    }
                } else {
                    c = lds32(cost_s + (cur * kRow + 32 * i) * 4);
                    if (okc) cm = lds32(cr + 128 * i);
                }
                const uint32_t arr = (okr ? lds32(vr + 128 * i) : 0u) + cm;
                const uint32_t st = max(fr[i], arr);
                const uint32_t en = st + c;
                flag[i] |= st | c;
                busy[i] += c;
                fr[i] = en;
                if (okw) sts32(vw + 128 * i, en);
                if constexpr (OPS) {
                    const int64_t x = x0 + i * G::kIPW;
                    if (act && x < a.n) {
                        const int64_t off = x * a.o_inst + ((int64_t)k * a.O + cnt) * a.o_op;
                        if (a.op_start) a.op_start[off] = (int32_t)st;
                        if (a.op_end) a.op_end[off] = (int32_t)en;
                    }
                }
            }
            if constexpr (OPS) cnt += act ? 1 : 0;
        };
        int q = 0;
#pragma unroll 1
        for (; q + G::kSlices <= n_r; q += G::kSlices) {
#pragma unroll
            for (int i = 0; i < G::kSlices; ++i) round(q + i, i, (i + G::kAhead) % G::kSlices);
        }
#pragma unroll 1
        for (; q < n_r; ++q) round(q, q % G::kSlices, (q + G::kAhead) % G::kSlices);
        if constexpr (MBZ) cp_async_wait<0>();  // the next block's table
        __syncthreads();
    }
    cp_async_wait<0>();

    // Per-instance reductions over the instance's PMAX lanes ("2. 1F1B" §4.3
    // and M040 §04: the window is the last end tick, a stage's idle time is
    // the window minus its busy time, the bubble is total idle over P
    // windows).  `flag` holds the sign bits of every start tick and cost: it
    // is clear exactly when no cost is negative and every tick fits in int32.
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int64_t x = x0 + i * G::kIPW;
        uint32_t mk = fr[i], fl = flag[i], nc = ncomm[i];
#pragma unroll
        for (int m = G::kIPW; m < 32; m <<= 1) {
            mk = max(mk, __shfl_xor_sync(0xFFFFFFFFu, mk, m));
            fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, m);
            nc |= __shfl_xor_sync(0xFFFFFFFFu, nc, m);
        }
        fl |= mk;
        const int idle = k < a.P ? (int)(mk - busy[i]) : 0;
        int64_t num = idle;
#pragma unroll
        for (int m = G::kIPW; m < 32; m <<= 1) num += __shfl_xor_sync(0xFFFFFFFFu, num, m);
        if (x >= a.n) continue;
        if (a.idle && k < a.P) a.idle[x * a.P + k] = idle;
        if (k == 0) {
            if (a.makespan) a.makespan[x] = (int)mk;
            if (a.bub_num) a.bub_num[x] = num;
            if (a.bub_den) a.bub_den[x] = (int64_t)a.P * (int)mk;
            if (a.status) {
                int8_t st = PP_ST_OK;
                if (nc >> 31) st = PP_ST_NEG_COST;
                else if (fl >> 31) st = any_negative_cost(a, x) ? PP_ST_NEG_COST : PP_ST_OVERFLOW;
                a.status[x] = st;
            }
        }
    }
}

template <int PMAX, int NI, bool VEC, bool OPS, bool MBZ>
__global__ void __launch_bounds__(512) k_eval_lane(const EvalArgs a, const uint4 *tab, int nblocks) {
    lane_body<PMAX, NI, VEC, OPS, MBZ>(a, tab, nblocks, blockIdx.x);
}

// Many interleaved problems with microbatch-shared costs in one launch (one
// instance set per lane): CTA c runs CTA c - block_begin of its problem.
template <int PMAX>
__global__ void __launch_bounds__(256) k_eval_lane_mbz_many(const ManyJob *jobs, int njobs) {
    const int j = many_job_of(jobs, njobs, blockIdx.x);
    const EvalArgs &a = jobs[j].a;  // read in place: uniform per CTA, cached
    lane_body<PMAX, 1, false, false, true>(a, jobs[j].tab, jobs[j].nblocks, (int64_t)blockIdx.x - jobs[j].block_begin);
}

namespace {

template <int PMAX, int NI>
int lane_tables_t(pp_plan *plan, int64_t s_stage, int64_t s_mb, cudaStream_t stream, const pp_ktab **out) {
    using G = LaneGeom<PMAX>;
    std::lock_guard<std::mutex> lk(plan->ktab_mu);
    for (const pp_ktab &t : plan->ltabs)
        if (t.s_stage == s_stage && t.s_mb == s_mb && t.variant == NI) { *out = &t; return PP_OK; }
    const bool word = lane_word_entries(plan->nlslots, plan->v, s_mb, NI);
    const int br = word ? G::kBRw : G::kBR;
    const int nblocks = (plan->R + br - 1) / br;
    pp_ktab t;
    t.s_stage = s_stage;
    t.s_mb = s_mb;
    t.variant = NI;
    t.words = G::kHeadWords + nblocks * G::kBlockWords;
    PPS_CUDA_TRY(cudaMalloc(&t.d, (size_t)t.words * sizeof(uint32_t)));
    const int blocks = (t.words + 255) / 256;
    const int64_t cells = (int64_t)plan->R * PMAX;
    k_ltab<PMAX><<<blocks, 256, 0, stream>>>(plan->d_desc, plan->d_lslot, plan->d_lslot + cells, plan->R, plan->P,
                                             plan->v, plan->nlslots, (int)s_stage, (int)s_mb, nblocks, 128 * NI,
                                             word, reinterpret_cast<uint32_t *>(t.d));
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        cudaFree(t.d);
        return cuda_status(e);
    }
    plan->ltabs.push_back(t);
    *out = &plan->ltabs.back();
    return PP_OK;
}

constexpr size_t kLaneSmemLimit = 227 * 1024;

template <int PMAX>
size_t lane_smem(const EvalArgs &a, int warps, int ni, bool mbz = false) {
    using G = LaneGeom<PMAX>;
    const size_t rows = (size_t)(mbz ? 0 : G::kSlices) + a.nslots + 2 + (size_t)(2 * a.v + 1) * (mbz ? 2 : 1);
    return 2 * (size_t)G::kBlockWords * 4 + (size_t)warps * rows * 32 * ni * 4;
}

// Two instance sets per lane halve the per-op share of the table reads, the
// loop and the warp barrier; they are used once the batch still gives the
// GPU about eight such warps per SM.
constexpr int64_t kLaneWarpsForTwoSets = 152 * 8;

// Warps per CTA: every CTA copies the whole table, so larger CTAs are
// cheaper, but a batch of a few thousand warps is one wave of CTAs and the
// busiest SM sets the time.  Take the size (8, 4 or 2 warps) whose busiest
// SM holds the fewest warps with every CTA resident at once, the larger size
// on a tie; with more than one wave, the largest size that fits.
template <int PMAX, int NI, bool VEC, bool OPS, bool MBZ>
int lane_warps(const EvalArgs &a, int64_t warps_total, int sms) {
    int best = 0;
    int64_t best_load = 0;
    for (int w = 8; w >= 2; w >>= 1) {
        const size_t smem = lane_smem<PMAX>(a, w, NI, MBZ);
        if (smem > kLaneSmemLimit) continue;
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_eval_lane<PMAX, NI, VEC, OPS, MBZ>, w * 32, smem) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            continue;
        }
        if (per_sm < 1) continue;
        const int64_t ctas = (warps_total + w - 1) / w;
        const int64_t need = (ctas + sms - 1) / sms;  // CTAs on the busiest SM
        const int64_t load = need > per_sm ? INT64_MAX : need * w;
        if (!best || load < best_load) { best = w; best_load = load; }
    }
    return best;
}

template <int PMAX, int NI, bool VEC, bool OPS, bool MBZ>
int launch_lane_t(const EvalArgs &a, const pp_ktab *t, cudaStream_t st) {
    using G = LaneGeom<PMAX>;
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    static std::atomic<bool> attr_set[64];  // per device, set once (idempotent)
    if (dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
        PPS_CUDA_TRY(cudaFuncSetAttribute(k_eval_lane<PMAX, NI, VEC, OPS, MBZ>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLaneSmemLimit));
        attr_set[dev].store(true, std::memory_order_release);
    }
    const int64_t nw = (a.n + G::kIPW * NI - 1) / (G::kIPW * NI);
    constexpr int kBr = MBZ ? G::kBRw : G::kBR;
    const int nblocks = (a.R + kBr - 1) / kBr;
    // A batch whose warps all fit on the GPU at once: one CTA per SM taking
    // warp tasks by range (SMs differ by one warp), launched as a
    // programmatic dependent launch.  Asking for at least half an SM's shared
    // memory keeps a second CTA -- of this grid or the next -- off the SM, so
    // the next grid's CTAs land one per SM as this grid's retire.
    {
        const int nsm = sm_count(dev);
        const int64_t grid = nw < nsm ? nw : nsm;
        const int64_t wpb = grid > 0 ? (nw + grid - 1) / grid : 0;
        int per_sm_smem = 0;
        PPS_CUDA_TRY(cudaDeviceGetAttribute(&per_sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev));
        size_t smem = wpb > 0 ? lane_smem<PMAX>(a, (int)wpb, NI, MBZ) : 0;
        if (smem < (size_t)per_sm_smem / 2) smem = (size_t)per_sm_smem / 2;
        int fit = 0;
        if (wpb >= 1 && wpb <= 16 && smem <= kLaneSmemLimit &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, k_eval_lane<PMAX, NI, VEC, OPS, MBZ>, (int)wpb * 32,
                                                          smem) == cudaSuccess &&
            fit >= 1) {
            EvalArgs b = a;
            b.tasks = nw;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)grid);
            cfg.blockDim = dim3((unsigned)wpb * 32);
            cfg.dynamicSmemBytes = smem;
            cfg.stream = st;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            at[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            PPS_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_eval_lane<PMAX, NI, VEC, OPS, MBZ>, b, t->d, nblocks));
            return PP_OK;
        }
        (void)cudaGetLastError();
    }
    const int warps = lane_warps<PMAX, NI, VEC, OPS, MBZ>(a, nw, sm_count(dev));
    if (!warps) return PP_ERR_SIZE;
    const size_t smem = lane_smem<PMAX>(a, warps, NI, MBZ);
    const int64_t grid = (nw + warps - 1) / warps;
    if (grid > 0x7FFFFFFF) return PP_ERR_SIZE;
    k_eval_lane<PMAX, NI, VEC, OPS, MBZ><<<(unsigned)grid, warps * 32, smem, st>>>(a, t->d, nblocks);
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}

template <int PMAX, int NI>
int launch_lane_n(pp_plan *plan, const EvalArgs &a, bool vec, bool ops, cudaStream_t st) {
    const pp_ktab *t = nullptr;
    const int rc = lane_tables_t<PMAX, NI>(plan, a.s_stage, a.s_mb, st, &t);
    if (rc) return rc;
    // costs shared by every microbatch: kept per lane, no cost ring (where
    // the table has one-word entries)
    if (lane_word_entries(a.nslots, a.v, a.s_mb, NI))
        return ops ? launch_lane_t<PMAX, NI, false, true, true>(a, t, st)
                   : launch_lane_t<PMAX, NI, false, false, true>(a, t, st);
    if (vec)
        return ops ? launch_lane_t<PMAX, NI, true, true, false>(a, t, st)
                   : launch_lane_t<PMAX, NI, true, false, false>(a, t, st);
    return ops ? launch_lane_t<PMAX, NI, false, true, false>(a, t, st)
               : launch_lane_t<PMAX, NI, false, false, false>(a, t, st);
}

template <int PMAX>
int launch_lane_p(pp_plan *plan, const EvalArgs &a, bool vec, bool ops, cudaStream_t st) {
    using G = LaneGeom<PMAX>;
    // (not where one set would have one-word entries and two would not)
    const bool two = a.n / (2 * G::kIPW) >= kLaneWarpsForTwoSets && lane_smem<PMAX>(a, 2, 2) <= kLaneSmemLimit &&
                     lane_word_entries(a.nslots, a.v, a.s_mb, 2) == lane_word_entries(a.nslots, a.v, a.s_mb, 1);
    return two ? launch_lane_n<PMAX, 2>(plan, a, vec, ops, st) : launch_lane_n<PMAX, 1>(plan, a, vec, ops, st);
}

}  // namespace

// The lane evaluator applies when the plan has value slots, every cost-row
// offset fits the loader table (below 2^30 elements) and a 2-warp CTA fits in
// shared memory.
bool lane_path(const pp_plan *plan, const EvalArgs &args) {
    if (!plan->d_lslot) return false;
    EvalArgs a = args;
    a.nslots = plan->nlslots;
    if ((int64_t)(a.S - 1) * a.s_stage + (int64_t)(a.M - 1) * a.s_mb >= ((int64_t)1 << 30)) return false;
    switch (plan->pmax) {
        case 4: return lane_smem<4>(a, 2, 1) <= kLaneSmemLimit;
        case 8: return lane_smem<8>(a, 2, 1) <= kLaneSmemLimit;
        case 16: return lane_smem<16>(a, 2, 1) <= kLaneSmemLimit;
        default: return false;
    }
}

int launch_eval_lane(pp_plan *plan, const EvalArgs &args, bool vec, bool ops, cudaStream_t st) {
    EvalArgs a = args;
    a.nslots = plan->nlslots;  // the lane evaluator's rows hold per-consumer slots
    switch (plan->pmax) {
        case 4: return launch_lane_p<4>(plan, a, vec, ops, st);
        case 8: return launch_lane_p<8>(plan, a, vec, ops, st);
        case 16: return launch_lane_p<16>(plan, a, vec, ops, st);
        default: return PP_ERR_INTERNAL;
    }
}

bool lane_word_entries(int nslots, int v, int64_t s_mb, int ni) {
    return s_mb == 0 && (int64_t)(nslots + 2) * 128 * ni <= (1 << 15) && 2 * v + 1 <= 127;
}

template <int PMAX>
static int64_t lane_table_words_t(int R, bool word, int *nblocks) {
    using G = LaneGeom<PMAX>;
    const int br = word ? G::kBRw : G::kBR;
    *nblocks = (R + br - 1) / br;
    return G::kHeadWords + (int64_t)*nblocks * G::kBlockWords;
}

int64_t lane_table_words(int pmax, int R, bool word, int *nblocks) {
    switch (pmax) {
        case 4: return lane_table_words_t<4>(R, word, nblocks);
        case 8: return lane_table_words_t<8>(R, word, nblocks);
        case 16: return lane_table_words_t<16>(R, word, nblocks);
        default: return -1;
    }
}

int launch_ltab_batch(int pmax, const TableJob *d_jobs, int njobs, int64_t max_words, cudaStream_t st) {
    const dim3 grid((unsigned)std::min<int64_t>(1024, std::max<int64_t>(1, (max_words + 255) / 256)),
                    (unsigned)njobs);
    switch (pmax) {
        case 4: kb_ltab<4><<<grid, 256, 0, st>>>(d_jobs); break;
        case 8: kb_ltab<8><<<grid, 256, 0, st>>>(d_jobs); break;
        case 16: kb_ltab<16><<<grid, 256, 0, st>>>(d_jobs); break;
        default: return PP_ERR_INTERNAL;
    }
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}

// The fused lane path over many problems: plans without the register path
// (interleaved) whose costs are the same for every microbatch, without
// per-op output or a separate backward latency.
bool lane_mbz_ok(const pp_plan *plan, EvalArgs &a) {
    if (plan->reg_ok || a.comm_b || a.op_start || a.op_end || a.s_mb != 0 || a.n <= 0) return false;
    if (!lane_path(plan, a) || !lane_word_entries(plan->nlslots, plan->v, a.s_mb, 1)) return false;
    a.nslots = plan->nlslots;
    return lane_mbz_smem(plan->pmax, a, kManyLaneWarps) <= kLaneSmemLimit;
}

int64_t lane_mbz_warps(int pmax, const EvalArgs &a) {
    const int64_t ipw = 32 / pmax;  // instances per warp
    return (a.n + ipw - 1) / ipw;
}

int64_t lane_mbz_ctas(int pmax, const EvalArgs &a, int warps) {
    return (lane_mbz_warps(pmax, a) + warps - 1) / warps;
}

size_t lane_mbz_smem(int pmax, const EvalArgs &a, int warps) {
    switch (pmax) {
        case 4: return lane_smem<4>(a, warps, 1, true);
        case 8: return lane_smem<8>(a, warps, 1, true);
        case 16: return lane_smem<16>(a, warps, 1, true);
        default: return ~(size_t)0;
    }
}

template <int PMAX>
static int launch_lane_many_t(int warps, const ManyJob *d_jobs, int njobs, int64_t ctas, size_t smem,
                              cudaStream_t st) {
    int dev = 0;
    PPS_CUDA_TRY(cudaGetDevice(&dev));
    static std::atomic<bool> attr_set[64];  // per device, set once (idempotent)
    if (dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
        PPS_CUDA_TRY(cudaFuncSetAttribute(k_eval_lane_mbz_many<PMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)kLaneSmemLimit));
        attr_set[dev].store(true, std::memory_order_release);
    }
    k_eval_lane_mbz_many<PMAX><<<(unsigned)ctas, warps * 32, smem, st>>>(d_jobs, njobs);
    PPS_CUDA_TRY(cudaGetLastError());
    return PP_OK;
}

int launch_lane_mbz_many(int pmax, int warps, const ManyJob *d_jobs, int njobs, int64_t ctas, size_t smem,
                         cudaStream_t st) {
    if (njobs <= 0 || ctas <= 0) return PP_OK;
    if (ctas > 0x7FFFFFFF || smem > kLaneSmemLimit || warps < 1 || warps > kManyLaneWarps) return PP_ERR_SIZE;
    switch (pmax) {
        case 4: return launch_lane_many_t<4>(warps, d_jobs, njobs, ctas, smem, st);
        case 8: return launch_lane_many_t<8>(warps, d_jobs, njobs, ctas, smem, st);
        case 16: return launch_lane_many_t<16>(warps, d_jobs, njobs, ctas, smem, st);
        default: return PP_ERR_INTERNAL;
    }
}

}  // namespace pps
