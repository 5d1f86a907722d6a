// internal.cuh -- definitions shared by the library's translation units.
#pragma once

#include <atomic>
#include <cstdint>
#include <deque>
#include <mutex>

#include <cuda_runtime.h>

#include "ppsched.h"

namespace pps {

// Per-round op descriptor, one uint32 per (round, device slot):
//   bits 0..1  kind: 0 idle, 1 forward, 2 backward
//   bits 2..7  chunk (virtual stage s = chunk*P + device)
//   bits 8..31 microbatch
constexpr uint32_t kIdle = 0, kFwd = 1, kBwd = 2;
__host__ __device__ inline uint32_t desc_pack(uint32_t kind, uint32_t chunk, uint32_t mb) {
    return kind | (chunk << 2) | (mb << 8);
}
__host__ __device__ inline uint32_t desc_kind(uint32_t d) { return d & 3u; }
__host__ __device__ inline uint32_t desc_chunk(uint32_t d) { return (d >> 2) & 63u; }
__host__ __device__ inline uint32_t desc_mb(uint32_t d) { return d >> 8; }

// Dependency-slot descriptor for the generic evaluator, one uint32 per
// (round, device slot):
//   bits 0..7   value slot this op reads its input arrival from (0xFF none)
//   bits 8..15  value slot this op writes its end tick to (0xFF none)
//   bits 16..23 boundary whose comm is added to the input (0xFF none)
constexpr uint32_t kNoSlot = 0xFFu;
__host__ __device__ inline uint32_t d2_pack(uint32_t rs, uint32_t ws, uint32_t cb) {
    return rs | (ws << 8) | (cb << 16);
}
__host__ __device__ inline uint32_t d2_rslot(uint32_t d) { return d & 0xFFu; }
__host__ __device__ inline uint32_t d2_wslot(uint32_t d) { return (d >> 8) & 0xFFu; }
__host__ __device__ inline uint32_t d2_cbnd(uint32_t d) { return (d >> 16) & 0xFFu; }

constexpr int kMaxValueSlots = 64;

// Per-round word, one uint64 per round:
//   bits 0..31  kind of device k in bits 2k..2k+1 (kIdle / kFwd / kBwd)
//   bits 32..39 pattern of the whole round, when every device runs an op and
//               the device count equals the table width:
//                 kPatAllF  every device runs a forward
//                 kPatAllB  every device runs a backward
//                 kPatAltA  even devices forward, odd devices backward
//                 kPatAltB  even devices backward, odd devices forward
//               (the 1F1B steady phase alternates A and B; GPipe's middle
//               rounds are all-F then all-B); kPatMasked + one of those when
//               only some devices run an op but each of them follows the
//               pattern (warmup and cooldown rounds); kPatGeneric otherwise.
//   bits 48..63 active-device mask (device k runs an op this round)
constexpr uint32_t kPatGeneric = 0, kPatAllF = 1, kPatAllB = 2, kPatAltA = 3, kPatAltB = 4;
constexpr uint32_t kPatMasked = 4;  // kPatMasked + kPatAllF .. kPatMasked + kPatAltB
__host__ __device__ inline uint32_t rw_kinds(uint64_t w) { return (uint32_t)w; }
__host__ __device__ inline uint32_t rw_pattern(uint64_t w) { return (uint32_t)(w >> 32) & 0xFFu; }
__host__ __device__ inline uint32_t rw_mask(uint64_t w) { return (uint32_t)(w >> 48); }

// Segments: maximal runs of rounds the register evaluator can run as one
// tight loop.  One uint4 per segment: {type, first round, end round, 0}.
//   kSegAltA / kSegAltB  rounds alternate kPatAltA / kPatAltB, starting as named
//   kSegAllF / kSegAllB  every round is kPatAllF / kPatAllB
//   kSegRound            one round, dispatched by its round word
constexpr uint32_t kSegRound = 0, kSegAltA = 1, kSegAltB = 2, kSegAllF = 3, kSegAllB = 4;

// Width of the device dimension a kernel is compiled for (>= P).
inline int pmax_for(int P) { return P <= 4 ? 4 : (P <= 8 ? 8 : 16); }

}  // namespace pps

// One device allocation shared by the tables of many plans (a batched build):
// freed when the last plan or table that references it is destroyed.
struct pp_arena {
    void *base = nullptr;
    std::atomic<int> refs{0};
};

// Kernel tables of the register evaluator for one (stride_stage, stride_mb)
// pair: loader table, round words and segments, contiguous, ready to be copied
// into shared memory.
struct pp_ktab {
    int64_t s_stage, s_mb;
    uint4 *d;         // words / 4 uint4
    int words;        // 32-bit words
    int variant = 0;  // layout variant (lane evaluator: instance sets per lane)
    pp_arena *arena = nullptr;  // the allocation d lives in, or null if d is its own
};

// The plan object (opaque to callers).
struct pp_plan {
    int policy, P, M, v, S, O;
    int R;              // rounds
    int pmax;           // row width of the per-round tables
    int nslots;         // value slots of the generic evaluator
    int nlslots;        // per-consumer value slots of the lane evaluator
    int reg_ok;         // 1 if the register evaluator applies
    int device;         // CUDA device the tables live on
    uint32_t *d_ops;    // [P][O] packed ops (PP_OP_* layout)
    int32_t *d_round;   // [P][O] wavefront round of each op
    uint32_t *d_desc;   // [R][pmax]
    uint32_t *d_desc2;  // [R][pmax] (generic evaluator), may be null
    uint8_t *d_lslot;   // [2][R][pmax] lane evaluator's local read / write slots (with d_desc2)
    uint64_t *d_rw;     // [R] per-round kind words and patterns
    uint4 *d_seg;       // [nseg] segments (register evaluator)
    int nseg;
    std::mutex ktab_mu; // guards ktabs
    std::deque<pp_ktab> ktabs;   // per stride pair, built on first use (stable addresses)
    std::deque<pp_ktab> ltabs;   // lane evaluator's tables, per stride pair (guarded by ktab_mu)
    int32_t *d_peak;    // [P]
    int32_t h_peak[PP_MAX_P];
    // Allocations the tables live in: [0] ops, rounds and peak; [1] desc, round
    // words and segments; [2] desc2 and lslot when built with the plan (then
    // slots_in_arena), else those two are allocations of their own.
    pp_arena *arena[3] = {nullptr, nullptr, nullptr};
    bool slots_in_arena = false;
};

namespace pps {

// Status helpers (host).
int cuda_status(cudaError_t e);

// Plan cache used by the evaluation entry points: returns the plan of the
// shape on the current device, building it on first use.
int cached_plan(int policy, int P, int M, int v, cudaStream_t stream, pp_plan **out);

// Build the plans of n shapes together: every step is one batched launch over
// all shapes, the tables of all shapes share three allocations, and the build
// synchronizes `stream` three times whatever n is.  out[i] is a new plan
// (value slots included for plans without the register path).
struct PlanShape {
    int policy, P, M, v;
};
int build_plans(const PlanShape *shapes, int n, cudaStream_t stream, pp_plan **out);
// cached_plan for n shapes: the shapes not cached yet are built in one batch.
int cached_plans(const PlanShape *shapes, int n, cudaStream_t stream, pp_plan **out);

// Kernel tables of many (plan, stride pair) requests: the missing ones are
// built in one allocation and a few batched launches on `stream`; the only
// synchronization is the upload of the job records from pageable host memory,
// which waits for `stream` to drain first.  Later work on `stream` sees the
// tables; other streams must wait for `stream`.  lane = 0: the register evaluator's tables (kernel_tables);
// lane = 1: the lane evaluator's tables with one instance set per lane.
struct TableReq {
    pp_plan *plan;
    int64_t s_stage, s_mb;
    int lane;
    const pp_ktab *out;
};
int build_tables(TableReq *reqs, int n, cudaStream_t stream);

// One table of a batched table build (device-side record).
struct TableJob {
    const uint32_t *desc;
    const uint64_t *rw;
    const uint4 *seg;
    const uint8_t *lslot;  // [2][R][pmax] (lane tables)
    int R, P, v, pmax, nseg, nslots, nblocks;
    int s_stage, s_mb;
    int word;  // lane tables: one-word entries
    int64_t words;
    uint32_t *out;
};
// Lane evaluator tables (eval_lane.cu): whether a table has one-word entries
// (costs shared by all microbatches, small enough offsets), words of one
// table with one instance set per lane, and the batched build of such tables
// for one table width.
bool lane_word_entries(int nslots, int v, int64_t s_mb, int ni);
int64_t lane_table_words(int pmax, int R, bool word, int *nblocks);
int launch_ltab_batch(int pmax, const TableJob *d_jobs, int njobs, int64_t max_words, cudaStream_t stream);
// Value slots for a plan built without them (register plans get them on
// first need); PP_ERR_SIZE if too many results would be in flight.
int plan_value_slots(pp_plan *plan, cudaStream_t stream);

// Argument validation shared by plan construction and evaluation.
int check_shape(int policy, int P, int M, int v);

// Shared-memory words of the register evaluator's per-block tables: loader
// table [R][pmax] (padded to 16 bytes), round words [R] (padded to 16 bytes),
// segments [nseg].
__host__ __device__ inline int ktab_words(int R, int pmax, int nseg) {
    return ((R * pmax + 3) & ~3) + 2 * ((R + 1) & ~1) + 4 * nseg;
}

// The kernel tables of `plan` for the given strides, built (allocating device
// memory and synchronizing `stream`) the first time a stride pair is seen.
int kernel_tables(pp_plan *plan, int64_t s_stage, int64_t s_mb, cudaStream_t stream, const pp_ktab **out);

// A GPipe / 1F1B plan laid out in device memory the caller provides (used by
// the entry point that allocates nothing).  Every table lives in `region`.
struct ScratchPlan {
    uint32_t *region;
    int64_t region_words, used_words;
    int policy, P, M, R, pmax, nseg;
    uint32_t *desc;
    uint64_t *rw;
    uint4 *seg;
    int32_t *peak;
    uint32_t *ktab;  // kernel tables for one stride pair, or null
    int ktab_words;
};

// Build the plan of (policy, P, M) for GPipe or 1F1B into `region` (device
// words).  Synchronizes `stream` twice; PP_ERR_SIZE if the region is too small.
int plan_into(int policy, int P, int M, uint32_t *region, int64_t region_words, cudaStream_t stream,
              ScratchPlan *sp);
// Append the kernel tables for one stride pair to the plan's region.
int ktab_into(ScratchPlan *sp, int64_t s_stage, int64_t s_mb, cudaStream_t stream);

}  // namespace pps

#define PPS_CUDA_TRY(expr)                                  \
    do {                                                    \
        cudaError_t e_ = (expr);                            \
        if (e_ != cudaSuccess) return pps::cuda_status(e_); \
    } while (0)
