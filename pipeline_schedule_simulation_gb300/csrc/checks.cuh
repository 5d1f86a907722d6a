// checks.cuh -- the bounds-checked build of the library (-DPPS_CHECKED).
//
// A memory checker is not available on every machine this library runs on,
// so the kernels can be compiled with checks of their own.  Every address a
// kernel takes from a run-time table or from caller-provided sizes -- a
// plan's loader entries, value-slot and comm-row offsets, a search's split
// points, the cost rows a state machine fetches -- is checked against the
// region it must stay in before it is used.  A failed check skips the access
// (a load reads 0, a copy is zero-filled, a store is dropped) and records the
// first failure of the translation unit in a device word: bit 63 set, the
// check site in bits 40..55, the low 40 bits of the offending offset below.
// Nothing traps, so the context stays usable.  In the normal build every
// check is the constant `true` and compiles to nothing.
// pp_sched_debug_checks (host_entry.cu) reads and clears the words.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace pps {

enum CheckSite : uint32_t {
    kChkCostRead = 1,   // a cost element outside what the strides reach
    kChkLaneSlotRead,   // lane evaluator: input slot cell outside the warp's value rows
    kChkLaneSlotWrite,  // lane evaluator: result slot cell outside the warp's value rows
    kChkLaneComm,       // lane evaluator: comm / {cost, comm} cell outside the warp's rows
    kChkSlotIndex,      // slot evaluator: a slot index at or beyond the plan's slot count
    kChkSearchSplit,    // search: a split point outside 0..L
};

// The elements a cost table addressed with these strides spans from its base:
// 1 + (n-1)*s_inst + (S-1)*s_stage + (M-1)*s_mb, 0 for an empty batch.
__host__ __device__ inline int64_t cost_reach(int64_t n, int S, int M, int64_t s_inst, int64_t s_stage,
                                              int64_t s_mb) {
    return n <= 0 ? 0 : 1 + (n - 1) * s_inst + (int64_t)(S - 1) * s_stage + (int64_t)(M - 1) * s_mb;
}

#ifdef PPS_CHECKED
// One word per translation unit (device code is compiled per unit).
static __device__ unsigned long long g_check_word;

__device__ __forceinline__ bool check_ok(bool ok, uint32_t site, uint64_t v) {
    if (!ok)
        atomicCAS(&g_check_word, 0ull,
                  (1ull << 63) | ((unsigned long long)(site & 0xFFFFu) << 40) | (v & ((1ull << 40) - 1)));
    return ok;
}

// Host side: every unit registers a reader of its word at load time.
int register_check_reader(uint64_t (*reader)());

static uint64_t take_check_word() {
    unsigned long long v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_check_word, sizeof(v)) != cudaSuccess) return 0;
    (void)cudaMemcpyToSymbol(g_check_word, &zero, sizeof(zero));
    return v;
}

[[maybe_unused]] static const int g_check_reader = register_check_reader(take_check_word);

#define PPS_CHECK(cond, site, value) ::pps::check_ok((cond), (site), (uint64_t)(value))
#else
#define PPS_CHECK(cond, site, value) true
#endif

}  // namespace pps
