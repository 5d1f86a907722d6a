// search_common.cuh -- pieces shared by the partition searches: the seeded
// candidate draw and binomial coefficients for colex unranking.
#pragma once

#include <cstdint>

#include "checks.cuh"

namespace pps {

// SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): add the golden gamma to the
// state, then apply the two xor-shift-multiply rounds and a final xor-shift.
__device__ __forceinline__ uint64_t splitmix64(uint64_t s) {
    uint64_t z = s + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// C(n, i) by the multiplicative formula, exact at every step (each partial
// product is itself a binomial coefficient); ~0 when it exceeds 64 bits.
__host__ __device__ inline uint64_t binom_u64(int n, int i) {
    if (i < 0 || i > n) return 0;
    if (i > n - i) i = n - i;
    unsigned __int128 acc = 1;
    for (int t = 1; t <= i; ++t) {
        acc = acc * (unsigned)(n - i + t) / (unsigned)t;
        if (acc > (unsigned __int128)0xFFFFFFFFFFFFFFFFull) return ~0ull;
    }
    return (uint64_t)acc;
}

}  // namespace pps
