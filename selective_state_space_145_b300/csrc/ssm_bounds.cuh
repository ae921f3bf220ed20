// ssm_bounds.cuh -- range checks of the debug build.
//
// Built with SSM_DEBUG_BOUNDS (libssm_debug.so), every checked global-memory access first tests
// its element range [first, first + count) against the extent of the tensor it touches. A range
// outside the tensor sets this translation unit's bit in a device error word (atomicOr) and the
// access is skipped (a skipped load reads as zero): a wrong index is recorded, never followed,
// and nothing traps. The host reads and clears the words through ssm_debug_bounds_status.
// Without the macro the checks are the constant true and the kernels are those of libssm.so.
#pragma once

#include <cuda_runtime.h>

namespace ssm {

// Bits of the error word, one per kernel family.
constexpr unsigned kBoundsScan = 1u;       // scan main and carry passes
constexpr unsigned kBoundsDecode = 2u;     // decode state update
constexpr unsigned kBoundsConv = 4u;       // standalone causal conv, forward and backward
constexpr unsigned kBoundsSegment = 8u;    // segment aggregate fold and composition
constexpr unsigned kBoundsBackward = 16u;  // scan backward: checkpoint, reverse and reduction kernels
constexpr unsigned kBoundsSsd = 32u;       // state-space-duality layer (its plain copies and stores)

// [first, first + count) lies within [0, extent).
__host__ __device__ constexpr bool range_ok(long long first, long long count, long long extent) {
  return first >= 0 && count >= 0 && first <= extent && count <= extent - first;
}
static_assert(range_ok(0, 0, 0) && range_ok(0, 4, 4) && range_ok(3, 1, 4) && range_ok(4, 0, 4), "in range");
static_assert(!range_ok(-1, 1, 4) && !range_ok(1, 4, 4) && !range_ok(4, 1, 4) && !range_ok(0, -1, 4), "out of range");
static_assert(!range_ok(1, 0x7fffffffffffffffLL, 8), "no overflow of first + count");

#ifdef SSM_DEBUG_BOUNDS
// One word per translation unit (the library is not compiled for separate device linking).
static __device__ unsigned int g_bounds_flags = 0u;

__device__ __forceinline__ bool in_bounds(long long first, long long count, long long extent, unsigned bit) {
  if (range_ok(first, count, extent)) return true;
  atomicOr(&g_bounds_flags, bit);
  return false;
}

// This translation unit's word (host side); cleared when `clear` is set.
static inline cudaError_t bounds_flags_read(unsigned* out, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_bounds_flags, sizeof(unsigned));
  if (e == cudaSuccess && clear) {
    const unsigned zero = 0u;
    e = cudaMemcpyToSymbol(g_bounds_flags, &zero, sizeof(unsigned));
  }
  return e;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(long long, long long, long long, unsigned) { return true; }
#endif

// The same check for a pointer p into the tensor that starts at base: [p, p + count) within
// [base, base + extent).
template <typename P>
__device__ __forceinline__ bool ptr_in(const P* base, const P* p, long long count, long long extent, unsigned bit) {
  return in_bounds((long long)(p - base), count, extent, bit);
}

}  // namespace ssm
