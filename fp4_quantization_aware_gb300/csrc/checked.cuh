// Bounds checks of the debug build (compiled with -DATTNQAT_CHECKED into
// libattnqat_checked.so; the product build compiles them away).
//
// Every plain global load and store of the kernels (TMA copies are clipped by
// their tensor maps and need none) sits behind ATTNQAT_IN_BOUNDS(cond), where
// cond states that the element index lies inside the extent of the buffer it
// addresses (the extent the host passes in the kernel's arguments, not the
// index arithmetic that produced it). In the debug build a false cond skips
// the access and counts it in a device counter of the translation unit, which
// attnqat_debug_oob_count reads and clears; the kernel carries on, so a bad
// index shows up as a count, never as a fault. In the product build the macro
// is the constant true and its condition is not compiled.
#pragma once
#include <cuda_runtime.h>

namespace attnqat {

#ifdef ATTNQAT_CHECKED
namespace {
__device__ unsigned long long g_oob_count;   // one per translation unit
}
__device__ __forceinline__ bool in_bounds(bool ok) {
  if (!ok) atomicAdd(&g_oob_count, 1ull);
  return ok;
}
#define ATTNQAT_IN_BOUNDS(cond) (::attnqat::in_bounds(cond))
#define ATTNQAT_CHECKED_ONLY(...) __VA_ARGS__
// Host reader of this translation unit's counter (adds it to *out; clears it
// when asked).
#define ATTNQAT_OOB_READER(name)                                                            \
  cudaError_t name(unsigned long long* out, bool clear) {                                   \
    unsigned long long v = 0;                                                               \
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_oob_count, sizeof(v));                       \
    if (e != cudaSuccess) return e;                                                         \
    *out += v;                                                                              \
    if (clear) {                                                                            \
      const unsigned long long zero = 0;                                                    \
      e = cudaMemcpyToSymbol(g_oob_count, &zero, sizeof(zero));                             \
    }                                                                                       \
    return e;                                                                               \
  }
#else
#define ATTNQAT_IN_BOUNDS(cond) (true)
#define ATTNQAT_CHECKED_ONLY(...)
#define ATTNQAT_OOB_READER(name) \
  cudaError_t name(unsigned long long*, bool) { return cudaSuccess; }
#endif

}  // namespace attnqat
