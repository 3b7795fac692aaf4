// checks.cuh - range checks of computed global-memory indices for the checked
// build of the library (compiled with -DNOMAS_BOUNDS_CHECK into
// libnomas_checked.so).  A failed check records NOMAS_ERR_INVALID_ARG in the
// device error word and the caller skips the access; nothing traps, so the
// context stays usable and the host reads the status afterwards.  In the
// regular build every check is the constant true and compiles away.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace nomas {

#ifdef NOMAS_BOUNDS_CHECK
constexpr bool kBoundsChecked = true;

// Elements [i, i + width) lie inside a buffer of n elements.
__device__ __forceinline__ bool in_bounds(long long i, long long width, long long n, uint32_t* err) {
  const bool ok = i >= 0 && width >= 0 && i + width <= n;
  if (!ok && err != nullptr) atomicCAS(err, 0u, 1u /* NOMAS_ERR_INVALID_ARG */);
  return ok;
}
#else
constexpr bool kBoundsChecked = false;

__device__ __forceinline__ bool in_bounds(long long, long long, long long, uint32_t*) { return true; }
#endif

}  // namespace nomas
