// check.cuh -- the range checks of a checked build.
//
// Compiled with -DULYSSES_CHECK_BOUNDS, every plain global load and store a
// kernel makes (the TMA's tensor copies check their own bounds in hardware)
// first asks in_range whether the elements [first, first + count) lie inside
// the buffer's [0, limit).  A failed check sets ULYSSES_STATUS_BOUNDS in the
// status word (when the kernel has one) and the access is skipped: no trap,
// no fault, the context stays usable.  In a normal build in_range is the
// constant true and the checks compile away.
#pragma once

#include <stdint.h>

#include "../../include/ulysses.h"

namespace ulysses {

#ifdef ULYSSES_CHECK_BOUNDS
__device__ __forceinline__ bool in_range(uint32_t *status, long long first, long long count, long long limit) {
  if (first >= 0 && count >= 0 && first + count <= limit) return true;
  if (status) atomicOr(status, (uint32_t)ULYSSES_STATUS_BOUNDS);
  return false;
}
#else
__device__ __forceinline__ constexpr bool in_range(uint32_t *, long long, long long, long long) { return true; }
#endif

}  // namespace ulysses
