// bounds.cuh — index checks of the bounds-checked build.
//
// Built with ORPO_DEBUG_BOUNDS, in_bounds(status, i, n) tests 0 <= i < n for an access whose index
// is computed (partial and block-max slots, skip bitmaps and tile lists, shared-memory tables,
// quantised weights and scales); a miss ORs ORPO_STATUS_BOUNDS into the status word and the caller
// skips the access, so a bad index is reported instead of touching memory.  Without the flag it is
// the constant true and every check compiles away.
#pragma once

#include <stdint.h>

#include "../../include/orpo_head.h"

namespace orpo {

__device__ __forceinline__ bool in_bounds(int32_t* status, int64_t i, int64_t n) {
#ifdef ORPO_DEBUG_BOUNDS
  if (i >= 0 && i < n) return true;
  if (status != nullptr) atomicOr(status, ORPO_STATUS_BOUNDS);
  return false;
#else
  (void)status;
  (void)i;
  (void)n;
  return true;
#endif
}

}  // namespace orpo
