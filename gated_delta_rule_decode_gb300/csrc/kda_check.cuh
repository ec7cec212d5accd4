// Bounds checks of the checked build (-DKDA_CHECKED), the stand-in for a
// memory checker: an access whose element range [off, off + n) leaves its
// buffer [0, size) records KDA_DEVERR_BOUNDS in the call's error flag and is
// skipped (no trap, no assert: the kernel carries on).  The normal build
// compiles every check to `true`.
#pragma once

#include <stdint.h>

#include "kda.h"

namespace kda {

__device__ __forceinline__ bool in_bounds(int64_t off, int64_t n, int64_t size, int32_t *flag) {
#ifdef KDA_CHECKED
    if (off >= 0 && n >= 0 && off <= size - n) return true;
    if (flag) atomicOr(flag, KDA_DEVERR_BOUNDS);
    return false;
#else
    (void)off, (void)n, (void)size, (void)flag;
    return true;
#endif
}

}  // namespace kda
