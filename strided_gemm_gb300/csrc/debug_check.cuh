// Device-side bounds checks of the debug build (compiled with -DSBGEMM_DEBUG).
//
// The host validates every operand's whole span before a launch (the
// StaleyNET "GPU Implementation" page, section "Safety": check every size the
// kernel depends on first).  A debug build also checks each address a kernel
// computes for a global load or store against that span, so that an indexing
// mistake in a kernel shows up as a status code instead of a stray access: an
// address outside the span records kBoundsViolation in the kernel's status
// word (read by sbgemm_device_status) and the caller skips the access.  The
// check never asserts or traps.  Release builds compile it away.
#pragma once

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace sbg {

// True when `ptr` lies inside the span of the operand whose base is `base`.
__device__ __forceinline__ bool dbg_in_span(const void* base, const void* ptr, const ElemSpan& s,
                                            unsigned int* status) {
#ifdef SBGEMM_DEBUG
    const int64_t off = static_cast<const float*>(ptr) - static_cast<const float*>(base);
    if (off < s.lo || off > s.hi) {
        record_status(status, kBoundsViolation);
        return false;
    }
#else
    (void)base; (void)ptr; (void)s; (void)status;
#endif
    return true;
}

// Whether this is the debug build.
constexpr bool kDebugChecks =
#ifdef SBGEMM_DEBUG
    true;
#else
    false;
#endif

}  // namespace sbg
