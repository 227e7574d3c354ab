// Per-CTA launch timeline for diagnostics: %globaltimer stamps at the phase
// boundaries of a kernel, one row of kTlSlots 64-bit words per CTA.
//
// The stamps are compiled only into a library built with -DSYMM_TIMELINE
// (the timeline variant of the build); the product library compiles every
// stamp to nothing.  Even there a kernel writes stamps only when the caller
// registered a buffer with symm_set_timeline, and only for CTAs whose row
// fits in it.  A slot holds either a time in ns (globaltimer) or a count
// (tl_value), as the kernel's own slot list says.
#pragma once

#include <stdint.h>

namespace symm {

constexpr int kTlSlots = 16;

#ifdef SYMM_TIMELINE
constexpr bool kTimeline = true;
#else
constexpr bool kTimeline = false;
#endif

__device__ __forceinline__ unsigned long long tl_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Writes the current time into slot `slot` of CTA `cta`'s row.
__device__ __forceinline__ void tl_stamp(unsigned long long *tl, int tl_ctas, int cta, int slot) {
    if constexpr (kTimeline) {
        if (tl && cta < tl_ctas) tl[(size_t)cta * kTlSlots + slot] = tl_now();
    }
}

// Writes a count into slot `slot` of CTA `cta`'s row.
__device__ __forceinline__ void tl_value(unsigned long long *tl, int tl_ctas, int cta, int slot,
                                         unsigned long long v) {
    if constexpr (kTimeline) {
        if (tl && cta < tl_ctas) tl[(size_t)cta * kTlSlots + slot] = v;
    }
}

}  // namespace symm
