// Per-CTA launch timeline for diagnostics: %globaltimer stamps at the phase
// boundaries of a kernel, one row of kTlSlots 64-bit words per CTA.
//
// The stamps are compiled only into a library built with -DSYMM_TIMELINE
// (the timeline variant of the build); the product library compiles every
// stamp to nothing.  Even there a kernel writes stamps only when the caller
// registered a buffer with symm_set_timeline, and only for CTAs whose row
// fits in it.  A slot holds either a time in ns (globaltimer) or a count
// (tl_value), as the kernel's own slot list says; a slot the launch did not
// reach holds 0.
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

// The CTA's row while the kernel runs: in shared memory, so that a stamp
// is not a global store that a later fence or release would have to wait
// for (that would stretch the very phases being measured); tl_end writes it
// out once, at the end.
__device__ __forceinline__ unsigned long long *tl_row() {
    __shared__ unsigned long long row[kTlSlots];
    return row;
}

// At kernel entry, by the thread that stamps first, before any stamp.
__device__ __forceinline__ void tl_begin() {
    if constexpr (kTimeline) {
        for (int i = 0; i < kTlSlots; ++i) tl_row()[i] = 0ull;
    }
}

// Writes the current time into slot `slot` of this CTA's row.
__device__ __forceinline__ void tl_stamp(unsigned long long *tl, int tl_ctas, int cta, int slot) {
    if constexpr (kTimeline) {
        if (tl && cta < tl_ctas) tl_row()[slot] = tl_now();
    }
}

// Writes a count into slot `slot` of this CTA's row.
__device__ __forceinline__ void tl_value(unsigned long long *tl, int tl_ctas, int cta, int slot,
                                         unsigned long long v) {
    if constexpr (kTimeline) {
        if (tl && cta < tl_ctas) tl_row()[slot] = v;
    }
}

// At kernel exit, by one thread, after every stamp of the CTA (a barrier
// between other threads' stamps and this): the row to CTA `cta`'s row of the
// registered buffer.
__device__ __forceinline__ void tl_end(unsigned long long *tl, int tl_ctas, int cta) {
    if constexpr (kTimeline) {
        if (tl && cta < tl_ctas)
            for (int i = 0; i < kTlSlots; ++i) tl[(size_t)cta * kTlSlots + i] = tl_row()[i];
    }
}

}  // namespace symm
