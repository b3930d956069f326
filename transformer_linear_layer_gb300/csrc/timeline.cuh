// Kernel timelines: %globaltimer stamps at fixed points of a CTA's schedule,
// a measurement aid in the spirit of the probes of "One multiply, one RTX
// 5090, eight kernels" ("Where the time goes": time the loads and the math of
// a kernel separately to see which one its time belongs to). Compiled in only
// when the library is built with -DLIN_TIMELINE (the separate timeline build);
// in the library build every stamp is an empty statement and lin_timeline
// returns LIN_ERR_UNSUPPORTED.
//
// Each kernel file that stamps defines its own device array of
// kTimelineCtas x kTimelineSlots 64-bit nanosecond times (0 = not reached) and
// a host function that copies it out or clears it (timeline_copy_*).
#pragma once

#include <stdint.h>

namespace lin {

constexpr int kTimelineSlots = 192;   // stamps per CTA
constexpr int kTimelineCtas = 1024;   // CTA records per array

#ifdef LIN_TIMELINE
__device__ __forceinline__ unsigned long long timeline_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Stamp slot `idx` of CTA record `rec` in array `arr`.
#define LIN_STAMP(arr, rec, idx)                                                                  \
    do {                                                                                          \
        if ((idx) < ::lin::kTimelineSlots && (rec) < (unsigned)::lin::kTimelineCtas)              \
            (arr)[(size_t)(rec) * ::lin::kTimelineSlots + (idx)] = ::lin::timeline_now();         \
    } while (0)
#else
#define LIN_STAMP(arr, rec, idx) ((void)0)
#endif

}  // namespace lin
