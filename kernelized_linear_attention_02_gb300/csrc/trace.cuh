// trace.cuh -- optional event trace of the tensor-core pipeline.
//
// Compiled in only with -DLA_TRACE (never in the shipped library): each
// role of the first kTraceCtas CTAs records (SM clock, role, event, index)
// at its pipeline hand-offs, so a timeline of one CTA can be reconstructed
// on the host.  Without LA_TRACE, LA_TR expands to nothing.
#pragma once

#include <stdint.h>

namespace la {
namespace trace {
constexpr int kTraceCtas = 4;
constexpr int kTraceEvents = 8192;
}  // namespace trace
}  // namespace la

#ifdef LA_TRACE
namespace la {
namespace trace {
// one buffer per translation unit (the head sizes compile separately)
static __device__ unsigned int g_count[kTraceCtas];
static __device__ unsigned long long g_time[kTraceCtas][kTraceEvents];
static __device__ unsigned int g_tag[kTraceCtas][kTraceEvents];
// Each role (up to 8) records from one thread into its own eighth of the buffer; the
// slot counter lives in shared memory so recording costs no global round trip.
__device__ __forceinline__ void record(unsigned* ctr, int role, int ev, int idx) {
#ifdef LA_TRACE_LAST_SEGMENT
    // the first kTraceCtas (batch, kv head) tiles of the last sequence segment
    const int cta = blockIdx.y + 1 == gridDim.y ? (int)blockIdx.x : kTraceCtas;
#else
    const int cta = blockIdx.x + blockIdx.y * gridDim.x;
#endif
    if (cta >= kTraceCtas) return;
    const unsigned slot = ctr[role]++;
    if (slot < (unsigned)(kTraceEvents / 8)) {
        const unsigned at = role * (kTraceEvents / 8) + slot;
        g_time[cta][at] = clock64();
        g_tag[cta][at] = (unsigned)(role << 24) | (unsigned)(ev << 16) | (unsigned)(idx & 0xffff);
    }
    if (role == 0 && ev == 9) g_count[cta] = kTraceEvents;  // end of the CTA
}
}  // namespace trace
}  // namespace la
#define LA_TR(role, ev, idx) ::la::trace::record(la_trace_ctr, (role), (ev), (idx))
#else
#define LA_TR(role, ev, idx) ((void)0)
#endif
