// Arrival counters of the decode kernel's split-KV merge, written for host and device so
// that the protocol can be driven on the CPU as well.
//
// A pair cut between CTAs leaves one piece per CTA; each piece is counted in at the pair's
// counter, and the arrival that completes the count merges the pieces.  A counter holds
// tag << 24 | count, the tag being 40 bits that differ from call to call.  A counter with
// another tag (an earlier call's, or workspace never written) counts as zero.  The
// arrival that completes a pair stores tag << 24 (count zero) in place of the full count,
// so the counter is zero again when the call ends: a later call with the same tag (a
// captured CUDA graph replayed) starts from zero as well.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define PA_HOST_DEVICE __host__ __device__ __forceinline__
#else
#define PA_HOST_DEVICE inline
#endif

namespace pa {

constexpr int kArriveTries = 1 << 20;
constexpr unsigned long long kArriveCountMask = 0xffffffull;

// Count one piece in at *ctr for a pair of n pieces.  cas(ptr, expected, desired) is an
// atomic compare-and-swap returning the old value; load(ptr) reads the counter.  Returns
// the count this arrival makes (1 .. n; n means it completed the pair), or -1 when `tries`
// compare-and-swaps in a row found the counter changed (the caller flags the pair).
#if defined(__CUDACC__)
#pragma nv_exec_check_disable
#endif
template <class Cas, class Load>
PA_HOST_DEVICE int arrive_count(unsigned long long* ctr, unsigned long long tag, int n, Cas cas,
                                Load load, int tries = kArriveTries) {
  unsigned long long cur = load(ctr);
  for (int t = 0; t < tries; ++t) {
    const unsigned long long base = (cur >> 24) == tag ? cur : (tag << 24);
    const int count = static_cast<int>(base & kArriveCountMask) + 1;
    const unsigned long long want = count >= n ? (tag << 24) : base + 1;
    const unsigned long long prev = cas(ctr, cur, want);
    if (prev == cur) return count;
    cur = prev;
  }
  return -1;
}

}  // namespace pa
