// Per-CTA timeline of a decode launch, for profiling only. Compiled in when
// PKV_TIMELINE is defined (the separate profiling build libpagedkv_timeline.so,
// see build.py); in the product build PKV_TL(...) expands to nothing and
// DecodeArgs carries no timeline pointer.
//
// Each CTA writes kTlEvents 64-bit words at timeline[cta * kTlEvents]: global
// timer readings (ns) of the events below, and one word of counts. The buffer
// is the caller's (attached with pkv_timeline_attach); CTAs past its length
// write nothing.
#pragma once

#include "pkv_ptx.cuh"

namespace pkv {

constexpr int kTlEvents = 12;
enum TimelineEvent {
  kTlStart = 0,       // kernel entry
  kTlPlanned = 1,     // the CTA's share is planned (after the wait for the previous grid)
  kTlFirstIssue = 2,  // producer: first tile copy issued
  kTlLastIssue = 3,   // producer: every tile copy issued (end of its walk)
  kTlFirstData = 4,   // consumers: first block (or chunk) has landed
  kTlLastData = 5,    // consumers: last block of the last piece consumed (recorded per piece)
  kTlExit = 6,        // consumers: done, epilogue and split merges included
  kTlInfo = 7,        // SM id (bits 0..15) | pieces (16..31) | blocks (32..63)
  kTlPieceOut = 8,    // last piece: its output or partial written (recorded per piece)
  kTlCounted = 9,     // last piece, if split: counted on the unit's counter
  kTlMerged = 10,     // last piece, if this CTA merged the unit: merge done
  kTlSpare = 11,
};

__device__ __forceinline__ unsigned long long sm_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

}  // namespace pkv

#ifdef PKV_TIMELINE
#define PKV_TL(a, ev)                                                                  \
  do {                                                                                 \
    if ((a).timeline && blockIdx.x < static_cast<unsigned>((a).timeline_ctas))        \
      (a).timeline[blockIdx.x * ::pkv::kTlEvents + (ev)] = ::pkv::global_timer_ns();   \
  } while (0)
#define PKV_TL_SET(a, ev, v)                                                           \
  do {                                                                                 \
    if ((a).timeline && blockIdx.x < static_cast<unsigned>((a).timeline_ctas))        \
      (a).timeline[blockIdx.x * ::pkv::kTlEvents + (ev)] = (v);                        \
  } while (0)
#else
#define PKV_TL(a, ev) ((void)0)
#define PKV_TL_SET(a, ev, v) ((void)0)
#endif
