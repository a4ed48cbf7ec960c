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

constexpr int kTlEvents = 28;
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
  // tcgen05 kernel: SM cycles (clock64) summed over the CTA's chunks
  kTlSteps = 12,      // 12..21: the softmax loop's steps, thread 0 (kTlStepNames in timeline.py)
  kTlMmaWaitK = 22,   // MMA thread: waiting for a chunk's K (and Q)
  kTlMmaWaitPV = 23,  // MMA thread: waiting for a chunk's P and V
  kTlMmaTotal = 24,   // MMA thread: its whole loop
  kTlProdWait = 25,   // producer: waiting for a free ring buffer
  kTlProdTotal = 26,  // producer: its whole loop
};
constexpr int kTlNumSteps = 10;

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
// Step accounting inside a loop: PKV_TL_STEP_BEGIN declares the accumulators,
// PKV_TL_STEP(k) adds the cycles since the previous mark to step k.
#define PKV_TL_STEP_BEGIN                      \
  long long tl_acc[::pkv::kTlNumSteps] = {};   \
  long long tl_last = clock64()
#define PKV_TL_STEP(k)                         \
  do {                                         \
    const long long tl_now = clock64();        \
    tl_acc[k] += tl_now - tl_last;             \
    tl_last = tl_now;                          \
  } while (0)
#define PKV_TL_STEP_FLUSH(a)                                         \
  do {                                                               \
    for (int tl_k = 0; tl_k < ::pkv::kTlNumSteps; ++tl_k)            \
      PKV_TL_SET(a, ::pkv::kTlSteps + tl_k, tl_acc[tl_k]);           \
  } while (0)
// The first wait of the CTA that gives up records where: site (bits 0..7), chunk
// (8..31), thread (32..47).
#define PKV_TL_TIMEOUT(a, site, chunk)                                                       \
  do {                                                                                       \
    if ((a).timeline && blockIdx.x < static_cast<unsigned>((a).timeline_ctas))              \
      atomicCAS((a).timeline + blockIdx.x * ::pkv::kTlEvents + ::pkv::kTlSpare, 0ull,      \
                static_cast<unsigned long long>(site) |                                      \
                    (static_cast<unsigned long long>((chunk) & 0xFFFFFF) << 8) |             \
                    (static_cast<unsigned long long>(threadIdx.x) << 32));                  \
  } while (0)
#else
#define PKV_TL(a, ev) ((void)0)
#define PKV_TL_SET(a, ev, v) ((void)0)
#define PKV_TL_TIMEOUT(a, site, chunk) ((void)0)
#define PKV_TL_STEP_BEGIN ((void)0)
#define PKV_TL_STEP(k) ((void)0)
#define PKV_TL_STEP_FLUSH(a) ((void)0)
#endif
