// Device code shared by the two decode kernels (the mma.sync kernel for narrow
// units and the tcgen05 kernel for wide ones): the CTA's share of the batch,
// bounded mbarrier waits, and the fused split-KV combine.
//
// Work partition. The batch's units (sequence, KV head), sequence-major, lie on
// a work line: each unit a fixed number of positions for its per-piece work, then
// one position per KV block. The line is cut into contiguous equal shares, one
// per active CTA. A CTA's share covers whole units and at most two partial ones
// (its first and last). A unit handled whole writes its output
// directly; a unit cut across CTAs is computed as pieces, each piece writes
// (m, l, o) -- running max, sum of exponentials, unnormalised output, in base 2
// -- to workspace slot (unit + cta), and the CTA that completes the unit's last
// piece merges them: M = max m, L = sum l 2^(m-M), out = sum o 2^(m-M) / L, the
// split-softmax rule of "AI 大模型推理优化技术详解" (2.2.1 Flash Attention).
#pragma once

#include <cuda_runtime.h>
#include <math.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {

// Blocks of one (sequence, KV head) unit. A context length outside
// [1, max_blocks*16] is clamped so that every unit owns at least one block (and
// so gets its output written) and never reads past its block-table row.
__device__ __forceinline__ int unit_blocks(int ctx, int mbs) {
  int c = ctx < 1 ? 1 : ctx;
  const int cap = mbs * kBlockSize;
  c = c > cap ? cap : c;
  return (c + kBlockSize - 1) / kBlockSize;
}

// Wait for an mbarrier phase; gives up after kWaitLimitNs or when another warp
// of the CTA has already given up (abort flag in shared memory).
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

template <int KV>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
  if constexpr (KV == kKvBf16) {
    return pack_bf16x2(lo, hi);
  } else {
    return pack_f16x2(lo, hi);
  }
}

// The work is a line of positions: unit (s, h) in order, each a fixed
// a.piece_cost positions (its per-piece work: queries, epilogue, split merge,
// counted in blocks) followed by one position per KV block. CTAs take equal
// shares of the line, so a CTA whose share starts more units takes fewer blocks.
// A unit whose blocks start at position ub is served by the CTAs that own
// positions ub .. ub + nb - 1.

// CTAs that take work: each active CTA's share spans at least piece_cost + 1
// positions, so it holds at least one block.
__device__ __forceinline__ long long active_ctas(long long ncta, long long total, int piece_cost) {
  const long long cap = total / (piece_cost + 1);
  return ncta < cap ? ncta : (cap > 0 ? cap : 1);
}

// The CTA that owns position p of the line.
__device__ __forceinline__ int position_owner(long long p, long long nact, long long total) {
  return static_cast<int>(((p + 1) * nact - 1) / total);
}

// This CTA's share [b0, b1) of the line. Every thread of the CTA calls it. One
// pass over context_lens: thread t owns a contiguous run of sequences, a
// block-wide scan of the runs' lengths on the line gives the total and every
// run's offset, and the thread whose run holds position b0 finds its sequence.
// Results in plan[0..4] = total, b0, b1, first sequence s0, and the line length
// per head of the sequences before s0 (plan[3] = -1 if the share is empty).
// red must hold one long long per warp.
__device__ inline void plan_cta_share(const DecodeArgs& a, long long* red, long long* plan) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nwarps = blockDim.x >> 5;
  const int S = a.num_seqs, Hkv = a.num_kv_heads, mbs = a.max_blocks_per_seq;
  const long long ncta = gridDim.x, cta = blockIdx.x;
  const int per = (S + blockDim.x - 1) / blockDim.x;
  const int s_lo = tid * per;
  const int s_hi = s_lo + per < S ? s_lo + per : S;
  long long mine = 0;
  for (int s = s_lo; s < s_hi; ++s) mine += unit_blocks(a.context_lens[s], mbs) + a.piece_cost;
  mine *= Hkv;
  long long v = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) red[warp] = v;
  if (tid == 0) plan[3] = -1;
  __syncthreads();
  long long pre = 0, tot = 0;
  for (int w = 0; w < nwarps; ++w) {
    if (w < warp) pre += red[w];
    tot += red[w];
  }
  const long long excl = pre + v - mine;
  // Only active_ctas() CTAs take work, so every active CTA owns at least one
  // block and every CTA between a unit's first and last owner wrote a piece of it.
  const long long nact = active_ctas(ncta, tot, a.piece_cost);
  const long long b0 = cta < nact ? cta * tot / nact : tot;
  const long long b1 = cta < nact ? (cta + 1) * tot / nact : tot;
  if (b0 < b1 && excl <= b0 && b0 < excl + mine) {
    long long cum = excl;
    for (int s = s_lo; s < s_hi; ++s) {
      const long long wblk = static_cast<long long>(Hkv) * (unit_blocks(a.context_lens[s], mbs) + a.piece_cost);
      if (b0 < cum + wblk) {
        plan[3] = s;
        plan[4] = cum / Hkv;
        break;
      }
      cum += wblk;
    }
  }
  if (tid == 0) { plan[0] = tot; plan[1] = b0; plan[2] = b1; }
  __syncthreads();
}

// After this CTA wrote its piece of unit u to slot (u + cta): count the piece on
// the unit's counter; the CTA that finishes the last piece merges all pieces
// into the output. Called by the nthr threads that wrote the slot (tid in
// [0, nthr)), which synchronise on named barrier bar_id. ustart is the line
// position of the unit's first block, nb its block count, Rs its real rows, qb its first query
// row. Counters are tagged with the call's epoch, so no workspace clearing is
// needed, and the CTA that completes a unit clears its counter, so a replayed
// CUDA graph (same epoch every replay) starts from clear counters too.
template <int KV, int D>
__device__ inline void finish_split_piece(const DecodeArgs& a, int u, long long ustart, int nb,
                                          long long total, long long ncta, int Rs, int qb, int h,
                                          int tid, int nthr, int bar_id, volatile int* fin) {
  constexpr float kNegInf = -INFINITY;
  const int R = a.rows, G = a.group, Hq = a.num_q_heads;
  // The barrier orders every thread's slot writes before thread 0's device-scope
  // release fence, which makes them visible before the counter update; the CTA
  // that sees the final count acquires the other CTAs' slots through the same
  // fence after its atomic.
  named_bar_sync(bar_id, nthr);
  if (tid == 0) {
    fence_acq_rel_gpu();
    const long long nact = active_ctas(ncta, total, a.piece_cost);
    const int c_first = position_owner(ustart, nact, total);
    const int c_last = position_owner(ustart + nb - 1, nact, total);
    unsigned long long* ctr = a.piece_counts + u;
    unsigned long long cur = atomicAdd(ctr, 0ull);
    unsigned long long want;
    for (;;) {
      want = (static_cast<uint32_t>(cur >> 32) == a.epoch)
                 ? cur + 1ull
                 : ((static_cast<unsigned long long>(a.epoch) << 32) | 1ull);
      const unsigned long long prev = atomicCAS(ctr, cur, want);
      if (prev == cur) break;
      cur = prev;
    }
    const bool last = static_cast<int>(want & 0xffffffffull) == c_last - c_first + 1;
    fin[0] = last ? 1 : 0;
    fin[1] = c_first;
    fin[2] = c_last;
    if (last) {
      // No other CTA touches this counter again in this launch. Leave it at 0
      // (epoch 0 is never issued, so 0 reads as "no pieces" for any later call):
      // a replayed CUDA graph reuses its epoch and must find the counters clear.
      *ctr = 0ull;
      fence_acq_rel_gpu();   // acquire: the other CTAs' slots are read next
    }
  }
  named_bar_sync(bar_id, nthr);
  if (!fin[0]) return;
  // Merge: out = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c with M = max_c m_c,
  // accumulated online (the running max moves as slots are read). A thread reads
  // four slots per step, so their loads are in flight together instead of one
  // round trip per slot.
  const int c_first = fin[1], c_last = fin[2];
  const int ooff = partial_o_offset(R);
  const float* base = a.partials + static_cast<size_t>(u) * a.slot_floats;   // slot of CTA c: + c * slot_floats
#pragma unroll 1
  for (int idx = tid; idx < Rs * (D / 4); idx += nthr) {
    const int r = idx / (D / 4), d4 = idx - (idx / (D / 4)) * (D / 4);
    float M = kNegInf, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int c0 = c_first; c0 <= c_last; c0 += 4) {
      float mc[4], lc[4];
      float4 oc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const bool live = c0 + k <= c_last;
        const float* P = base + static_cast<size_t>(live ? c0 + k : c_first) * a.slot_floats;
        mc[k] = live ? __ldcg(P + r) : kNegInf;
        lc[k] = live ? __ldcg(P + R + r) : 0.f;
        oc[k] = live ? __ldcg(reinterpret_cast<const float4*>(P + ooff + r * D + d4 * 4))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float Mn = fmaxf(M, mc[k]);
        const float Mu = (Mn == kNegInf) ? 0.f : Mn;
        const float fo = fast_exp2(M - Mu), fc = fast_exp2(mc[k] - Mu);
        L = L * fo + fc * lc[k];
        acc.x = acc.x * fo + fc * oc[k].x;
        acc.y = acc.y * fo + fc * oc[k].y;
        acc.z = acc.z * fo + fc * oc[k].z;
        acc.w = acc.w * fo + fc * oc[k].w;
        M = Mn;
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int j = r / G, gi = r - j * G;
    const size_t dst = (static_cast<size_t>(qb + j) * Hq + h * G + gi) * D + d4 * 4;
    uint2 pk;
    pk.x = pack_p<KV>(acc.x * inv, acc.y * inv);
    pk.y = pack_p<KV>(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + dst) = pk;
  }
}

}  // namespace pkv
