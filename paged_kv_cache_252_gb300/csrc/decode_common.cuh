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
#include "pkv_timeline.cuh"

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

// Wait for an mbarrier phase; gives up after limit_ns or when another warp of the
// CTA has already given up (abort flag in shared memory).
__device__ __forceinline__ bool wait_or_abort_for(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
}

// The decode kernels' waits: limit kWaitLimitNs.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag) {
  return wait_or_abort_for(bar, parity, abort_flag, kWaitLimitNs);
}

template <int KV>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
  if constexpr (KV == kKvBf16) {
    return pack_bf16x2(lo, hi);
  } else {
    return pack_f16x2(lo, hi);
  }
}

// Before the wait for the previous grid: bring into L2 the lines the plan and the
// first copies read, context_lens (every CTA plans from all of it) and the block
// tables (each CTA fetches its slice of them, so the grid fetches them all; skipped
// when a slice would exceed 32 lines). L2 is where a previous grid's writes land,
// so a line fetched early still reads current after the wait; nothing is read here.
// Out of line: inlined, its few registers shifted the kernels' allocation.
static __device__ __noinline__ void prefetch_plan_inputs(const int32_t* context_lens, const int32_t* block_tables,
                                                        int num_seqs, int max_blocks_per_seq) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  for (int line = tid; line < (num_seqs + 31) / 32; line += nthr) prefetch_l2(context_lens + 32 * line);
  // Lines of the block tables (32 entries each; the host keeps num_seqs * max_blocks_per_seq < 2^31).
  const int bt_lines = static_cast<int>((static_cast<long long>(num_seqs) * max_blocks_per_seq + 31) / 32);
  const int per = (bt_lines + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
  if (per <= 32 && tid < per) {
    const long long line = static_cast<long long>(blockIdx.x) * per + tid;
    if (line < bt_lines) prefetch_l2(block_tables + 32 * line);
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

// Merge the pieces of unit u into its output rows: M = max m, L = sum l 2^(m-M),
// out = sum o 2^(m-M) / L over the pieces of CTAs c_first..c_last, in that order,
// accumulated online. Each piece comes from its workspace slot (unit + cta),
// except that when own_o is not null the piece of CTA c_first (this CTA) is read
// from shared memory (o at own_o[r * own_stride + d], m and l at own_ml[r] and
// own_ml[rows + r]) -- the same values its slot would hold, combined in the same
// order, so either way gives the same output bits. A thread reads four slots per
// step, so their loads are in flight together instead of one round trip per slot.
template <int KV, int D>
__device__ inline void merge_split_pieces(const DecodeArgs& a, int u, int c_first, int c_last,
                                          const float* own_o, int own_stride, const float* own_ml,
                                          int Rs, int qb, int h, int tid, int nthr) {
  constexpr float kNegInf = -INFINITY;
  const int R = a.rows, G = a.group, Hq = a.num_q_heads;
  const int ooff = partial_o_offset(R);
  const float* base = a.partials + static_cast<size_t>(u) * a.slot_floats;   // slot of CTA c: + c * slot_floats
  const int c_read = own_o ? c_first + 1 : c_first;                           // first slot read from memory
#pragma unroll 1
  for (int idx = tid; idx < Rs * (D / 4); idx += nthr) {
    const int r = idx / (D / 4), d4 = idx - (idx / (D / 4)) * (D / 4);
    float M = kNegInf, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (own_o) {
      // Combining the first piece into the empty state gives exactly its own values.
      M = own_ml[r];
      L = own_ml[R + r];
      acc = *reinterpret_cast<const float4*>(own_o + r * own_stride + d4 * 4);
    }
#pragma unroll 1
    for (int c0 = c_read; c0 <= c_last; c0 += 4) {
      float mc[4], lc[4];
      float4 oc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const bool live = c0 + k <= c_last;
        const float* P = base + static_cast<size_t>(live ? c0 + k : c_read) * a.slot_floats;
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

// CTAs that hold pieces of a unit whose first block is at line position ustart
// (nb blocks): c_first .. c_last.
__device__ __forceinline__ void unit_owners(const DecodeArgs& a, long long ustart, int nb, long long total,
                                            long long ncta, int* c_first, int* c_last) {
  const long long nact = active_ctas(ncta, total, a.piece_cost);
  *c_first = position_owner(ustart, nact, total);
  *c_last = position_owner(ustart + nb - 1, nact, total);
}

// Count a published piece on unit u's counter (thread 0 only; the slot writes of
// the CTA are ordered before it by the caller's barrier and the release fence
// here). cur is a guess of the counter's value; a wrong guess costs one more CAS,
// which returns the actual value. Counters are tagged with the call's epoch, so
// no workspace clearing is needed: a counter left by an earlier call reads as
// zero. Returns true for the piece that completes the unit (then with acquire
// ordering for the other CTAs' slots).
__device__ __forceinline__ bool count_published_piece(const DecodeArgs& a, int u, unsigned long long cur,
                                                      int c_first, int c_last) {
  fence_acq_rel_gpu();
  unsigned long long* ctr = a.piece_counts + u;
  const unsigned long long tag = static_cast<unsigned long long>(a.epoch) << 32;
  unsigned long long want;
  for (;;) {
    want = (static_cast<uint32_t>(cur >> 32) == a.epoch) ? cur + 1ull : (tag | 1ull);
    const unsigned long long prev = atomicCAS(ctr, cur, want);
    if (prev == cur) break;
    cur = prev;
  }
  const bool last = static_cast<int>(want & 0xffffffffull) == c_last - c_first + 1;
  if (last) fence_acq_rel_gpu();   // acquire: the other CTAs' slots are read next
  return last;
}

// After this CTA wrote its piece of unit u to slot (u + cta): count the piece on
// the unit's counter; the CTA that finishes the last piece merges all pieces
// into the output. Called by the nthr threads that wrote the slot (tid in
// [0, nthr)), which synchronise on named barrier bar_id. ustart is the line
// position of the unit's first block, nb its block count, Rs its real rows, qb its first query
// row. The CTA that completes a unit clears its counter after the merge (no
// other CTA touches it again in this launch), so a replayed CUDA graph (same
// epoch every replay) starts from clear counters too.
template <int KV, int D>
__device__ inline void finish_split_piece(const DecodeArgs& a, int u, long long ustart, int nb,
                                          long long total, long long ncta, int Rs, int qb, int h,
                                          int tid, int nthr, int bar_id, volatile int* fin) {
  // The barrier orders every thread's slot writes before thread 0's release fence.
  named_bar_sync(bar_id, nthr);
  if (tid == 0) {
    int c_first, c_last;
    unit_owners(a, ustart, nb, total, ncta, &c_first, &c_last);
    // The CTA holding the unit's first block reaches this piece at the end of its
    // share and is most likely the last to arrive (every other piece counted);
    // any other CTA most likely the first (a cleared counter).
    const unsigned long long guess =
        (static_cast<int>(blockIdx.x) == c_first)
            ? ((static_cast<unsigned long long>(a.epoch) << 32) | static_cast<unsigned long long>(c_last - c_first))
            : 0ull;
    const bool last = count_published_piece(a, u, guess, c_first, c_last);
    fin[0] = last ? 1 : 0;
    fin[1] = c_first;
    fin[2] = c_last;
    PKV_TL(a, kTlCounted);
  }
  named_bar_sync(bar_id, nthr);
  if (!fin[0]) return;
  merge_split_pieces<KV, D>(a, u, fin[1], fin[2], nullptr, 0, nullptr, Rs, qb, h, tid, nthr);
  if (tid == 0) {
    a.piece_counts[u] = 0ull;
    PKV_TL(a, kTlMerged);
  }
}

// The same for a piece whose merged partial is still in shared memory (o at
// own_o[r * own_stride + d], m and l at own_ml[r], own_ml[rows + r]). The CTA
// holding the unit's first block usually finishes the unit: it first tries to
// count its piece as the completing one without publishing it; when that
// succeeds it merges from its own shared memory and the other CTAs' slots, so
// neither its slot write nor the fence that publishes it is on its critical
// path. Otherwise (or on any other CTA) the piece is written to its slot and
// counted as in finish_split_piece. cur_slot is 8 bytes of shared memory.
template <int KV, int D>
__device__ inline void finish_split_piece_smem(const DecodeArgs& a, int u, long long ustart, int nb,
                                               long long total, long long ncta, int Rs, int qb, int h,
                                               int tid, int nthr, int bar_id, volatile int* fin,
                                               volatile unsigned long long* cur_slot, const float* own_o,
                                               int own_stride, const float* own_ml) {
  const int R = a.rows;
  const int cta = static_cast<int>(blockIdx.x);
  named_bar_sync(bar_id, nthr);   // the piece's merged partial is complete in shared memory
  if (tid == 0) {
    int c_first, c_last;
    unit_owners(a, ustart, nb, total, ncta, &c_first, &c_last);
    int state = 0;                 // 0: publish, then count; 1: counted as the completing piece
    unsigned long long cur = 0ull;
    if (cta == c_first) {
      unsigned long long* ctr = a.piece_counts + u;
      const unsigned long long all_others =
          (static_cast<unsigned long long>(a.epoch) << 32) | static_cast<unsigned long long>(c_last - c_first);
      const unsigned long long prev = atomicCAS(ctr, all_others, all_others + 1ull);
      if (prev == all_others) {
        state = 1;
        fence_acq_rel_gpu();       // acquire: the other CTAs' slots are read next
        PKV_TL(a, kTlCounted);
      } else {
        cur = prev;                // counted nothing: publish, then count from this value
      }
    }
    fin[0] = state;
    fin[1] = c_first;
    fin[2] = c_last;
    *cur_slot = cur;
  }
  named_bar_sync(bar_id, nthr);
  const int c_first = fin[1], c_last = fin[2];
  if (fin[0] == 0) {
    float* P = a.partials + static_cast<size_t>(u + cta) * a.slot_floats;
    const int ooff = partial_o_offset(R);
#pragma unroll 1
    for (int idx = tid; idx < Rs * (D / 4); idx += nthr) {
      const int r = idx / (D / 4), d4 = idx - (idx / (D / 4)) * (D / 4);
      if (d4 == 0) {
        P[r] = own_ml[r];
        P[R + r] = own_ml[R + r];
      }
      *reinterpret_cast<float4*>(P + ooff + r * D + d4 * 4) =
          *reinterpret_cast<const float4*>(own_o + r * own_stride + d4 * 4);
    }
    named_bar_sync(bar_id, nthr);  // every slot write before thread 0's release fence
    if (tid == 0) {
      const bool last = count_published_piece(a, u, *cur_slot, c_first, c_last);
      fin[0] = last ? 2 : 3;
      PKV_TL(a, kTlCounted);
    }
    named_bar_sync(bar_id, nthr);
    if (fin[0] == 3) return;
  }
  merge_split_pieces<KV, D>(a, u, c_first, c_last, fin[0] == 1 ? own_o : nullptr, own_stride, own_ml, Rs, qb,
                            h, tid, nthr);
  if (tid == 0) {
    a.piece_counts[u] = 0ull;
    PKV_TL(a, kTlMerged);
  }
}

}  // namespace pkv
