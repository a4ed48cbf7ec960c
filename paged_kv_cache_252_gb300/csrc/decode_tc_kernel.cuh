// Paged decode attention on the 5th-generation tensor core (tcgen05) for wide
// units: 17..64 query rows per (sequence, KV head) -- a GQA group times several
// speculative query tokens -- over an E5M2 KV cache with head size 128.
//
// What it computes is the same as the mma.sync kernel (decode_kernel.cuh):
// PagedAttention over blocks reached through a block table, the E5M2 cache
// widened to fp16 on read ("AI大模型推理速度翻倍，Colossal-Inference开源发布",
// 分页注意力算法 and KV缓存量化), softmax reduced chunk by chunk with a running
// max and sum ("AI 大模型推理优化技术详解", 2.2.1 Flash Attention), one KV head
// serving its query-head group (2.2.2 GQA), query token j of n seeing the
// context up to its own position (or the draft tokens its tree mask allows).
// The CTA's share of the batch and the split-KV combine are shared with that
// kernel (decode_common.cuh).
//
// Work is done in chunks of 8 KV blocks (128 tokens) of one unit.
//   S^T (128 tokens x RP rows)  = K_chunk (128 x 128, fp16) . Q^T      [TMEM, fp32]
//   O^T (128 dims   x 64 rows) += V_chunk^T (128 x 128 tokens) . P^T   [TMEM, fp32]
// with RP = 32 or 64 (rows padded; padding rows of Q are zero; with RP = 32 the
// P^T rows 32..63, and O^T's columns 32..63, are never written or read). K_chunk
// is the A operand straight from tensor memory (token t in lane t); Q^T, V^T and
// P^T come from shared memory, P^T MN-major so that a thread's probabilities for
// its rows are adjacent (16-byte stores).
//
// Warp roles (320 threads, one CTA per SM):
//   warp 9      : TMA producer. Copies the chunk's K and V tiles (E5M2,
//                 [16 tokens][128 bytes], 128-byte swizzle) into a ring of
//                 chunk buffers.
//   warp 8      : one thread issues every tcgen05.mma and commits each group
//                 to an mbarrier; the warp owns the tensor-memory allocation.
//   warps 0..7  : warp w reads TMEM lane quarter q = w % 4, so its thread owns
//                 token t = 32q + lane of the chunk (TMEM lane t of S^T and of
//                 K, head dimension t of O^T) and half h = w / 4 of the unit's
//                 rows and of the head dimensions. Each chunk: widen half h of
//                 the next chunk's K row of token t to fp16 into TMEM and of its
//                 V row into the shared-memory operand layout, read its scores
//                 from TMEM, mask, exponentiate against the rows' running max,
//                 add to its partial row sums and write P^T; at the end of a
//                 unit piece reduce the sums over the CTA, read O^T from TMEM
//                 and write the output or a split partial.
// The running max of a row moves only when a score exceeds it by more than
// kRescaleSlack (base 2): then the chunk's exact row maxima are reduced across
// the softmax threads and O^T and the partial sums are rescaled. Probabilities are
// therefore at most 2^kRescaleSlack, well inside fp16. Everything that runs once
// per piece or on that rare path lives in out-of-line functions, so the per-chunk
// loop stays small enough for the instruction cache.
//
// Pipeline per chunk c (softmax warps): read S(c); widen K(c+1) (+ Q of a new
// piece) -> the MMA thread issues S(c+1) while the softmax of chunk c runs;
// wait O(c-1); write P(c) -> the MMA thread issues O(c) while V(c+1) is widened.
// P^T is single-buffered; K (TMEM), S^T (TMEM), V16 and Q double-buffered.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "decode_common.cuh"
#include "pkv_internal.h"
#include "pkv_ptx.cuh"
#include "pkv_tc.cuh"
#include "pkv_timeline.cuh"

namespace pkv {

constexpr int kTcSoftmaxThreads = 256;       // warps 0..7
constexpr int kTcMmaWarp = 8;
constexpr int kTcProducerWarp = 9;
constexpr uint32_t kTcSCols = 64;            // TMEM columns per S^T buffer (two buffers from column 0)
constexpr uint32_t kTcOCol = 128;            // first TMEM column of O^T
constexpr uint32_t kTcKCol = 256;            // first TMEM column of the K buffers (64 columns each)
constexpr float kRescaleSlack = 8.f;         // base-2 headroom before the running max moves
// Running max of a row that has seen no visible score yet. Finite, so that
// x - max stays -inf for masked scores and needs no special case; any visible
// score exceeds it by more than the slack, which moves the max first.
constexpr float kNoMax = -1.0e30f;

// Order-preserving map between floats and signed ints, for integer max reductions.
__device__ __forceinline__ int float_order_key(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : (i ^ 0x7FFFFFFF);
}
__device__ __forceinline__ float float_from_order_key(int k) {
  return __int_as_float(k >= 0 ? k : (k ^ 0x7FFFFFFF));
}

// v[lane] without dynamic register indexing.
__device__ __forceinline__ float select_lane32(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int k = 0; k < s; ++k) v[k] = up ? v[k + s] : v[k];
  }
  return v[0];
}

// Bounded mbarrier wait in which a waiting warp sleeps (takes no issue slots)
// until the phase completes; it gives up after kWaitLimitNs or once another
// warp of the CTA has given up (abort flag). A phase that is already complete
// is seen by a plain test first (the test with a suspend hint costs more); the
// rest is one out-of-line function, so the many inlined waits of the chunk loop
// stay small for the instruction cache.
constexpr uint32_t kTcSleepNs = 1000000;
static __device__ __noinline__ bool tc_wait_sleeping(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait_sleep(bar, parity, kTcSleepNs)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kTcSleepNs)) return true;
    if (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  return tc_wait_sleeping(bar, parity, abort_flag);
}

// Widen half `half` (dimensions 64*half .. 64*half+63) of token row t of an
// E5M2 chunk (128 rows x 128 bytes, 128-byte swizzle, as TMA wrote it) into the
// fp16 operand layout: two 64-dimension halves of [128 rows][128 bytes], same
// swizzle. E5M2 byte b is the fp16 pattern b << 8. Rows that are not part of
// the sequence are written as zeros.
__device__ __forceinline__ void widen_e5m2_half_row(const uint8_t* src, uint8_t* dst, int t, int half,
                                                    bool valid) {
  const int sw = t & 7;
  const uint8_t* s = src + t * 128;
  uint8_t* d = dst + half * (128 * 128) + t * 128;
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const int c = 4 * half + cc;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (valid) v = *reinterpret_cast<const uint4*>(s + ((c ^ sw) << 4));
    uint4 lo, hi;
    lo.x = __byte_perm(v.x, 0, 0x1404);
    lo.y = __byte_perm(v.x, 0, 0x3424);
    lo.z = __byte_perm(v.y, 0, 0x1404);
    lo.w = __byte_perm(v.y, 0, 0x3424);
    hi.x = __byte_perm(v.z, 0, 0x1404);
    hi.y = __byte_perm(v.z, 0, 0x3424);
    hi.z = __byte_perm(v.w, 0, 0x1404);
    hi.w = __byte_perm(v.w, 0, 0x3424);
    *reinterpret_cast<uint4*>(d + (((2 * cc) ^ sw) << 4)) = lo;
    *reinterpret_cast<uint4*>(d + (((2 * cc + 1) ^ sw) << 4)) = hi;
  }
}

// Widen half `half` (dimensions 64*half .. 64*half+63) of token row t of an
// E5M2 chunk (as TMA wrote it, see above) to fp16 pairs in tensor memory:
// column j of the K buffer = dimensions 2j, 2j+1 (the A operand layout of
// tcgen05.mma). taddr addresses this warp's lane quarter and the K buffer.
__device__ __forceinline__ void widen_e5m2_half_row_tmem(const uint8_t* src, int t, int half, bool valid,
                                                         uint32_t taddr) {
  const int sw = t & 7;
  const uint8_t* s = src + t * 128;
  uint32_t v[32];
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const int c = 4 * half + cc;
    uint4 x = make_uint4(0, 0, 0, 0);
    if (valid) x = *reinterpret_cast<const uint4*>(s + ((c ^ sw) << 4));
    v[8 * cc + 0] = __byte_perm(x.x, 0, 0x1404);
    v[8 * cc + 1] = __byte_perm(x.x, 0, 0x3424);
    v[8 * cc + 2] = __byte_perm(x.y, 0, 0x1404);
    v[8 * cc + 3] = __byte_perm(x.y, 0, 0x3424);
    v[8 * cc + 4] = __byte_perm(x.z, 0, 0x1404);
    v[8 * cc + 5] = __byte_perm(x.z, 0, 0x3424);
    v[8 * cc + 6] = __byte_perm(x.w, 0, 0x1404);
    v[8 * cc + 7] = __byte_perm(x.w, 0, 0x3424);
  }
  tmem_st32(taddr + 32 * half, v);
}

// v[k] holds this lane's value for row k (N = 16 or 32 rows); returns the sum
// over the warp's 32 lanes of row (lane % N) (halving exchange, then the halves).
template <int N>
__device__ __forceinline__ float warp_rows_sum(float (&v)[N], int lane) {
#pragma unroll
  for (int s = N / 2; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int k = 0; k < s; ++k) {
      const float send = up ? v[k] : v[k + s];
      const float keep = up ? v[k + s] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
#pragma unroll
  for (int s = N; s < 32; s <<= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], s);
  return v[0];
}

// Position in a CTA's share: the current piece (unit (s, h), blocks
// [lb, lb + take) of it) and the current chunk (blocks cofs .. cofs + 7 of the piece).
struct TcWalk {
  long long ub;     // work-line position of the unit's first block
  long long b1;     // end of the CTA's share
  int s, h, lb, nb, ctx, take, cofs;

  __device__ bool done() const { return take <= 0; }
  __device__ int nblk() const { return take - cofs < kTcChunk ? take - cofs : kTcChunk; }
  __device__ bool first() const { return cofs == 0; }
  __device__ bool last() const { return cofs + kTcChunk >= take; }
  __device__ int first_token() const { return (lb + cofs) * kBlockSize; }
  __device__ void advance(const DecodeArgs& a) {
    cofs += kTcChunk;
    if (cofs < take) return;
    cofs = 0;
    if (lb + take < nb) {   // the piece stopped before the unit's end: the share is done
      take = 0;
      return;
    }
    ub += nb + a.piece_cost;
    lb = 0;
    if (++h == a.num_kv_heads) {
      h = 0;
      ++s;
      if (ub < b1) {
        ctx = a.context_lens[s];
        nb = unit_blocks(ctx, a.max_blocks_per_seq);
      }
    }
    take = ub < b1 ? (b1 - ub < nb ? static_cast<int>(b1 - ub) : nb) : 0;
  }
};

// Per-piece facts the softmax warps need.
struct TcPiece {
  int n_s, qb, Rs, ctx_eff, cb, u;
  bool split;
};

__device__ __forceinline__ TcPiece tc_piece(const DecodeArgs& a, const TcWalk& w, int tid) {
  TcPiece p;
  const int n = a.q_per_seq;
  const int cap = a.max_blocks_per_seq * kBlockSize;
  p.ctx_eff = w.ctx < cap ? w.ctx : cap;
  // Query tokens of sequence s: n_s of them at rows qb.. of q/out; a count
  // outside [1, q_per_seq], or rows past the end of q, is flagged and the
  // sequence gets no rows.
  int n_s = n, qb = w.s * n;
  if (a.cu_q_lens) {
    qb = a.cu_q_lens[w.s];
    n_s = a.cu_q_lens[w.s + 1] - qb;
  }
  // The sequence's rows must also lie inside q / out (a.q_rows rows).
  const bool rows_ok = n_s >= 1 && n_s <= n && qb >= 0 && qb <= a.q_rows - n_s;
  p.Rs = rows_ok ? a.group * n_s : 0;
  if (!rows_ok) {
    n_s = 1;
    qb = 0;
  }
  if (w.lb == 0 && tid == 0 && (!rows_ok || w.ctx < n_s || w.ctx > cap) && a.status) {
    atomicOr(a.status, kDevBadCtx);
  }
  p.n_s = n_s;
  p.qb = qb;
  p.cb = p.ctx_eff - n_s;
  p.u = w.s * a.num_kv_heads + w.h;
  p.split = !(w.lb == 0 && w.lb + w.take == w.nb);
  return p;
}

// Start the asynchronous copy of a piece's query rows into the K-major operand
// layout [2 halves][RP rows][128 B], row r = j*G + gi (query token j, query head
// h*G + gi); rows >= Rs are zero-filled. Each of the NT threads copies
// RP*16/NT chunks of 16 bytes.
template <int RP, int NT>
__device__ __forceinline__ void tc_copy_q(const DecodeArgs& a, const TcPiece& p, int h, int t, uint8_t* qdst) {
#pragma unroll
  for (int k = 0; k < RP * 16 / NT; ++k) {
    const int idx = t + NT * k;
    const int r = idx >> 4, ch = idx & 15;
    const bool real = r < p.Rs;
    const int j = real ? r / a.group : 0, gi = real ? r - j * a.group : 0;
    const uint16_t* src = static_cast<const uint16_t*>(a.q) +
                          (static_cast<size_t>(p.qb + j) * a.num_q_heads + h * a.group + gi) * 128 + ch * 8;
    cp_async_16(smem_addr(qdst + (ch >> 3) * (RP * 128) + r * 128 + (((ch & 7) ^ (r & 7)) << 4)),
                real ? static_cast<const void*>(src) : a.q, real ? 16u : 0u);
  }
}

// Rows that see token p of a piece, as a bit mask over rows r0 .. r0+63: every
// row for positions before the draft tokens; draft token i = p - cb is seen by
// query token j when its tree mask has bit i (or, causally, j >= i). Padding
// rows (>= Rs) are kept finite and never written out. Not part of the sequence: none.
__device__ __forceinline__ unsigned long long tc_row_visibility(const DecodeArgs& a, const TcPiece& pc, int p,
                                                             bool valid, int r0) {
  if (!valid) return 0ull;
  if (p < pc.cb) return ~0ull;
  const int G = a.group;
  const int i = p - pc.cb;
  const unsigned long long pad = pc.Rs >= 64 ? 0ull : (~0ull << pc.Rs);
  unsigned long long vis;
  if (a.tree_masks) {
    const unsigned long long gm = G >= 64 ? ~0ull : ((1ull << G) - 1ull);
    unsigned long long m = 0ull;
    for (int j = 0; j < pc.n_s; ++j)
      if ((__ldg(a.tree_masks + pc.qb + j) >> i) & 1ull) m |= gm << (j * G);
    vis = m | pad;
  } else {
    const int lo = i * G;
    vis = (lo >= 64 ? 0ull : (~0ull << lo)) | pad;
  }
  return vis >> r0;
}

// Chunk maximum of row r over the four lane quarters.
__device__ __forceinline__ float tc_chunk_max(const float* red_m, int RP, int r) {
  return fmaxf(fmaxf(red_m[r], red_m[RP + r]), fmaxf(red_m[2 * RP + r], red_m[3 * RP + r]));
}

// Rare path, part 1: the chunk's exact maxima of this thread's rows over the
// 128 tokens into red_m[quarter][row], re-reading the scores from the S^T
// columns (still intact: S(c+2) is not issued before the next chunk's K).
// Runs about once per piece, so the loop stays rolled.
__device__ __forceinline__ void tc_chunk_maxima(uint32_t s_cols, unsigned long long vis, float scale_log2,
                                                float* red_m, int RP, int q, int r0, int RH, int lane) {
#pragma unroll 1
  for (int k = 0; k < RH; ++k) {
    // Every lane loads (the load is warp-collective); the mask is applied after.
    const float sk = __uint_as_float(tmem_ld1(s_cols + k));
    const float xv = ((vis >> k) & 1ull) ? sk * scale_log2 : -INFINITY;
    const int km = __reduce_max_sync(0xffffffffu, float_order_key(xv));
    if (lane == k) red_m[q * RP + r0 + k] = float_from_order_key(km);
  }
  named_bar_sync(2, kTcSoftmaxThreads);
}

// Rare path, part 2: threads r < RP move row r's running max to the larger of
// it and the chunk maximum (into the other max buffer) and record the factor
// 2^(old - new) that rescales what the row accumulated so far.
__device__ __forceinline__ void tc_new_maxima(const float* red_m, const float* mold, float* mnew, float* alpha,
                                              int RP, int tid) {
  if (tid < RP) {
    const float mo = mold[tid];
    const float mn = fmaxf(mo, tc_chunk_max(red_m, RP, tid));
    mnew[tid] = mn;
    alpha[tid] = mn > mo ? fast_exp2(mo - mn) : 1.f;
  }
  named_bar_sync(2, kTcSoftmaxThreads);
}

// Rare path, part 3: rescale this warp's columns of O^T (they hold earlier
// chunks of the piece), one TMEM column per row.
__device__ __forceinline__ void tc_rescale_o(uint32_t t_cols, const float* alpha, int r0, int RH) {
  tc_fence_after_sync();
#pragma unroll 1
  for (int k = 0; k < RH; ++k) {
    const float al = alpha[r0 + k];
    if (al != 1.f) {
      const uint32_t col = t_cols + kTcOCol + k;
      tmem_st1(col, __float_as_uint(__uint_as_float(tmem_ld1(col)) * al));
    }
  }
}

// End of a piece, once the per-quarter row sums are in red_l: threads r < RP
// turn row r's sum into 1 / L (row_inv) or, for a split piece, write its m and
// l to the partial slot.
__device__ __forceinline__ void tc_piece_rows(const DecodeArgs& a, const TcPiece& pc, int RP, int tid,
                                              const float* mcur, const float* red_l, float* row_inv,
                                              long long cta) {
  if (tid < RP) {
    const float L = (red_l[tid] + red_l[RP + tid]) + (red_l[2 * RP + tid] + red_l[3 * RP + tid]);
    row_inv[tid] = L > 0.f ? 1.f / L : 0.f;
    if (pc.split && tid < a.rows) {
      float* slot = a.partials + static_cast<size_t>(pc.u + cta) * a.slot_floats;
      slot[tid] = mcur[tid];
      slot[a.rows + tid] = L;
    }
  }
}

// O^T of this thread's rows (head dimension t), one TMEM column per row (a
// rolled loop: this runs once per piece): the normalised output, or the
// split partial's o.
__device__ __forceinline__ void tc_piece_output(const DecodeArgs& a, uint32_t t_cols, const TcPiece& pc,
                                                int h, int r0, int RH, int t, const float* row_inv,
                                                long long cta) {
  constexpr int D = 128;
  const int G = a.group, Hq = a.num_q_heads;
  tc_fence_after_sync();
  const int r_end = r0 + RH < pc.Rs ? r0 + RH : pc.Rs;
  // Four columns per TMEM load (RH and r0 are multiples of 4; r_end is the same for
  // the whole warp, so every lane takes part in every load).
  if (!pc.split) {
    int j = r0 / G, gi = r0 - j * G;
    uint16_t* dst = static_cast<uint16_t*>(a.out) + (static_cast<size_t>(pc.qb + j) * Hq + h * G + gi) * D + t;
#pragma unroll 1
    for (int r4 = r0; r4 < r_end; r4 += 4) {
      uint32_t ov[4];
      tmem_ld4(t_cols + kTcOCol + (r4 - r0), ov);
      const float4 inv = *reinterpret_cast<const float4*>(row_inv + r4);
      const float iv[4] = {inv.x, inv.y, inv.z, inv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (r4 + e < r_end) {
          *dst = __half_as_ushort(__float2half_rn(__uint_as_float(ov[e]) * iv[e]));
          // next row: next head of the group, or the first head for the next query token
          dst += (++gi == G) ? static_cast<ptrdiff_t>(Hq - G + 1) * D : D;
          if (gi == G) gi = 0;
        }
      }
    }
  } else {
    float* slot = a.partials + static_cast<size_t>(pc.u + cta) * a.slot_floats + partial_o_offset(a.rows) + t;
#pragma unroll 1
    for (int r4 = r0; r4 < r_end; r4 += 4) {
      uint32_t ov[4];
      tmem_ld4(t_cols + kTcOCol + (r4 - r0), ov);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (r4 + e < r_end) slot[(r4 + e) * D] = __uint_as_float(ov[e]);
    }
  }
}

__device__ __forceinline__ void tc_finish_split(const DecodeArgs& a, const TcPiece& pc, long long ustart, int nb,
                                             long long total, long long ncta, int h, int tid, volatile int* fin) {
  finish_split_piece<kKvE5m2, 128>(a, pc.u, ustart, nb, total, ncta, pc.Rs, pc.qb, h, tid, kTcSoftmaxThreads,
                                   3, fin);
}

__device__ __forceinline__ void tc_plan(const DecodeArgs& a, long long* red, long long* plan) {
  plan_cta_share(a, red, plan);
}

template <int RC>
__global__ void __launch_bounds__(kTcThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ DecodeArgs a) {
  constexpr int RP = 32 * RC;                         // padded rows = the MMA's N
  constexpr int RH = RP / 2;                          // rows per softmax thread
  constexpr int D = 128;
  constexpr int TILE = kBlockSize * D;                // bytes of one E5M2 (block, head) tile
  constexpr int CHUNK_BYTES = 2 * kTcChunk * TILE;    // one ring buffer: 8 K tiles, then 8 V tiles
  constexpr uint32_t kHalf = 128 * 128;               // one 64-dim half of a widened chunk
  constexpr uint32_t kWide = 2 * kHalf;               // one widened chunk
  constexpr uint32_t kRowsHalf = RP * 128;            // one 64-element half of Q
  constexpr bool kFusedMax = RC == 1;                 // x = score less the running max (see (3))
  constexpr float kNegInf = -INFINITY;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int nbuf = a.stages;
  const TcSmem lay = tc_smem_layout(RP, nbuf);
  uint8_t* v16 = smem + lay.v16;
  uint8_t* pst = smem + lay.p;
  uint8_t* qst = smem + lay.q;
  uint8_t* ring = smem + lay.ring;
  const uint32_t bars = smem_addr(smem + lay.bars);   // full[k]: +8k, empty[k]: +8(nbuf+k)
  const uint32_t bar_kready = bars + 16 * nbuf;        // K (+Q) of a chunk written (256 arrivals)
  const uint32_t bar_pvready = bar_kready + 8;         // P^T (+V16 of the next chunk) written (256 arrivals)
  const uint32_t bar_sfull = bar_kready + 16;          // S^T MMAs of a chunk complete
  const uint32_t bar_odone = bar_kready + 24;          // O^T MMAs of a chunk complete
  const uint32_t bar_final = bar_kready + 32;          // every MMA complete (teardown)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + lay.misc);
  float* red_m = reinterpret_cast<float*>(smem + lay.misc + 16);   // [4][RP] per-quarter row maxima
  float* red_l = red_m + 4 * RP;                                    // [4][RP] per-quarter row sums
  float* row_m = red_l + 4 * RP;                                    // [2][RP] running max, two buffers
  float* row_inv = row_m + 2 * RP;                                  // [RP] 1 / row sum at a piece's end
  float* row_alpha = row_inv + RP;                                  // [RP] rescale factor when the max moves
  long long* red = reinterpret_cast<long long*>(row_alpha + RP);    // [16] plan scan scratch, one per warp
  long long* plan = red + 16;                                       // total, b0, b1, s0, cum0
  volatile int* abort_flag = reinterpret_cast<volatile int*>(plan + 5);
  volatile int* fin = abort_flag + 1;                               // is_last, first CTA, last CTA

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) PKV_TL(a, kTlStart);

  if (tid == 0) {
    for (int k = 0; k < nbuf; ++k) {
      mbar_init(bars + 8 * k, 1);
      mbar_init(bars + 8 * (nbuf + k), kTcSoftmaxThreads / 32);   // one arrival per softmax warp
    }
    mbar_init(bar_kready, kTcSoftmaxThreads);
    mbar_init(bar_pvready, kTcSoftmaxThreads);
    mbar_init(bar_sfull, 1);
    mbar_init(bar_odone, 1);
    mbar_init(bar_final, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kTcMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), kTcTmemCols);
    tmem_relinquish();
  }
  if (warp == kTcProducerWarp && lane == 0) {
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }
  for (int r = tid; r < 2 * RP; r += blockDim.x) row_m[r] = kNoMax;
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  prefetch_plan_inputs(a.context_lens, a.block_tables, a.num_seqs, a.max_blocks_per_seq);
  // Everything below reads inputs a previous kernel in the stream may write.
  pdl_wait_prior_grid();
  tc_plan(a, red, plan);
  pdl_launch_dependents();
  if (tid == 0) PKV_TL(a, kTlPlanned);

  const long long total = plan[0], b0 = plan[1], b1 = plan[2];
  if (b0 < b1 && plan[3] >= 0) {
    TcWalk w0;
    {
      const int mbs = a.max_blocks_per_seq, Hkv = a.num_kv_heads, pc0 = a.piece_cost;
      w0.b1 = b1;
      w0.s = static_cast<int>(plan[3]);
      w0.ctx = a.context_lens[w0.s];
      w0.nb = unit_blocks(w0.ctx, mbs);
      const long long off = b0 - static_cast<long long>(Hkv) * plan[4];
      w0.h = static_cast<int>(off / (w0.nb + pc0));
      const int o = static_cast<int>(off % (w0.nb + pc0));
      w0.lb = o > pc0 ? o - pc0 : 0;
      w0.ub = b0 - o + pc0;
      w0.take = static_cast<int>(b1 - w0.ub < w0.nb ? b1 - w0.ub : w0.nb) - w0.lb;
      w0.cofs = 0;
    }

    if (warp == kTcProducerWarp) {
      // ------------------------------- producer ----------------------------------
      const uint64_t pol = l2_policy_evict_first();
      const int total_rows = a.num_blocks * a.num_kv_heads * kBlockSize;   // host guarantees < 2^31
#ifdef PKV_TIMELINE
      long long tl_prod_wait = 0;
      const long long tl_prod0 = clock64();
#endif
      TcWalk w = w0;
      int c = 0;
      int buf = 0;          // c % nbuf
      uint32_t wrap = 0;    // (c / nbuf) & 1
      while (!w.done()) {
        const int nbk = w.nblk();
        const int32_t* bt = a.block_tables + static_cast<size_t>(w.s) * a.max_blocks_per_seq + w.lb + w.cofs;
        const int mine = lane < nbk ? bt[lane] : 0;
        int blk[kTcChunk];
#pragma unroll
        for (int k = 0; k < kTcChunk; ++k) blk[k] = __shfl_sync(0xffffffffu, mine, k);
        int good = 1;
        if (lane == 0) {
#ifdef PKV_TIMELINE
          const long long tl_w0 = clock64();
          const bool tl_ok = c < nbuf || tc_wait(bars + 8 * (nbuf + buf), wrap ^ 1u, abort_flag);
          tl_prod_wait += clock64() - tl_w0;
          if (!tl_ok) {
            PKV_TL_TIMEOUT(a, 0x70, c);
#else
          if (c >= nbuf && !tc_wait(bars + 8 * (nbuf + buf), wrap ^ 1u, abort_flag)) {
#endif
            good = 0;
            *abort_flag = 1;
            if (a.status) atomicOr(a.status, kDevTimeout);
          } else {
            const uint32_t full = bars + 8 * buf;
            const uint32_t kdst = smem_addr(ring + buf * CHUNK_BYTES);
            mbar_arrive_expect_tx(full, nbk * 2 * TILE);
#pragma unroll
            for (int k = 0; k < kTcChunk; ++k) {
              if (k < nbk) {
                const bool bad = static_cast<unsigned>(blk[k]) >= static_cast<unsigned>(a.num_blocks);
                if (bad && a.status) atomicOr(a.status, kDevBadBlock);
                // A bad block id reads a box wholly past the end: TMA fills it with zeros.
                const int row = bad ? total_rows : (blk[k] * a.num_kv_heads + w.h) * kBlockSize;
                tma_load_2d(kdst + k * TILE, &tm_k, 0, row, full, pol);
                tma_load_2d(kdst + kTcChunk * TILE + k * TILE, &tm_v, 0, row, full, pol);
              }
            }
            if (c == 0) PKV_TL(a, kTlFirstIssue);
          }
        }
        if (__shfl_sync(0xffffffffu, good, 0) == 0) break;   // chunk c was not issued
        ++c;
        if (++buf == nbuf) {
          buf = 0;
          wrap ^= 1u;
        }
        w.advance(a);
      }
      if (lane == 0) {
        PKV_TL(a, kTlLastIssue);
#ifdef PKV_TIMELINE
        PKV_TL_SET(a, kTlProdWait, tl_prod_wait);
        PKV_TL_SET(a, kTlProdTotal, clock64() - tl_prod0);
#endif
      }
      // Drain: every copy issued into this CTA's shared memory lands before exit.
      if (lane == 0) {
        for (int k = (c > nbuf ? c - nbuf : 0); k < c; ++k) mbar_wait(bars + 8 * (k % nbuf), (k / nbuf) & 1);
      }
    } else if (warp == kTcMmaWarp) {
      // ------------------------------ MMA issue -----------------------------------
      if (lane == 0) {
        const uint32_t id_s = idesc_kind_f16(128, RP, 0, 0, 0);   // K (TMEM, K-major) x Q^T (K-major)
        const uint32_t id_o = idesc_kind_f16(128, 64, 0, 1, 1);   // V^T (MN-major) x P^T (MN-major, 64 rows)
        const uint32_t t_o = tmem + kTcOCol;
        const uint32_t v16a = smem_addr(v16), pa = smem_addr(pst), qa = smem_addr(qst);
        // Descriptors of the buffers' first atoms, built once: a later atom is the same
        // descriptor with its address field (bits 0..13, 16-byte units) advanced, and
        // every shared-memory address here stays below 2^18 bytes, so the field never carries.
        const uint64_t dq0 = smem_desc_sw128(qa, 0, 1024), dq1 = smem_desc_sw128(qa + 2 * kRowsHalf, 0, 1024);
        const uint64_t dv0 = smem_desc_sw128(v16a, kHalf, 1024), dv1 = smem_desc_sw128(v16a + kWide, kHalf, 1024);
        const uint64_t dp = smem_desc_sw128(pa, 128 * 128, 1024);
        TcWalk w = w0;
        int c = 0, piece = 0;
        bool prev = false, prev_first = false, ok = true;
#ifdef PKV_TIMELINE
        long long tl_wk = 0, tl_wpv = 0;
        const long long tl_mma0 = clock64();
#endif
        for (;;) {
          const bool cur = !w.done();
          if (cur) {
            // S^T(c) = K(c) Q^T: S and K buffer c % 2
#ifdef PKV_TIMELINE
            const long long tl_t0 = clock64();
#endif
            ok = tc_wait(bar_kready, c & 1, abort_flag);
#ifdef PKV_TIMELINE
            tl_wk += clock64() - tl_t0;
#endif
            if (!ok) {
              PKV_TL_TIMEOUT(a, 0x61, c);
              break;
            }
            tc_fence_after_sync();
            const uint64_t dqs = (piece & 1) ? dq1 : dq0;
            const uint32_t t_s = tmem + (c & 1) * kTcSCols;
            const uint32_t t_k = tmem + kTcKCol + (c & 1) * 64;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t db = dqs + (((kk >> 2) * kRowsHalf + (kk & 3) * 32) >> 4);
              tc_mma_f16_ts(t_s, t_k + kk * 8, db, id_s, kk > 0 ? 1u : 0u);
            }
            tc_commit(bar_sfull);
          }
          if (prev) {
            // O^T += V(c-1)^T P^T
#ifdef PKV_TIMELINE
            const long long tl_t1 = clock64();
#endif
            ok = tc_wait(bar_pvready, (c - 1) & 1, abort_flag);
#ifdef PKV_TIMELINE
            tl_wpv += clock64() - tl_t1;
#endif
            if (!ok) {
              PKV_TL_TIMEOUT(a, 0x63, c);
              break;
            }
            tc_fence_after_sync();
            const uint64_t dvs = ((c - 1) & 1) ? dv1 : dv0;
#pragma unroll
            for (int kk = 0; kk < kTcChunk; ++kk) {
              tc_mma_f16_ss(t_o, dvs + ((kk * 2048) >> 4), dp + ((kk * 2048) >> 4), id_o,
                            (kk > 0 || !prev_first) ? 1u : 0u);
            }
            tc_commit(bar_odone);
          }
          if (!cur) break;
          prev = true;
          prev_first = w.first();
          if (w.last()) ++piece;
          w.advance(a);
          ++c;
        }
        if (!ok) {
          *abort_flag = 1;
          if (a.status) atomicOr(a.status, kDevTimeout);
        }
#ifdef PKV_TIMELINE
        PKV_TL_SET(a, kTlMmaWaitK, tl_wk);
        PKV_TL_SET(a, kTlMmaWaitPV, tl_wpv);
        PKV_TL_SET(a, kTlMmaTotal, clock64() - tl_mma0);
#endif
        // Every MMA issued above completes before the tensor memory is released.
        tc_commit(bar_final);
        mbar_wait(bar_final, 0);
      }
      __syncwarp();
    } else {
      // ---------------------- widen / softmax / epilogue (warps 0..7) --------------
      const int q = warp & 3, hh = warp >> 2;
      const int t = 32 * q + lane;   // token of the chunk, TMEM lane of S^T and K, head dimension of O^T
      const int r0 = hh * RH;        // first of this thread's RH rows (TMEM columns)
      const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * q) << 16);
      const uint32_t t_cols = t_lane + r0;
      const long long ncta = gridDim.x, cta = blockIdx.x;
      const float scale_log2 = a.scale_log2;
      bool alive = true;
      int o_waited = -1;
      int mp = 0;   // current running-max buffer
      int c = 0;

      auto wait_bar = [&](uint32_t bar, uint32_t parity) {
        if (!alive) return;
        const bool ok = tc_wait(bar, parity, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          alive = false;
          *abort_flag = 1;
          if (lane == 0 && a.status) atomicOr(a.status, kDevTimeout);
          if (lane == 0) PKV_TL_TIMEOUT(a, 0x40 + (bar - bars) / 8, c);
        }
      };
      auto wait_o = [&](int k) {
        if (o_waited < k) {
          wait_bar(bar_odone, static_cast<uint32_t>(k & 1));
          o_waited = k;
        }
      };

      // P^T is MN-major with 64 row slots per token: token t's line (128 bytes, 8-token
      // groups 1024 bytes apart) holds rows 0..63, rows 8j..8j+7 in 16-byte chunk j ^ (t % 8).
      // This thread's RH rows r0.. are chunks r0/8 .. r0/8 + RH/8 - 1 of its line.
      uint8_t* pline = pst + (t >> 3) * 1024 + (t & 7) * 128;

      float l_run[RH];   // this thread's (token's) share of each row's sum of exponentials
#pragma unroll
      for (int k = 0; k < RH; ++k) l_run[k] = 0.f;

      TcWalk cur = w0;
      TcPiece pc = tc_piece(a, cur, tid);
      int piece = 0;
      int buf_next = 1;          // (c + 1) % nbuf (nbuf >= 2)
      uint32_t wrap_next = 0;    // ((c + 1) / nbuf) & 1

      // Prologue: chunk 0 and the first piece's queries.
      {
        tc_copy_q<RP, kTcSoftmaxThreads>(a, pc, cur.h, tid, qst);
        wait_bar(bars, 0);
        if (tid == 0) PKV_TL(a, kTlFirstData);
        const bool valid = (t >> 4) < cur.nblk() && cur.first_token() + t < pc.ctx_eff;
        if (alive) {
          widen_e5m2_half_row_tmem(ring, t, hh, valid, t_lane + kTcKCol);
          widen_e5m2_half_row(ring + kTcChunk * TILE, v16, t, hh, valid);
        }
        cp_async_wait_all();
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncwarp();
        if (alive) {
          if (lane == 0) mbar_arrive(bars + 8 * nbuf);
          mbar_arrive(bar_kready);
        }
      }

#ifdef PKV_TIMELINE
      PKV_TL_STEP_BEGIN;
#endif
      while (!cur.done()) {
        TcWalk nxt = cur;
        nxt.advance(a);
        const bool has_next = !nxt.done();
        const bool new_piece = has_next && nxt.first();
        TcPiece pn = pc;
        if (new_piece) {
          // The other query buffer was last read by S^T MMAs of an earlier piece, all complete.
          pn = tc_piece(a, nxt, tid);
          tc_copy_q<RP, kTcSoftmaxThreads>(a, pn, nxt.h, tid, qst + ((piece + 1) & 1) * 2 * kRowsHalf);
        }
        const uint8_t* ring_next = ring + buf_next * CHUNK_BYTES;
        const bool valid_next =
            has_next && (t >> 4) < nxt.nblk() && nxt.first_token() + t < pn.ctx_eff;

        // (1) scores of chunk c, rows r0 .. r0+RH-1, from S buffer c % 2
        uint32_t sv[RH];
        PKV_TL_STEP(0);
        wait_bar(bar_sfull, c & 1);
        if (alive) {
          tc_fence_after_sync();
          tmem_ld<RH>(t_cols + (c & 1) * kTcSCols, sv);
        } else {
#pragma unroll
          for (int k = 0; k < RH; ++k) sv[k] = 0u;
        }

        // (2) K of chunk c+1 into K buffer (c+1) % 2, last read by S(c-1) (complete):
        //     S(c+1) overlaps the softmax below
        PKV_TL_STEP(1);
        if (has_next) {
          wait_bar(bars + 8 * buf_next, wrap_next);
          PKV_TL_STEP(2);
          if (alive) widen_e5m2_half_row_tmem(ring_next, t, hh, valid_next, t_lane + kTcKCol + ((c + 1) & 1) * 64);
          cp_async_wait_all();
          fence_proxy_async_smem();
          tc_fence_before_sync();
          if (alive) mbar_arrive(bar_kready);
        }

        PKV_TL_STEP(3);
        // (3) scores in base 2, masked; does any exceed its row's running max by the slack?
        //     With 32 rows per unit x holds the score less the running max (one FMA
        //     each; the rare path below recomputes it from S when the max moves). With
        //     64 rows that recompute's live scores spill registers (64-row units: 109 ->
        //     119 us), so x holds the score and the max comes off at the exponential.
        const int p = cur.first_token() + t;
        const bool valid = (t >> 4) < cur.nblk() && p < pc.ctx_eff;
        const bool allvis = valid && p < pc.cb;
        const unsigned long long vis = allvis ? ~0ull : tc_row_visibility(a, pc, p, valid, r0);
        float x[RH];
        float excess = kNegInf;
        if constexpr (kFusedMax) {
          const float* mrow = row_m + mp * RP + r0;
#pragma unroll
          for (int k4 = 0; k4 < RH / 4; ++k4) {
            const float4 m4 = *reinterpret_cast<const float4*>(mrow + 4 * k4);
            x[4 * k4] = fmaf(__uint_as_float(sv[4 * k4]), scale_log2, -m4.x);
            x[4 * k4 + 1] = fmaf(__uint_as_float(sv[4 * k4 + 1]), scale_log2, -m4.y);
            x[4 * k4 + 2] = fmaf(__uint_as_float(sv[4 * k4 + 2]), scale_log2, -m4.z);
            x[4 * k4 + 3] = fmaf(__uint_as_float(sv[4 * k4 + 3]), scale_log2, -m4.w);
          }
          if (!allvis) {
#pragma unroll
            for (int k = 0; k < RH; ++k) x[k] = ((vis >> k) & 1ull) ? x[k] : kNegInf;
          }
#pragma unroll
          for (int k = 0; k < RH; ++k) excess = fmaxf(excess, x[k]);
        } else {
          if (allvis) {
#pragma unroll
            for (int k = 0; k < RH; ++k) x[k] = __uint_as_float(sv[k]) * scale_log2;
          } else {
#pragma unroll
            for (int k = 0; k < RH; ++k) x[k] = ((vis >> k) & 1ull) ? __uint_as_float(sv[k]) * scale_log2 : kNegInf;
          }
          const float* mrow = row_m + mp * RP + r0;
#pragma unroll
          for (int k4 = 0; k4 < RH / 4; ++k4) {
            const float4 m4 = *reinterpret_cast<const float4*>(mrow + 4 * k4);
            excess = fmaxf(excess, fmaxf(fmaxf(x[4 * k4] - m4.x, x[4 * k4 + 1] - m4.y),
                                         fmaxf(x[4 * k4 + 2] - m4.z, x[4 * k4 + 3] - m4.w)));
          }
        }
        const bool rare = bar_red_or(1, kTcSoftmaxThreads, excess > kRescaleSlack);
        PKV_TL_STEP(4);
        if (rare) {
          // Rare: the running maxima move to this chunk's maxima, and what the
          // rows accumulated so far is rescaled.
          if (alive) tc_chunk_maxima(t_cols + (c & 1) * kTcSCols, vis, scale_log2, red_m, RP, q, r0, RH, lane);
          else named_bar_sync(2, kTcSoftmaxThreads);
          tc_new_maxima(red_m, row_m + mp * RP, row_m + (mp ^ 1) * RP, row_alpha, RP, tid);
          mp ^= 1;
          if (!cur.first()) {
            wait_o(c - 1);   // O^T holds earlier chunks
            if (alive) tc_rescale_o(t_cols, row_alpha, r0, RH);
          }
#pragma unroll
          for (int k = 0; k < RH; ++k) l_run[k] *= row_alpha[r0 + k];
          if constexpr (kFusedMax) {
            // The scores again (S(c) is intact) against the moved maxima.
            if (alive) {
              tc_fence_after_sync();
              tmem_ld<RH>(t_cols + (c & 1) * kTcSCols, sv);
            }
            const float* mrow = row_m + mp * RP + r0;
#pragma unroll
            for (int k4 = 0; k4 < RH / 4; ++k4) {
              const float4 m4 = *reinterpret_cast<const float4*>(mrow + 4 * k4);
              x[4 * k4] = fmaf(__uint_as_float(sv[4 * k4]), scale_log2, -m4.x);
              x[4 * k4 + 1] = fmaf(__uint_as_float(sv[4 * k4 + 1]), scale_log2, -m4.y);
              x[4 * k4 + 2] = fmaf(__uint_as_float(sv[4 * k4 + 2]), scale_log2, -m4.z);
              x[4 * k4 + 3] = fmaf(__uint_as_float(sv[4 * k4 + 3]), scale_log2, -m4.w);
            }
#pragma unroll
            for (int k = 0; k < RH; ++k) x[k] = ((vis >> k) & 1ull) ? x[k] : kNegInf;
          }
        }

        PKV_TL_STEP(5);
        // (4) P^T of chunk c (MN-major, see pline); the buffer was read by O(c-1).
        if (c > 0) wait_o(c - 1);
        PKV_TL_STEP(6);
        if (alive) {
          const float* mrow = row_m + mp * RP + r0;
          uint32_t pw[4];
#pragma unroll
          for (int k4 = 0; k4 < RH / 4; ++k4) {
            float4 m4 = make_float4(0.f, 0.f, 0.f, 0.f);   // x already less the max
            if constexpr (!kFusedMax) m4 = *reinterpret_cast<const float4*>(mrow + 4 * k4);
            const __half2 p01 = __floats2half2_rn(fast_exp2(x[4 * k4] - m4.x), fast_exp2(x[4 * k4 + 1] - m4.y));
            const __half2 p23 = __floats2half2_rn(fast_exp2(x[4 * k4 + 2] - m4.z), fast_exp2(x[4 * k4 + 3] - m4.w));
            // The sums add exactly the fp16 values the P V product uses.
            l_run[4 * k4] += __low2float(p01);
            l_run[4 * k4 + 1] += __high2float(p01);
            l_run[4 * k4 + 2] += __low2float(p23);
            l_run[4 * k4 + 3] += __high2float(p23);
            pw[2 * (k4 & 1)] = *reinterpret_cast<const uint32_t*>(&p01);
            pw[2 * (k4 & 1) + 1] = *reinterpret_cast<const uint32_t*>(&p23);
            if (k4 & 1) {
              const int j = (r0 >> 3) + (k4 >> 1);
              *reinterpret_cast<uint4*>(pline + ((j ^ (t & 7)) << 4)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
            }
          }
        }

        // P(c) is written (and V(c) was widened a chunk ago): the MMA thread may issue O(c).
        fence_proxy_async_smem();
        tc_fence_before_sync();
        if (alive) mbar_arrive(bar_pvready);

        PKV_TL_STEP(7);
        // (5) V of chunk c+1 (its buffer was read by O(c-1)); release the ring buffer.
        //     These writes are ordered for the tensor core by the fence before the
        //     next chunk's arrival.
        if (has_next) {
          if (alive) widen_e5m2_half_row(ring_next + kTcChunk * TILE, v16 + ((c + 1) & 1) * kWide, t, hh, valid_next);
          __syncwarp();
          if (alive && lane == 0) mbar_arrive(bars + 8 * (nbuf + buf_next));
        }

        PKV_TL_STEP(8);
        // (6) end of a piece: normalise and write, or write the split partial.
        if (cur.last()) {
          {
            float v[RH];
#pragma unroll
            for (int k = 0; k < RH; ++k) {
              v[k] = l_run[k];
              l_run[k] = 0.f;
            }
            const float ls = warp_rows_sum<RH>(v, lane);
            if (lane < RH) red_l[q * RP + r0 + lane] = ls;
          }
          named_bar_sync(2, kTcSoftmaxThreads);
          tc_piece_rows(a, pc, RP, tid, row_m + mp * RP, red_l, row_inv, cta);
          named_bar_sync(2, kTcSoftmaxThreads);
          wait_o(c);
          if (alive) tc_piece_output(a, t_cols, pc, cur.h, r0, RH, t, row_inv, cta);
          if (tid == 0) PKV_TL(a, kTlPieceOut);
          if (pc.split) tc_finish_split(a, pc, cur.ub, cur.nb, total, ncta, cur.h, tid, fin);
          // The next piece starts from an empty running max.
          named_bar_sync(2, kTcSoftmaxThreads);
          if (tid < RP) row_m[mp * RP + tid] = kNoMax;
          named_bar_sync(2, kTcSoftmaxThreads);
        }

        if (new_piece) {
          pc = pn;
          ++piece;
        }
        if (tid == 0 && cur.last()) PKV_TL(a, kTlLastData);
        PKV_TL_STEP(9);
        cur = nxt;
        ++c;
        if (++buf_next == nbuf) {
          buf_next = 0;
          wrap_next ^= 1u;
        }
      }
#ifdef PKV_TIMELINE
      if (tid == 0) {
        PKV_TL_STEP_FLUSH(a);
        PKV_TL(a, kTlExit);
        PKV_TL_SET(a, kTlInfo, sm_id() | (static_cast<unsigned long long>(piece + 1) << 16) |
                                   (static_cast<unsigned long long>(c) * kTcChunk << 32));
      }
#endif
    }
  }

  // Teardown: every role is done with the tensor memory.
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

}  // namespace pkv
