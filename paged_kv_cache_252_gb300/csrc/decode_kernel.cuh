// Paged decode attention for sm_103a: one persistent wave of CTAs splits the
// whole batch's work evenly (a line over (sequence, KV head, block), each unit
// weighted with its fixed per-piece work), each CTA streaming its share through
// a TMA-fed shared-memory ring.
//
// What it computes follows "AI大模型推理速度翻倍，Colossal-Inference开源发布"
// (分页注意力算法 PagedAttention: decode attention over KV blocks reached through
// a block table; KV缓存量化 KVCache Quant: the E5M2 cache is cast back to fp16
// on read), "AI 大模型推理优化技术详解" (2.2.1 Flash Attention: softmax reduced
// block by block with a running max and sum; 2.2.2 GQA: one KV head serves a
// group of query heads) and the speculative-decoding sections (several query
// tokens per sequence, causal among themselves).
//
// Structure of one CTA
//   warp NC (the last) : producer. Walks the CTA's block range, reads physical
//                        block ids from the block table and issues the TMA copies
//                        of the K tile and the V tile of each block.
//   warps 0..NC-1      : consumers, a WR x WB grid. Row-group wr owns 8*NTW of
//                        the unit's G*n query rows; block-stream wb takes every
//                        WB-th block. Per block: S^T = K Q^T and O^T += V^T P^T on
//                        tensor cores (mma.sync m16n8k16, fp32 accumulate), online
//                        softmax in base 2 with quad shuffles. E5M2 tiles are
//                        widened to fp16 in registers (byte << 8 is exact);
//                        INT8 tiles (offset-binary bytes u = code + 128) to
//                        code + 1152 (0x64 | u, one byte permute), the bias
//                        taken off once per row after the MMAs, with each token's
//                        K scale applied to its scores and its V scale folded into P.
//   Block i of the CTA goes to ring stage i mod STAGES and to block-stream
//   i mod WB; STAGES is a multiple of WB, so each stage has a single consumer
//   stream and every wait on its mbarrier is for the next phase in order.
//   At the end of each (sequence, KV head) piece the block streams are merged in
//   shared memory; a piece covering a whole unit writes the normalised output,
//   a partial piece writes (m, l, o) to its workspace slot and counts itself on
//   the unit's counter; the CTA that finishes the unit's last piece combines all
//   pieces (M = max m, L = sum l 2^(m-M), out = sum o 2^(m-M) / L) and writes
//   the output, so no separate reduce launch is needed.
//
// Tile layout in shared memory: a (block, head) tile is [16 tokens][row bytes]
// (split into two [16][128-byte] halves when a row is 256 bytes) with the
// 128-byte (or 64-byte) TMA swizzle applied, so ldmatrix reads of 8 token rows
// hit 8 different bank groups.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "decode_common.cuh"
#include "pkv_internal.h"
#include "pkv_ptx.cuh"
#include "pkv_timeline.cuh"

namespace pkv {

// Unswizzled byte offset of 16-byte chunk `ch` of token `tok` inside a tile.
// 256-byte token rows (16-bit elements, head size 128) arrive as two TMA boxes
// of [16 tokens][128 bytes], one per half row, so that 8 consecutive tokens fall
// on 8 consecutive 128-byte lines and the swizzle spreads them over all banks.
template <int RB>
__device__ __forceinline__ uint32_t tile_off(int tok, int ch) {
  if constexpr (RB == 256) {
    return static_cast<uint32_t>((ch >> 3) * (kBlockSize * 128) + tok * 128 + (ch & 7) * 16);
  } else {
    return static_cast<uint32_t>(tok * RB + ch * 16);
  }
}

template <int RB>
__device__ __forceinline__ uint32_t swz(uint32_t off) {
  if constexpr (RB >= 128) {
    return off ^ ((off >> 3) & 0x70u);   // 16-byte chunk ^= 128-byte line index (mod 8)
  } else {
    return off ^ ((off >> 3) & 0x30u);   // 64-byte swizzle
  }
}

// Two bytes of a tile register as an fp16 pair: E5M2 (the byte is the fp16
// pattern's top byte) or INT8 (the byte is the offset-binary code u = code + 128,
// and 0x64 | u is the fp16 value 1024 + u = code + kI8Bias). sel_e5m2 places the
// two chosen bytes as fp16 high bytes; sel_i8 picks the same two. The INT8 bias
// is not taken off element by element: q . (c + bias) and sum_t P_t (c_t + bias)
// are corrected once per row by bias * sum(q) and bias * sum_t P_t.
constexpr float kI8Bias = 1152.f;
template <int KV>
__device__ __forceinline__ uint32_t widen_pair(uint32_t r, uint32_t sel_e5m2, uint32_t sel_i8) {
  if constexpr (KV == kKvInt8) {
    return __byte_perm(r, 0x64646464u, sel_i8);
  } else {
    return __byte_perm(r, 0, sel_e5m2);
  }
}

template <int KV>
__device__ __forceinline__ void mma_kv(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                       uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (KV == kKvBf16) {
    mma_bf16(d, a0, a1, a2, a3, b0, b1);
  } else {
    mma_f16(d, a0, a1, a2, a3, b0, b1);
  }
}

// The decode CTA's work (inlined into the kernels below; tm_* and a are their
// grid-constant parameters).
template <int KV, int D, int NTW>
__device__ __forceinline__ void decode_body(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                            const CUtensorMap& tm_k1, const CUtensorMap& tm_v1,
                                            const DecodeArgs& a) {
  constexpr int RB = tile_row_bytes(KV, D);   // bytes of one token row of a tile
  constexpr int TILE = tile_bytes(KV, D);     // bytes of one (block, head) tile
  constexpr int KS = D / 16;                  // k-steps of S^T = K Q^T
  constexpr int MT = D / 16;                  // m-tiles of O^T = V^T P^T
  constexpr bool kFp8 = (KV == kKvE5m2 || KV == kKvInt8);   // one byte per element
  constexpr bool kInt8 = (KV == kKvInt8);
  constexpr int QS = D * 2 + 16;              // query row stride in shared memory (bytes)
  constexpr float kNegInf = -INFINITY;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int WR = a.warps_rows, WB = a.warps_blocks, NC = WR * WB, stages = a.stages;
  const int R = a.rows, R_pad = 8 * NTW * WR;
  const DecodeSmem lay = decode_smem_layout(KV, D, NTW, WR, WB, stages, R);
  const uint32_t ring = smem_addr(smem + lay.ring);
  const uint32_t bars = smem_addr(smem + lay.bars);   // full[k]: +8k, empty[k]: +8(stages+k)
  uint8_t* qs = smem + lay.qs;
  float* mrg_o = reinterpret_cast<float*>(smem + lay.mrg_o);
  float* mrg_m = reinterpret_cast<float*>(smem + lay.mrg_ml);
  float* mrg_l = mrg_m + WB * R;
  long long* red = reinterpret_cast<long long*>(smem + lay.misc);   // [10] block-reduce scratch
  long long* plan = red + 10;                                      // total, b0, b1, s0, cum0
  volatile int* abort_flag = reinterpret_cast<volatile int*>(plan + 5);
  volatile int* fin = reinterpret_cast<volatile int*>(plan + 6);   // split-finish state, first CTA, last CTA
  volatile unsigned long long* fin_cur = reinterpret_cast<volatile unsigned long long*>(plan + 8);
  float* fin_ml = reinterpret_cast<float*>(smem + lay.fin_ml);     // a split piece's merged m[R], l[R]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool is_producer = (warp == NC);
  if (tid == 0) PKV_TL(a, kTlStart);

  if (tid == 0) {
    for (int k = 0; k < stages; ++k) {
      mbar_init(bars + 8 * k, 1);
      mbar_init(bars + 8 * (stages + k), WR);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (is_producer && lane == 0) {
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    if constexpr (RB == 256) {
      prefetch_tensormap(&tm_k1);
      prefetch_tensormap(&tm_v1);
    }
  }
  // Padding rows of the query tile stay zero for the whole kernel.
  for (int idx = tid; idx < (R_pad - R) * (QS / 16); idx += blockDim.x) {
    reinterpret_cast<uint4*>(qs + R * QS)[idx] = make_uint4(0, 0, 0, 0);
  }

  prefetch_plan_inputs(a.context_lens, a.block_tables, a.num_seqs, a.max_blocks_per_seq);
  // Everything below reads inputs a previous kernel in the stream may write.
  pdl_wait_prior_grid();

  const int Hkv = a.num_kv_heads, mbs = a.max_blocks_per_seq;
  const int n = a.q_per_seq, G = a.group, Hq = a.num_q_heads;
  const long long ncta = gridDim.x, cta = blockIdx.x;

  plan_cta_share(a, red, plan);
  pdl_launch_dependents();
  if (tid == 0) PKV_TL(a, kTlPlanned);

  const long long total = plan[0], b0 = plan[1], b1 = plan[2];
  if (b0 >= b1 || plan[3] < 0) return;

  // Walk state, identical in every warp: current unit (s, h), its first block's
  // position ub on the work line, and the first block lb this CTA takes in it.
  const int pc0 = a.piece_cost;
  int s = static_cast<int>(plan[3]);
  int ctx = a.context_lens[s];
  int nb = unit_blocks(ctx, mbs);
  int h, lb;
  long long ub;
  {
    const long long off = b0 - (long long)Hkv * plan[4];
    h = static_cast<int>(off / (nb + pc0));
    const int o = static_cast<int>(off % (nb + pc0));
    lb = o > pc0 ? o - pc0 : 0;
    ub = b0 - o + pc0;
  }

  if (is_producer) {
    // ------------------------------- producer ------------------------------------
    const uint64_t pol = l2_policy_evict_first();
    const int total_rows = a.num_blocks * Hkv * kBlockSize;   // host guarantees < 2^31
    int i = 0;
    int pst = 0;           // i % stages
    uint32_t pwrap = 0;    // (i / stages) & 1
    bool ok = true;
#ifdef PKV_TIMELINE
    long long tl_pwait = 0;
    const long long tl_p0 = clock64();
#endif
    while (ub < b1 && ok) {
      const int take = static_cast<int>(min(static_cast<long long>(nb), b1 - ub)) - lb;
      const int32_t* bt = a.block_tables + static_cast<size_t>(s) * mbs + lb;
      int nxt = (lane < take) ? bt[lane] : 0;
      for (int k0 = 0; k0 < take && ok; k0 += 32) {
        const int cur = nxt;
        const int cnt = min(32, take - k0);
        if (k0 + 32 < take) nxt = (k0 + 32 + lane < take) ? bt[k0 + 32 + lane] : 0;
        for (int k = 0; k < cnt; ++k, ++i) {
          const int blk = __shfl_sync(0xffffffffu, cur, k);
          int good = ok ? 1 : 0;
          if (lane == 0 && good) {
            const int stage = pst;
#ifdef PKV_TIMELINE
            const long long tl_w0 = clock64();
            const bool got = i < stages || wait_or_abort(bars + 8 * (stages + stage), pwrap ^ 1u, abort_flag);
            tl_pwait += clock64() - tl_w0;
            if (!got) {
#else
            if (i >= stages && !wait_or_abort(bars + 8 * (stages + stage), pwrap ^ 1u, abort_flag)) {
#endif
              good = 0;
              *abort_flag = 1;
              if (a.status) atomicOr(a.status, kDevTimeout);
            } else {
              const bool bad = static_cast<unsigned>(blk) >= static_cast<unsigned>(a.num_blocks);
              if (bad && a.status) atomicOr(a.status, kDevBadBlock);
              // A bad block id reads a box wholly past the end: TMA fills it with zeros.
              const int row = bad ? total_rows : (blk * Hkv + h) * kBlockSize;
              const uint32_t full = bars + 8 * stage;
              const uint32_t kdst = ring + stage * 2 * TILE;
              mbar_arrive_expect_tx(full, 2 * TILE + ((kInt8 && !bad) ? 128 : 0));
              if constexpr (kInt8) {
                // The block's 16 K and 16 V row scales, adjacent in memory: one
                // 128-byte copy (a bad block id reads none).
                if (!bad) {
                  const size_t stile = static_cast<size_t>(blk) * Hkv + h;
                  bulk_load(smem_addr(smem + lay.scales + stage * 128), a.scales + stile * 32, 128, full);
                }
              }
              if constexpr (RB == 256) {
                // Two 2-D maps per cache, one per 128-byte half of a token row.
                tma_load_2d(kdst, &tm_k, 0, row, full, pol);
                tma_load_2d(kdst + TILE / 2, &tm_k1, 0, row, full, pol);
                tma_load_2d(kdst + TILE, &tm_v, 0, row, full, pol);
                tma_load_2d(kdst + TILE + TILE / 2, &tm_v1, 0, row, full, pol);
              } else {
                tma_load_2d(kdst, &tm_k, 0, row, full, pol);
                tma_load_2d(kdst + TILE, &tm_v, 0, row, full, pol);
              }
              if (i == 0) PKV_TL(a, kTlFirstIssue);
            }
          }
          ok = __shfl_sync(0xffffffffu, good, 0) != 0;
          if (!ok) break;   // block i was not issued
          if (++pst == stages) {
            pst = 0;
            pwrap ^= 1u;
          }
        }
      }
      // Next unit (a piece that stops before the unit's end ended the share).
      if (lb + take < nb) break;
      ub += nb + pc0;
      lb = 0;
      if (++h == Hkv) {
        h = 0;
        ++s;
        if (ub < b1) {
          ctx = a.context_lens[s];
          nb = unit_blocks(ctx, mbs);
        }
      }
    }
    if (lane == 0) PKV_TL(a, kTlLastIssue);
#ifdef PKV_TIMELINE
    if (lane == 0) {
      PKV_TL_SET(a, kTlProdWait, tl_pwait);
      PKV_TL_SET(a, kTlProdTotal, clock64() - tl_p0);
    }
#endif
    // Drain: every copy issued into this CTA's shared memory lands before exit.
    if (lane == 0) {
      for (int k = (i > stages ? i - stages : 0); k < i; ++k) {
        mbar_wait(bars + 8 * (k % stages), (k / stages) & 1);
      }
    }
    return;
  }

  // --------------------------------- consumers -------------------------------------
  const int wr = warp % WR, wb = warp / WR;
  const int g8 = lane >> 2, c4 = lane & 3;
  const int nthr_c = NC * 32;
  const int row_base = wr * 8 * NTW;
  bool alive = true;
  int i = 0;
  // This block-stream takes the blocks ib = wb, wb + WB, ... of the share in order;
  // their ring stage and phase advance by WB blocks at a time (stages is a multiple of WB).
  int cst = wb;          // ib % stages of the stream's next block
  uint32_t cph = 0;      // (ib / stages) & 1
#ifdef PKV_TIMELINE
  unsigned long long tl_blocks = 0, tl_pieces = 0;
  // Consumer thread 0's cycles per phase, summed over pieces (timeline.py MMA_STEPS).
  PKV_TL_STEP_BEGIN;
#endif

  while (ub < b1) {
    if (tid == 0) PKV_TL_STEP(7);
    const int take = static_cast<int>(min(static_cast<long long>(nb), b1 - ub)) - lb;
    const bool first = (lb == 0), last = (lb + take == nb);
    const bool split = !(first && last);
    const int u = s * Hkv + h;
    const int cap = mbs * kBlockSize;
    const int ctx_eff = ctx < cap ? ctx : cap;
    // Query tokens of sequence s: n_s of them, rows qb.. of q/out ("nopadding"
    // packed tokens). With cu_q_lens a sequence may carry fewer than q_per_seq;
    // a count outside [1, q_per_seq], or rows past the end of q, is flagged and
    // the sequence gets no rows.
    int n_s = n, qb = s * n;
    if (a.cu_q_lens) {
      qb = a.cu_q_lens[s];
      n_s = a.cu_q_lens[s + 1] - qb;
    }
    // The sequence's rows must also lie inside q / out (a.q_rows rows).
    const bool rows_ok = n_s >= 1 && n_s <= n && qb >= 0 && qb <= a.q_rows - n_s;
    const int Rs = rows_ok ? G * n_s : 0;          // real rows of this unit
    if (!rows_ok) {
      n_s = 1;
      qb = 0;
    }
    if (first && warp == 0 && lane == 0 && (!rows_ok || ctx < n_s || ctx > cap) && a.status) {
      atomicOr(a.status, kDevBadCtx);
    }

    // Query rows of this unit -> shared memory. Row r = j*G + gi is query token j,
    // query head h*G + gi. Rows past Rs keep stale finite values; every row is an
    // independent column of S and O, and only rows below Rs are written out.
    for (int idx = tid; idx < Rs * (D / 8); idx += nthr_c) {
      const int r = idx / (D / 8), ch = idx % (D / 8);
      const int j = r / G, gi = r - j * G;
      const size_t src = (static_cast<size_t>(qb + j) * Hq + h * G + gi) * D + ch * 8;
      *reinterpret_cast<uint4*>(qs + r * QS + ch * 16) =
          *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) + src);
    }
    named_bar_sync(1, nthr_c);
    if (tid == 0) PKV_TL_STEP(0);

    // B fragments of Q^T for this warp's rows (held for the whole piece).
    uint32_t qf[NTW][KS][2];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) {
      const int rb = row_base + nt * 8;
      if constexpr (kFp8) {
        // k-slot permutation matching the widened E5M2 K fragments: slots
        // {2c,2c+1} <-> d = 16ks+4c+{0,1}, slots {2c+8,2c+9} <-> d = 16ks+4c+{2,3}.
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint2 v = *reinterpret_cast<const uint2*>(qs + (rb + g8) * QS + (16 * ks + 4 * c4) * 2);
          qf[nt][ks][0] = v.x;
          qf[nt][ks][1] = v.y;
        }
      } else {
#pragma unroll
        for (int kp = 0; kp < KS / 2; ++kp) {
          const uint32_t addr = smem_addr(qs) + (rb + (lane & 7)) * QS + (4 * kp + (lane >> 3)) * 16;
          ldsm_x4(addr, qf[nt][2 * kp][0], qf[nt][2 * kp][1], qf[nt][2 * kp + 1][0],
                  qf[nt][2 * kp + 1][1]);
        }
      }
    }

    // INT8: kI8Bias * sum_d q[r][d] for this lane's rows (the 8 lanes of a row
    // group each add D/8 dimensions). The output's bias, kI8Bias times the running
    // sum of the (V-scaled) P values the P V product uses, accumulates on the tensor
    // core (o_bias: the P V product with every V element replaced by kI8Bias).
    float kq[NTW][2];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        kq[nt][e] = 0.f;
        if constexpr (kInt8) {
          const uint8_t* qr = qs + (row_base + nt * 8 + 2 * c4 + e) * QS + g8 * (D / 4);
          float acc = 0.f;
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(qr + 16 * c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
              acc += f.x + f.y;
            }
          }
          acc += __shfl_xor_sync(0xffffffffu, acc, 4);
          acc += __shfl_xor_sync(0xffffffffu, acc, 8);
          acc += __shfl_xor_sync(0xffffffffu, acc, 16);
          kq[nt][e] = kI8Bias * acc;
        }
      }

    float m_run[NTW][2], l_run[NTW][2];
    float o_acc[MT][NTW][4];
    float o_bias[kInt8 ? NTW : 1][4];   // INT8: kI8Bias * sum of P per row (rows 2c4, 2c4+1, 2c4, 2c4+1)
    // Visibility of the n_s query (draft) tokens: the context before them,
    // positions < cb, is visible to every row; draft token i (position cb + i) is
    // visible to query token j when bit i of j's mask is set. Without tree masks
    // the mask is the causal chain, bits 0..j.
    const int cb = ctx_eff - n_s;
    unsigned long long vis[NTW][2];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        m_run[nt][e] = kNegInf;
        l_run[nt][e] = 0.f;
        const int r = row_base + nt * 8 + 2 * c4 + e;
        const int j = r / G;
        if (a.tree_masks && r < Rs) {
          vis[nt][e] = a.tree_masks[qb + j];
        } else {
          vis[nt][e] = (j >= 63) ? ~0ull : ((2ull << j) - 1ull);
        }
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        o_acc[mt][nt][0] = o_acc[mt][nt][1] = o_acc[mt][nt][2] = o_acc[mt][nt][3] = 0.f;
      }
      if constexpr (kInt8) o_bias[nt][0] = o_bias[nt][1] = o_bias[nt][2] = o_bias[nt][3] = 0.f;
    }

    if (tid == 0) PKV_TL_STEP(1);
    const int k_first = ((wb - (i % WB)) % WB + WB) % WB;
    for (int k = k_first; k < take; k += WB) {
      const int stage = cst;
      const uint32_t parity = cph;
      cst += WB;
      if (cst >= stages) {
        cst -= stages;
        cph ^= 1u;
      }
      const uint32_t kt = ring + stage * 2 * TILE, vt = kt + TILE;
      if (alive && !wait_or_abort(bars + 8 * stage, parity, abort_flag)) {
        alive = false;
        *abort_flag = 1;
        if (lane == 0 && a.status) atomicOr(a.status, kDevTimeout);
      }
      if (tid == 0) PKV_TL_STEP(2);
#ifdef PKV_TIMELINE
      if (tid == 0 && tl_blocks == 0) PKV_TL(a, kTlFirstData);
      tl_blocks += (tid == 0);
#endif
      // A warp whose rows are all padding for this sequence (fewer query tokens
      // than the unit's row capacity) only waits for and releases its stages.
      if (alive && row_base < Rs) {
        const int tok0 = (lb + k) * kBlockSize;
        if (tok0 + kBlockSize > ctx_eff) {
          // Positions >= ctx are not part of the sequence; their V rows may hold
          // anything (even NaN), so zero them before P V (their weight is 0).
          const int tv = ctx_eff - tok0 > 0 ? ctx_eff - tok0 : 0;
          uint8_t* vt_ptr = smem + lay.ring + stage * 2 * TILE + TILE;
          for (int idx = lane; idx < (kBlockSize - tv) * (RB / 16); idx += 32) {
            const int t = tv + idx / (RB / 16), ch = idx % (RB / 16);
            *reinterpret_cast<uint4*>(vt_ptr + tile_off<RB>(t, ch)) = make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
          fence_proxy_async_smem();
        }

        // INT8: this lane's K and V row scales (tokens g8 and g8+8 of the block),
        // loaded before the S^T MMAs so that their latency overlaps them.
        float sc_k_lo = 0.f, sc_k_hi = 0.f, sc_v_lo = 0.f, sc_v_hi = 0.f;
        if constexpr (kInt8) {
          const uint32_t sca = smem_addr(smem + lay.scales + stage * 128) + 4 * g8;
          sc_k_lo = lds_f32_early(sca);
          sc_k_hi = lds_f32_early(sca + 32);
          sc_v_lo = lds_f32_early(sca + 64);
          sc_v_hi = lds_f32_early(sca + 96);
        }

        // ---- S^T (16 tokens x 8*NTW rows) = K Q^T, two independent chains ----
        // (INT8: the first chain starts from -kq, which takes the K bias off the scores.)
        float sa[2][NTW][4];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
          sa[0][nt][0] = sa[0][nt][2] = -kq[nt][0];
          sa[0][nt][1] = sa[0][nt][3] = -kq[nt][1];
          sa[1][nt][0] = sa[1][nt][1] = sa[1][nt][2] = sa[1][nt][3] = 0.f;
        }
        {
          const int mi = lane >> 3;
          const int tok = (lane & 7) + 8 * (mi & 1);
          if constexpr (!kFp8) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
              const int ch = 2 * ks + (mi >> 1);
              uint32_t a0, a1, a2, a3;
              ldsm_x4(kt + swz<RB>(tile_off<RB>(tok, ch)), a0, a1, a2, a3);
#pragma unroll
              for (int nt = 0; nt < NTW; ++nt)
                mma_kv<KV>(sa[ks & 1][nt], a0, a1, a2, a3, qf[nt][ks][0], qf[nt][ks][1]);
            }
          } else {
#pragma unroll
            for (int kp = 0; kp < KS / 2; ++kp) {
              const int ch = 2 * kp + (mi >> 1);
              uint32_t r0, r1, r2, r3;
              ldsm_x4(kt + swz<RB>(tile_off<RB>(tok, ch)), r0, r1, r2, r3);
              // Widen bytes (0,1) and (2,3) of each register to fp16 pairs.
              const uint32_t k0 = widen_pair<KV>(r0, 0x1404, 0x4140), k2 = widen_pair<KV>(r0, 0x3424, 0x4342);
              const uint32_t k1 = widen_pair<KV>(r1, 0x1404, 0x4140), k3 = widen_pair<KV>(r1, 0x3424, 0x4342);
              const uint32_t k4 = widen_pair<KV>(r2, 0x1404, 0x4140), k6 = widen_pair<KV>(r2, 0x3424, 0x4342);
              const uint32_t k5 = widen_pair<KV>(r3, 0x1404, 0x4140), k7 = widen_pair<KV>(r3, 0x3424, 0x4342);
#pragma unroll
              for (int nt = 0; nt < NTW; ++nt) {
                mma_f16(sa[0][nt], k0, k1, k2, k3, qf[nt][2 * kp][0], qf[nt][2 * kp][1]);
                mma_f16(sa[1][nt], k4, k5, k6, k7, qf[nt][2 * kp + 1][0], qf[nt][2 * kp + 1][1]);
              }
            }
          }
        }

        // ---- online softmax (base 2) over this block ----
        const bool masked = tok0 + (kBlockSize - 1) >= cb;
        const int p_lo = tok0 + g8, p_hi = p_lo + 8;
        // INT8: this lane's tokens g8 and g8+8 of the block. Their K scales
        // scale the scores; their V scales are folded into P (0 past the context,
        // where the stage may hold stale scales). The scales are fp16 values, so a
        // token whose P is 1 (the row's maximum) enters the P V product with exactly
        // its scale; the rounding of P * sv to fp16 otherwise perturbs a weight by
        // at most 2^-11, as the rounding of P does in the other paths.
        float sk_lo = a.scale_log2, sk_hi = a.scale_log2, sv_lo = 1.f, sv_hi = 1.f;
        if constexpr (kInt8) {
          sk_lo *= sc_k_lo;
          sk_hi *= sc_k_hi;
          sv_lo = p_lo < ctx_eff ? sc_v_lo : 0.f;
          sv_hi = p_hi < ctx_eff ? sc_v_hi : 0.f;
        }
        uint32_t pb[NTW][2];
        uint32_t pb_lo[NTW][2];   // bf16 only: P - bf16(P), a second bf16 term
        float alpha[NTW][2];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
          float pv[4];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float x_lo = (sa[0][nt][e] + sa[1][nt][e]) * sk_lo;
            float x_hi = (sa[0][nt][2 + e] + sa[1][nt][2 + e]) * sk_hi;
            if (masked) {
              const bool v_lo = p_lo < cb || (p_lo < ctx_eff && p_lo - cb < 64 &&
                                               ((vis[nt][e] >> (p_lo - cb)) & 1ull));
              const bool v_hi = p_hi < cb || (p_hi < ctx_eff && p_hi - cb < 64 &&
                                               ((vis[nt][e] >> (p_hi - cb)) & 1ull));
              x_lo = v_lo ? x_lo : kNegInf;
              x_hi = v_hi ? x_hi : kNegInf;
            }
            float mx = fmaxf(x_lo, x_hi);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m_run[nt][e], mx);
            const float m_use = (m_new == kNegInf) ? 0.f : m_new;
            alpha[nt][e] = fast_exp2(m_run[nt][e] - m_use);
            pv[e] = fast_exp2(x_lo - m_use);
            pv[2 + e] = fast_exp2(x_hi - m_use);
            l_run[nt][e] = l_run[nt][e] * alpha[nt][e] + pv[e] + pv[2 + e];
            m_run[nt][e] = m_new;
          }
          // P^T fragments: the S^T accumulator layout (token g, rows 2c..2c+1) is an
          // 8x8 b16 tile per 8 tokens; transposing it gives (row g, tokens 2c..2c+1),
          // which is exactly the B operand of O^T += V^T P^T.
          const uint32_t h01 = pack_p<KV>(pv[0] * sv_lo, pv[1] * sv_lo);
          const uint32_t h23 = pack_p<KV>(pv[2] * sv_hi, pv[3] * sv_hi);
          pb[nt][0] = movmatrix_t(h01);
          pb[nt][1] = movmatrix_t(h23);
          if constexpr (KV == kKvBf16) {
            // bf16 keeps 8 significant bits; P = hi + lo with both in bf16 keeps
            // about 16, so the P V product is as accurate as with an fp16 P.
            const uint32_t l01 = pack_bf16x2(pv[0] - __uint_as_float(h01 << 16),
                                             pv[1] - __uint_as_float(h01 & 0xFFFF0000u));
            const uint32_t l23 = pack_bf16x2(pv[2] - __uint_as_float(h23 << 16),
                                             pv[3] - __uint_as_float(h23 & 0xFFFF0000u));
            pb_lo[nt][0] = movmatrix_t(l01);
            pb_lo[nt][1] = movmatrix_t(l23);
          }
        }
        // alpha is exactly 1 for a row whose running max did not change; once the
        // max settles that holds for the whole warp and the rescale is skipped.
        bool rescale = false;
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) rescale |= (alpha[nt][0] != 1.f) | (alpha[nt][1] != 1.f);
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) {
              o_acc[mt][nt][0] *= alpha[nt][0];
              o_acc[mt][nt][1] *= alpha[nt][1];
              o_acc[mt][nt][2] *= alpha[nt][0];
              o_acc[mt][nt][3] *= alpha[nt][1];
            }
          if constexpr (kInt8) {
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) {
              o_bias[nt][0] *= alpha[nt][0];
              o_bias[nt][1] *= alpha[nt][1];
              o_bias[nt][2] *= alpha[nt][0];
              o_bias[nt][3] *= alpha[nt][1];
            }
          }
        }

        // ---- O^T (head_size x rows) += V^T P^T ----
        {
          const int mi = lane >> 3;
          if constexpr (!kFp8) {
            const int tok = (lane & 7) + 8 * (mi >> 1);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              const int ch = 2 * mt + (mi & 1);
              uint32_t a0, a1, a2, a3;
              ldsm_x4_t(vt + swz<RB>(tile_off<RB>(tok, ch)), a0, a1, a2, a3);
#pragma unroll
              for (int nt = 0; nt < NTW; ++nt) {
                mma_kv<KV>(o_acc[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                if constexpr (KV == kKvBf16)
                  mma_kv<KV>(o_acc[mt][nt], a0, a1, a2, a3, pb_lo[nt][0], pb_lo[nt][1]);
              }
            }
          } else {
            const int tok = (lane & 7) + 8 * (mi & 1);
#pragma unroll
            for (int mp = 0; mp < MT / 2; ++mp) {
              const int ch = 2 * mp + (mi >> 1);
              uint32_t r0, r1, r2, r3;
              ldsm_x4_t(vt + swz<RB>(tile_off<RB>(tok, ch)), r0, r1, r2, r3);
              // Transposed load of byte pairs: register = {V[2c][2g], V[2c][2g+1],
              // V[2c+1][2g], V[2c+1][2g+1]}; m-row g <-> d 2g, m-row g+8 <-> d 2g+1.
              const uint32_t v0 = widen_pair<KV>(r0, 0x2404, 0x4240), v1 = widen_pair<KV>(r0, 0x3414, 0x4341);
              const uint32_t v2 = widen_pair<KV>(r1, 0x2404, 0x4240), v3 = widen_pair<KV>(r1, 0x3414, 0x4341);
              const uint32_t v4 = widen_pair<KV>(r2, 0x2404, 0x4240), v5 = widen_pair<KV>(r2, 0x3414, 0x4341);
              const uint32_t v6 = widen_pair<KV>(r3, 0x2404, 0x4240), v7 = widen_pair<KV>(r3, 0x3414, 0x4341);
#pragma unroll
              for (int nt = 0; nt < NTW; ++nt) {
                mma_f16(o_acc[2 * mp][nt], v0, v1, v2, v3, pb[nt][0], pb[nt][1]);
                mma_f16(o_acc[2 * mp + 1][nt], v4, v5, v6, v7, pb[nt][0], pb[nt][1]);
              }
            }
            if constexpr (kInt8) {
              // The bias product: every element of the A operand is kI8Bias (fp16 0x6480).
              constexpr uint32_t kBias2 = 0x64806480u;
#pragma unroll
              for (int nt = 0; nt < NTW; ++nt)
                mma_f16(o_bias[nt], kBias2, kBias2, kBias2, kBias2, pb[nt][0], pb[nt][1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8 * (stages + stage));
      if (tid == 0) PKV_TL_STEP(3);
    }
    if (tid == 0) PKV_TL(a, kTlLastData);
    i += take;
#ifdef PKV_TIMELINE
    ++tl_pieces;
#endif

    // ---- merge the WB block streams of this piece ----
    if constexpr (kInt8) {
      // Take the INT8 bias off O^T: kI8Bias * (sum over the warp's tokens of the P it used).
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o_acc[mt][nt][e] -= o_bias[nt][e];
    }
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float lsum = l_run[nt][e];
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 4);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 8);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);
        const int r = row_base + nt * 8 + 2 * c4 + e;
        if (g8 == 0 && r < R) {
          mrg_m[wb * R + r] = m_run[nt][e];
          mrg_l[wb * R + r] = lsum;
        }
      }
    {
      float* mo = mrg_o + static_cast<size_t>(wb) * R * (D + 4);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int d_lo = kFp8 ? 16 * mt + 2 * g8 : 16 * mt + g8;
        const int d_hi = kFp8 ? d_lo + 1 : d_lo + 8;
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
          const int r0 = row_base + nt * 8 + 2 * c4;
          if (r0 < R) {
            mo[r0 * (D + 4) + d_lo] = o_acc[mt][nt][0];
            mo[r0 * (D + 4) + d_hi] = o_acc[mt][nt][2];
          }
          if (r0 + 1 < R) {
            mo[(r0 + 1) * (D + 4) + d_lo] = o_acc[mt][nt][1];
            mo[(r0 + 1) * (D + 4) + d_hi] = o_acc[mt][nt][3];
          }
        }
      }
    }
    named_bar_sync(2, nthr_c);
    if (tid == 0) PKV_TL_STEP(4);
    for (int idx = tid; idx < Rs * (D / 4); idx += nthr_c) {
      const int r = idx / (D / 4), d4 = idx - (idx / (D / 4)) * (D / 4);
      float M = kNegInf;
      for (int w = 0; w < WB; ++w) M = fmaxf(M, mrg_m[w * R + r]);
      const float Mu = (M == kNegInf) ? 0.f : M;
      float lsum = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int w = 0; w < WB; ++w) {
        const float f = fast_exp2(mrg_m[w * R + r] - Mu);
        lsum += f * mrg_l[w * R + r];
        const float4 v =
            *reinterpret_cast<const float4*>(mrg_o + static_cast<size_t>(w * R + r) * (D + 4) + d4 * 4);
        acc.x += f * v.x;
        acc.y += f * v.y;
        acc.z += f * v.z;
        acc.w += f * v.w;
      }
      if (!split) {
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        const int j = r / G, gi = r - j * G;
        const size_t dst = (static_cast<size_t>(qb + j) * Hq + h * G + gi) * D + d4 * 4;
        uint2 pk;
        pk.x = pack_p<KV>(acc.x * inv, acc.y * inv);
        pk.y = pack_p<KV>(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + dst) = pk;
      } else {
        // A split piece keeps its merged partial in shared memory: o in place of
        // block-stream 0's rows (only this thread reads or writes these four
        // values), m and l beside.
        *reinterpret_cast<float4*>(mrg_o + static_cast<size_t>(r) * (D + 4) + d4 * 4) = acc;
        if (d4 == 0) {
          fin_ml[r] = M;
          fin_ml[R + r] = lsum;
        }
      }
    }

    if (tid == 0) PKV_TL(a, kTlPieceOut);
    if (tid == 0) PKV_TL_STEP(5);
    if (split) {
      finish_split_piece_smem<KV, D>(a, u, ub, nb, total, ncta, Rs, qb, h, tid, nthr_c, 3, fin, fin_cur, mrg_o,
                                     D + 4, fin_ml);
    }
    if (tid == 0) PKV_TL_STEP(6);

    // ---- advance the walk (a piece that stops before the unit's end ended the share) ----
    if (lb + take < nb) break;
    ub += nb + pc0;
    lb = 0;
    if (++h == Hkv) {
      h = 0;
      ++s;
      if (ub < b1) {
        ctx = a.context_lens[s];
        nb = unit_blocks(ctx, mbs);
      }
    }
  }
#ifdef PKV_TIMELINE
  if (tid == 0) {
    PKV_TL(a, kTlExit);
    PKV_TL_SET(a, kTlInfo, sm_id() | (tl_pieces << 16) | (tl_blocks << 32));
    PKV_TL_STEP(7);
    PKV_TL_STEP_FLUSH(a);
  }
#endif
}

template <int KV, int D, int NTW>
__global__ void __launch_bounds__(160, NTW == 1 ? 3 : 2)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_k1, const __grid_constant__ CUtensorMap tm_v1,
                  const DecodeArgs a) {
  decode_body<KV, D, NTW>(tm_k, tm_v, tm_k1, tm_v1, a);
}

// Units of at most 8 rows (one row warp, two block-stream warps and the producer:
// 96 threads) with a register budget of its own (REGS; the shared kernel above
// stays within 128 so that three 160-thread CTAs fit an SM): four such CTAs per SM
// instead of five, with fewer instructions spent working around a register limit.
template <int KV, int D, int REGS>
__global__ void __maxnreg__(REGS)
    decode_kernel_narrow(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_k1, const __grid_constant__ CUtensorMap tm_v1,
                         const DecodeArgs a) {
  decode_body<KV, D, 1>(tm_k, tm_v, tm_k1, tm_v1, a);
}

}  // namespace pkv
