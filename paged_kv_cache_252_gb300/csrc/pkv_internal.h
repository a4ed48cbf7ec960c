// Internal declarations shared by the library's translation units (host and
// device). Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace pkv {

constexpr int kBlockSize = 16;       // tokens per KV block
constexpr int kMaxRows = 64;         // GQA group size x query tokens handled per CTA
constexpr int kMaxCtasPerSm = 8;     // upper bound on resident decode CTAs per SM
constexpr int kKvF16 = 0, kKvBf16 = 1, kKvE5m2 = 2, kKvInt8 = 3;

// Device-status bits (mirror the public PKV_DEV_* values).
constexpr int32_t kDevBadSlot = 0x1;
constexpr int32_t kDevBadBlock = 0x2;
constexpr int32_t kDevBadCtx = 0x4;
constexpr int32_t kDevTimeout = 0x8;

// Arguments of the decode kernel (passed by value).
struct DecodeArgs {
  void* out;                   // [S*n][Hq][D] fp16/bf16
  const void* q;               // same layout
  const int32_t* block_tables; // [S][max_blocks_per_seq]
  const int32_t* context_lens; // [S]
  const int32_t* cu_q_lens;    // [S+1] query-token offsets, or null: q_per_seq tokens each
  int32_t q_rows;              // rows of q / out (and tree_masks): a sequence's rows must lie below
  const unsigned long long* tree_masks;  // [rows] draft tokens visible to each query token, or null: causal
  const float* scales;         // INT8 cache: [num_blocks][Hkv][2][16] K then V row scales, else null
  float* partials;             // split-KV partial slots
  unsigned long long* piece_counts;  // [S*Hkv]: (call epoch << 32) | pieces finished
  int32_t* status;             // optional device status word
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t q_per_seq;           // query tokens per sequence (the maximum when cu_q_lens is set)
  int32_t group;               // Hq / Hkv
  int32_t rows;                // group * q_per_seq (row capacity of one (seq, KV head) unit)
  int32_t max_blocks_per_seq;
  int32_t num_blocks;
  int32_t warps_rows;          // consumer warps splitting the rows
  int32_t warps_blocks;        // consumer warp groups splitting the blocks
  int32_t stages;              // depth of the shared-memory ring
  int32_t slot_floats;         // floats per partial slot
  float scale_log2;            // softmax scale * log2(e)
  uint32_t epoch;              // distinct for every call (tags the piece counters)
  int32_t piece_cost;          // fixed cost of a unit piece, in blocks, for the CTA shares
#ifdef PKV_TIMELINE
  unsigned long long* timeline;  // profiling build only: per-CTA event times (pkv_timeline.cuh)
  int32_t timeline_ctas;
#endif
};


// Shared-memory and launch geometry of one decode instantiation.
struct DecodeGeometry {
  int tc;             // 1: tcgen05 kernel (then rc = 32-row column groups, stages = ring buffers)
  int rc;
  int ntw;            // n-tiles (8 rows each) per consumer warp
  int warps_rows;
  int warps_blocks;
  int stages;
  int threads;
  size_t smem_bytes;
};

// Sizes derived from (kv dtype, head size).
__host__ __device__ constexpr int kv_elem_bytes(int kv) { return (kv == kKvE5m2 || kv == kKvInt8) ? 1 : 2; }
__host__ __device__ constexpr int tile_row_bytes(int kv, int d) { return d * kv_elem_bytes(kv); }
__host__ __device__ constexpr int tile_bytes(int kv, int d) { return kBlockSize * tile_row_bytes(kv, d); }

// Floats in one split-KV partial slot: m[rows], l[rows] (padded to 4), o[rows][D].
// Bytes of a decode workspace's per-unit piece counters (8 each, rounded to 256):
// the workspace starts with them, then holds the partial slots.
__host__ __device__ constexpr size_t decode_counter_bytes(long long units) {
  return static_cast<size_t>((units * 8 + 255) / 256 * 256);
}
__host__ __device__ constexpr int partial_o_offset(int rows) { return ((2 * rows + 3) / 4) * 4; }
__host__ __device__ constexpr int partial_slot_floats(int rows, int d) {
  return partial_o_offset(rows) + rows * d;
}

// Shared-memory layout of the decode kernel, relative to a 1024-aligned base.
// An INT8 cache adds, per ring stage, the 16 K and 16 V row scales (128 bytes).
struct DecodeSmem {
  size_t ring, scales, bars, qs, mrg_o, mrg_ml, fin_ml, misc, total;
};
// The merge buffers hold only the unit's real rows (rows <= 8*ntw*wr).
__host__ __device__ inline DecodeSmem decode_smem_layout(int kv, int d, int ntw, int wr, int wb,
                                                         int stages, int rows) {
  DecodeSmem s{};
  const int rows_pad = 8 * ntw * wr;
  s.ring = 0;
  s.scales = s.ring + (size_t)stages * 2 * tile_bytes(kv, d);
  s.bars = s.scales + (kv == kKvInt8 ? (size_t)stages * 128 : 0);
  s.qs = s.bars + (size_t)stages * 2 * 8;
  s.qs = (s.qs + 15) & ~(size_t)15;
  s.mrg_o = s.qs + (size_t)rows_pad * (d * 2 + 16);
  s.mrg_ml = s.mrg_o + (size_t)wb * rows * (d + 4) * 4;
  s.fin_ml = s.mrg_ml + (size_t)((wb * rows * 2 * 4 + 15) & ~15);   // a split piece's merged m, l
  s.misc = s.fin_ml + (size_t)((rows * 2 * 4 + 15) & ~15);
  s.total = s.misc + 256;   // block-reduce scratch, CTA plan, abort flag, split-finish state
  return s;
}

// Tensor-core (tcgen05) decode kernel for wide units: 128-token chunks (8 KV
// blocks, the MMA's M), 8 softmax warps, 1 MMA-issue warp, 1 TMA warp.
constexpr int kTcChunk = 8;          // KV blocks per chunk
constexpr int kTcThreads = 320;
// Tensor memory: S^T buffers at columns [0, 64) and [64, 128), O^T at
// [128, 192), fp16 K buffers (two per column) at [256, 320) and [320, 384).
constexpr int kTcTmemCols = 512;

// Shared memory of the tcgen05 kernel for rows_pad (32 or 64) query rows and
// nbuf ring buffers of one E5M2 chunk each (8 K tiles + 8 V tiles, 32 KB).
struct TcSmem {
  size_t v16, p, q, ring, bars, misc, total;
};
__host__ __device__ inline TcSmem tc_smem_layout(int rows_pad, int nbuf) {
  TcSmem s{};
  const size_t wide = 128 * 128 * 2;          // one chunk of V widened to fp16
  const size_t rows_bytes = (size_t)rows_pad * 256;
  s.v16 = 0;                                   // two buffers
  s.p = s.v16 + 2 * wide;                      // P^T: 128 tokens x 64 row slots (fp16)
  s.q = s.p + 128 * 64 * 2;                    // two buffers
  s.ring = s.q + 2 * rows_bytes;
  s.bars = s.ring + (size_t)nbuf * 2 * kTcChunk * kBlockSize * 128;
  s.misc = s.bars + (size_t)(2 * nbuf + 5) * 8;
  s.misc = (s.misc + 15) & ~(size_t)15;
  // TMEM address, per-quarter row maxima and row sums [4][rows_pad] each,
  // running max [2][rows_pad], 1 / row sum and rescale factor [rows_pad] each,
  // plan scan scratch, plan, abort and finish flags.
  s.total = s.misc + 16 + (size_t)12 * rows_pad * 4 + 16 * 8 + 5 * 8 + 16 * 4;
  return s;
}
const void* decode_tc_kernel_ptr(int kv, int rc);

// Kernel entry points, one set per KV dtype translation unit (nullptr if the
// head size / rows-per-warp combination is not instantiated).
const void* decode_kernel_ptr_f16(int d, int ntw);
const void* decode_kernel_ptr_bf16(int d, int ntw);
const void* decode_kernel_ptr_e5m2(int d, int ntw);
const void* decode_kernel_ptr_int8(int d, int ntw);
// The 96-thread kernel for units of at most 8 rows over a bf16 cache (nullptr if none).
const void* decode_kernel_narrow_ptr_bf16(int d);
const void* kv_cache_write_kernel_ptr();
const void* kv_cache_write_int8_kernel_ptr();

struct CacheWriteArgs {
  const uint4* key;            // [T][Hkv][D] 16-bit elements, 8 per uint4
  const uint4* value;
  const int32_t* slot_mapping; // [T]
  void* k_cache;
  void* v_cache;
  int32_t* status;
  long long num_slots;         // num_blocks * 16
  int32_t num_tokens;
  int32_t num_kv_heads;
  int32_t head_size;
  int32_t kv;                  // kKvF16 / kKvBf16 / kKvE5m2 / kKvInt8
  float* scales;               // INT8 cache: [num_blocks][num_kv_heads][2][16] K then V row scales
};

}  // namespace pkv
