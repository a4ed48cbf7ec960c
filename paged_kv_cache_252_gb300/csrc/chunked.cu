// Decode attention for batches whose sequences may carry any number of query tokens
// (prefill chunks beside decode and verify tokens: the mixed batch of the
// Continuous Batching section of "AI大模型推理速度翻倍，Colossal-Inference开源发布").
//
// A sequence's query tokens are cut into row tiles of q_tile tokens: 64 / G (G query
// heads per KV head), the most one decode unit holds, or fewer when no sequence has
// that many (a batch of plain decodes keeps the one-token units, and the kernels'
// narrow geometry, of the other entry points). Tile t of sequence s
// (tokens t*q_tile .. t*q_tile + n_t - 1 of its n_s) runs as a sequence of its own:
// its token j' is token j = t*q_tile + j' of s, which sees positions
// <= ctx_s - n_s + j, so the tile is a sequence of n_t tokens with context length
// ctx_s - n_s + t*q_tile + n_t under the same causal rule. The tiles' lengths and
// query-row offsets are computed here from the caller's host arrays and passed to
// a setup kernel as its parameters (copied at launch: no host synchronisation, and
// the call can be captured in a CUDA graph), which writes them into the workspace
// and copies each tile's block-table row from its sequence's; the varlen decode
// then runs over the tiles.
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace pkv {

// Tiles v0 .. v0+n-1 of a chunked call (at most kSetupTiles per launch, so that the
// parameters stay under 4 KB).
constexpr int kSetupTiles = 320;
struct ChunkSetup {
  int32_t v0, n, tiles, rows, mbs;
  int32_t ctx[kSetupTiles];   // context length of each tile
  int32_t cu[kSetupTiles];    // first query row of each tile
  int32_t seq[kSetupTiles];   // the sequence whose block-table row it reads
};

// Writes the tiles' lengths and row offsets (cu[tiles] = rows after the last tile)
// and copies their block-table rows: vbt[v][k] = block_tables[seq[v]][k].
__global__ void chunk_setup_kernel(const __grid_constant__ ChunkSetup p, const int32_t* block_tables,
                                   int32_t* ctx, int32_t* cu, int32_t* vbt) {
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = tid; i < p.n; i += stride) {
    ctx[p.v0 + i] = p.ctx[i];
    cu[p.v0 + i] = p.cu[i];
  }
  if (tid == 0 && p.v0 + p.n == p.tiles) cu[p.tiles] = p.rows;
  const long long n = static_cast<long long>(p.n) * p.mbs;
  for (long long i = tid; i < n; i += stride) {
    const long long v = i / p.mbs, k = i - v * p.mbs;
    vbt[(p.v0 + v) * p.mbs + k] = block_tables[static_cast<long long>(p.seq[v]) * p.mbs + k];
  }
}

}  // namespace pkv

namespace {

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Tiles of the batch: q_tile tokens each (the last of a sequence may hold fewer).
// Returns false for arguments that cannot describe a batch.
bool count_tiles(const int32_t* host_q_lens, int32_t num_seqs, int32_t num_q_heads, const pkv_cache_desc* cache,
                 int* q_tile, long long* tiles, long long* rows) {
  if (num_seqs < 0 || num_q_heads <= 0 || !cache || cache->num_kv_heads <= 0) return false;
  if (num_q_heads % cache->num_kv_heads != 0) return false;
  const int group = num_q_heads / cache->num_kv_heads;
  if (group > 64) return false;
  if (num_seqs > 0 && !host_q_lens) return false;
  int max_n = 1;
  for (int32_t s = 0; s < num_seqs; ++s) {
    if (host_q_lens[s] < 1) return false;
    if (host_q_lens[s] > max_n) max_n = host_q_lens[s];
  }
  *q_tile = 64 / group < max_n ? 64 / group : max_n;
  *tiles = 0;
  *rows = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t n = host_q_lens[s];
    *tiles += (n + *q_tile - 1) / *q_tile;
    *rows += n;
  }
  return *tiles < (1ll << 31) && *rows < (1ll << 31);
}

// Workspace: [the varlen decode's workspace] [tile context lengths | tile cu_q_lens
// (tiles + 1)] [tile block-table rows], each part 256-aligned.
// The decode's part comes first, where every decode call keeps its piece counters,
// so a buffer shared with the other entry points holds counters there.
struct ChunkedLayout {
  size_t decode, decode_bytes, meta, vbt, total;
};

ChunkedLayout chunked_layout(long long tiles, int32_t max_blocks_per_seq, size_t decode_bytes) {
  ChunkedLayout L{};
  L.decode = 0;
  L.decode_bytes = decode_bytes;
  L.meta = round256(decode_bytes);
  L.vbt = L.meta + round256(static_cast<size_t>(2 * tiles + 1) * sizeof(int32_t));
  L.total = L.vbt + round256(static_cast<size_t>(tiles) * max_blocks_per_seq * sizeof(int32_t));
  return L;
}

}  // namespace

extern "C" {

size_t pkv_decode_chunked_workspace_bytes(const int32_t* host_q_lens, int32_t num_seqs, int32_t num_q_heads,
                                          int32_t max_blocks_per_seq, const pkv_cache_desc* cache) {
  int q_tile = 0;
  long long tiles = 0, rows = 0;
  if (max_blocks_per_seq <= 0 || !count_tiles(host_q_lens, num_seqs, num_q_heads, cache, &q_tile, &tiles, &rows))
    return 0;
  const size_t dec = pkv_decode_workspace_bytes(static_cast<int32_t>(tiles), num_q_heads, q_tile, cache);
  if (dec == 0 && tiles > 0) return 0;
  return chunked_layout(tiles, max_blocks_per_seq, dec).total;
}

int pkv_paged_attention_decode_chunked(void* out, const void* q, const int32_t* host_q_lens,
                                       const int32_t* host_context_lens, int32_t num_seqs, int32_t num_q_heads,
                                       const void* k_cache, const void* v_cache, const float* scales,
                                       pkv_dtype kv_dtype, const pkv_cache_desc* cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq, float scale,
                                       void* workspace, size_t workspace_bytes, int32_t* device_status,
                                       void* stream) {
  int q_tile = 0;
  long long tiles = 0, rows = 0;
  if (max_blocks_per_seq <= 0 || !count_tiles(host_q_lens, num_seqs, num_q_heads, cache, &q_tile, &tiles, &rows))
    return PKV_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0) return PKV_OK;
  if (!host_context_lens || !block_tables || !workspace) return PKV_ERR_INVALID_ARGUMENT;
  for (int32_t s = 0; s < num_seqs; ++s)
    if (host_context_lens[s] < host_q_lens[s]) return PKV_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || (reinterpret_cast<uintptr_t>(block_tables) & 3u) != 0)
    return PKV_ERR_INVALID_ARGUMENT;
  const size_t dec = pkv_decode_workspace_bytes(static_cast<int32_t>(tiles), num_q_heads, q_tile, cache);
  if (dec == 0) return PKV_ERR_UNSUPPORTED;
  const ChunkedLayout L = chunked_layout(tiles, max_blocks_per_seq, dec);
  if (workspace_bytes < L.total) return PKV_ERR_WORKSPACE_TOO_SMALL;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long T = tiles;
  int32_t* d_ctx = reinterpret_cast<int32_t*>(ws + L.meta);
  int32_t* d_cu = d_ctx + T;
  int32_t* d_vbt = reinterpret_cast<int32_t*>(ws + L.vbt);
  // Tiles in order, kSetupTiles per setup launch.
  pkv::ChunkSetup p{};
  p.tiles = static_cast<int32_t>(T);
  p.rows = static_cast<int32_t>(rows);
  p.mbs = max_blocks_per_seq;
  auto flush = [&]() -> bool {
    if (p.n == 0) return true;
    const long long work = static_cast<long long>(p.n) * max_blocks_per_seq;
    const unsigned blocks = static_cast<unsigned>(work / 256 + 1 < 1024 ? work / 256 + 1 : 1024);
    pkv::chunk_setup_kernel<<<blocks, 256, 0, st>>>(p, block_tables, d_ctx, d_cu, d_vbt);
    if (cudaGetLastError() != cudaSuccess) return false;
    p.v0 += p.n;
    p.n = 0;
    return true;
  };
  long long row = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t n = host_q_lens[s], ctx = host_context_lens[s];
    for (int32_t t0 = 0; t0 < n; t0 += q_tile) {
      const int32_t nt = n - t0 < q_tile ? n - t0 : q_tile;
      p.ctx[p.n] = ctx - n + t0 + nt;
      p.cu[p.n] = static_cast<int32_t>(row + t0);
      p.seq[p.n] = s;
      if (++p.n == pkv::kSetupTiles && !flush()) return PKV_ERR_CUDA;
    }
    row += n;
  }
  if (!flush()) return PKV_ERR_CUDA;

  void* wdec = ws + L.decode;
  // The tiles' piece counters start clear (the region may hold another call's data).
  if (cudaMemsetAsync(wdec, 0, pkv::decode_counter_bytes(T * cache->num_kv_heads), st) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  if (kv_dtype == PKV_INT8) {
    return pkv_paged_attention_decode_int8_varlen(out, q, d_cu, static_cast<int32_t>(rows), static_cast<int32_t>(T),
                                                  num_q_heads, q_tile, k_cache, v_cache, scales, cache, d_vbt,
                                                  max_blocks_per_seq, d_ctx, scale, wdec, L.decode_bytes,
                                                  device_status, stream);
  }
  return pkv_paged_attention_decode_varlen(out, q, d_cu, static_cast<int32_t>(rows), static_cast<int32_t>(T),
                                           num_q_heads, q_tile, k_cache, v_cache, kv_dtype, cache, d_vbt,
                                           max_blocks_per_seq, d_ctx, scale, wdec, L.decode_bytes, device_status,
                                           stream);
}

}  // extern "C"
