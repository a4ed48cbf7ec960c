// Decode attention for batches whose sequences may carry any number of query tokens
// (prefill chunks beside decode and verify tokens: the mixed batch of the
// Continuous Batching section of "AI大模型推理速度翻倍，Colossal-Inference开源发布").
//
// A sequence's query tokens are cut into row tiles of q_tile = 64 / G tokens (G
// query heads per KV head), the most one decode unit holds. Tile t of sequence s
// (tokens t*q_tile .. t*q_tile + n_t - 1 of its n_s) runs as a sequence of its own:
// its token j' is token j = t*q_tile + j' of s, which sees positions
// <= ctx_s - n_s + j, so the tile is a sequence of n_t tokens with context length
// ctx_s - n_s + t*q_tile + n_t under the same causal rule. The tiles' lengths and
// query-row offsets are computed here from the caller's host arrays and uploaded
// into the workspace; one kernel copies each tile's block-table row from its
// sequence's; the varlen decode then runs over the tiles.
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace pkv {

// dst[v][k] = src[map[v]][k] for v < tiles, k < mbs.
__global__ void gather_block_rows_kernel(int32_t* dst, const int32_t* src, const int32_t* map, int tiles,
                                         int mbs) {
  const long long n = static_cast<long long>(tiles) * mbs;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long v = i / mbs, k = i - v * mbs;
    dst[i] = src[static_cast<long long>(map[v]) * mbs + k];
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
  *q_tile = 64 / group;
  *tiles = 0;
  *rows = 0;
  if (num_seqs > 0 && !host_q_lens) return false;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t n = host_q_lens[s];
    if (n < 1) return false;
    *tiles += (n + *q_tile - 1) / *q_tile;
    *rows += n;
  }
  return *tiles < (1ll << 31) && *rows < (1ll << 31);
}

// Workspace: [the varlen decode's workspace] [tile context lengths | tile cu_q_lens
// (tiles + 1) | tile -> sequence] [tile block-table rows], each part 256-aligned.
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
  L.vbt = L.meta + round256(static_cast<size_t>(3 * tiles + 1) * sizeof(int32_t));
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

  // Per tile: context length, first query row (prefix, tiles + 1 entries), sequence.
  const long long T = tiles;
  std::vector<int32_t> meta(static_cast<size_t>(3 * T + 1));
  int32_t* t_ctx = meta.data();
  int32_t* t_cu = t_ctx + T;
  int32_t* t_seq = t_cu + T + 1;
  long long v = 0, row = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t n = host_q_lens[s], ctx = host_context_lens[s];
    for (int32_t t0 = 0; t0 < n; t0 += q_tile, ++v) {
      const int32_t nt = n - t0 < q_tile ? n - t0 : q_tile;
      t_ctx[v] = ctx - n + t0 + nt;
      t_cu[v] = static_cast<int32_t>(row + t0);
      t_seq[v] = s;
    }
    row += n;
  }
  t_cu[T] = static_cast<int32_t>(row);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // A pageable source: the call returns once the bytes are staged, so `meta` may go.
  if (cudaMemcpyAsync(ws + L.meta, meta.data(), meta.size() * sizeof(int32_t), cudaMemcpyHostToDevice, st) !=
      cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  const int32_t* d_ctx = reinterpret_cast<const int32_t*>(ws + L.meta);
  const int32_t* d_cu = d_ctx + T;
  const int32_t* d_seq = d_cu + T + 1;
  int32_t* d_vbt = reinterpret_cast<int32_t*>(ws + L.vbt);
  const long long n = T * max_blocks_per_seq;
  const unsigned blocks = static_cast<unsigned>(n / 256 + 1 < 4096 ? n / 256 + 1 : 4096);
  pkv::gather_block_rows_kernel<<<blocks, 256, 0, st>>>(d_vbt, block_tables, d_seq, static_cast<int>(T),
                                                       max_blocks_per_seq);
  if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;

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
