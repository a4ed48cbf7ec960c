// Block copy for copy-on-write (declared in include/pagedkv.h): physical block
// dst[i] of the K and the V cache (and, for an INT8 cache, of its row scales)
// becomes a copy of block src[i]. A block of one cache is contiguous
// ([num_kv_heads][16][head_size] elements), and so are its scales
// ([num_kv_heads][2][16] floats), so the copy is a grid-stride loop of 16-byte
// loads and stores over (pair, array, chunk).
#include <cuda_runtime.h>

#include <cstdint>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace pkv {

struct CopyBlocksArgs {
  uint4* k_cache;
  uint4* v_cache;
  uint4* scales;                // INT8 row scales, or null
  const int32_t* src;
  const int32_t* dst;
  int32_t* status;
  long long chunks_per_block;   // 16-byte chunks in one block of one cache
  long long scale_chunks;       // 16-byte chunks of one block's scales (0 without scales)
  int32_t num_blocks;
  int32_t n;
};

__global__ void __launch_bounds__(256) copy_blocks_kernel(const CopyBlocksArgs a) {
  const long long per_pair = 2 * a.chunks_per_block + a.scale_chunks;
  const long long total = static_cast<long long>(a.n) * per_pair;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int pair = static_cast<int>(i / per_pair);
    const long long r = i - pair * per_pair;
    // r: K chunks, then V chunks, then scale chunks
    uint4* base;
    long long c, stride;
    if (r < 2 * a.chunks_per_block) {
      const bool is_v = r >= a.chunks_per_block;
      base = is_v ? a.v_cache : a.k_cache;
      c = is_v ? r - a.chunks_per_block : r;
      stride = a.chunks_per_block;
    } else {
      base = a.scales;
      c = r - 2 * a.chunks_per_block;
      stride = a.scale_chunks;
    }
    const int s = a.src[pair], d = a.dst[pair];
    if (static_cast<unsigned>(s) >= static_cast<unsigned>(a.num_blocks) ||
        static_cast<unsigned>(d) >= static_cast<unsigned>(a.num_blocks)) {
      if (r == 0 && a.status) atomicOr(a.status, kDevBadBlock);
      continue;
    }
    base[static_cast<long long>(d) * stride + c] = base[static_cast<long long>(s) * stride + c];
  }
}

}  // namespace pkv

extern "C" int pkv_copy_blocks(void* k_cache, void* v_cache, float* scales, pkv_dtype kv_dtype,
                               const pkv_cache_desc* cache, const int32_t* src, const int32_t* dst, int32_t n,
                               int32_t* device_status, void* stream) {
  using namespace pkv;
  if (!cache || n < 0) return PKV_ERR_INVALID_ARGUMENT;
  if (kv_dtype != PKV_FP16 && kv_dtype != PKV_BF16 && kv_dtype != PKV_FP8_E5M2 && kv_dtype != PKV_INT8)
    return PKV_ERR_UNSUPPORTED;
  // An INT8 cache's blocks are copied with their row scales; other caches have none.
  if ((kv_dtype == PKV_INT8) != (scales != nullptr)) return PKV_ERR_INVALID_ARGUMENT;
  if (scales && (reinterpret_cast<uintptr_t>(scales) & 15u)) return PKV_ERR_INVALID_ARGUMENT;
  if (cache->block_size != kBlockSize || cache->num_blocks <= 0 || cache->num_kv_heads <= 0 ||
      (cache->head_size != 64 && cache->head_size != 128))
    return PKV_ERR_INVALID_ARGUMENT;
  if (n == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src || !dst) return PKV_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15u)
    return PKV_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 3u) return PKV_ERR_INVALID_ARGUMENT;
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u)) return PKV_ERR_INVALID_ARGUMENT;
  CopyBlocksArgs a{};
  a.k_cache = static_cast<uint4*>(k_cache);
  a.v_cache = static_cast<uint4*>(v_cache);
  a.scales = reinterpret_cast<uint4*>(scales);
  a.src = src;
  a.dst = dst;
  a.status = device_status;
  a.chunks_per_block = static_cast<long long>(cache->num_kv_heads) * kBlockSize * cache->head_size *
                       kv_elem_bytes(static_cast<int>(kv_dtype)) / 16;
  a.scale_chunks = scales ? static_cast<long long>(cache->num_kv_heads) * 2 * kBlockSize * 4 / 16 : 0;
  a.num_blocks = cache->num_blocks;
  a.n = n;
  const long long total = static_cast<long long>(n) * (2 * a.chunks_per_block + a.scale_chunks);
  long long blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  copy_blocks_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  return PKV_OK;
}
