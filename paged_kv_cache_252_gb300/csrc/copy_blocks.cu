// Block copy for copy-on-write (declared in include/pagedkv.h): physical block
// dst[i] of the K and the V cache becomes a copy of block src[i]. A block of one
// cache is contiguous ([num_kv_heads][16][head_size] elements), so the copy is a
// grid-stride loop of 16-byte loads and stores over (pair, cache, chunk).
#include <cuda_runtime.h>

#include <cstdint>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace pkv {

struct CopyBlocksArgs {
  uint4* k_cache;
  uint4* v_cache;
  const int32_t* src;
  const int32_t* dst;
  int32_t* status;
  long long chunks_per_block;   // 16-byte chunks in one block of one cache
  int32_t num_blocks;
  int32_t n;
};

__global__ void __launch_bounds__(256) copy_blocks_kernel(const CopyBlocksArgs a) {
  const long long per_pair = 2 * a.chunks_per_block;
  const long long total = static_cast<long long>(a.n) * per_pair;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int pair = static_cast<int>(i / per_pair);
    const long long r = i - pair * per_pair;
    const bool is_v = r >= a.chunks_per_block;
    const long long c = is_v ? r - a.chunks_per_block : r;
    const int s = a.src[pair], d = a.dst[pair];
    if (static_cast<unsigned>(s) >= static_cast<unsigned>(a.num_blocks) ||
        static_cast<unsigned>(d) >= static_cast<unsigned>(a.num_blocks)) {
      if (c == 0 && !is_v && a.status) atomicOr(a.status, kDevBadBlock);
      continue;
    }
    uint4* base = is_v ? a.v_cache : a.k_cache;
    base[static_cast<long long>(d) * a.chunks_per_block + c] = base[static_cast<long long>(s) * a.chunks_per_block + c];
  }
}

}  // namespace pkv

extern "C" int pkv_copy_blocks(void* k_cache, void* v_cache, pkv_dtype kv_dtype, const pkv_cache_desc* cache,
                               const int32_t* src, const int32_t* dst, int32_t n, int32_t* device_status,
                               void* stream) {
  using namespace pkv;
  if (!cache || n < 0) return PKV_ERR_INVALID_ARGUMENT;
  if (kv_dtype != PKV_FP16 && kv_dtype != PKV_BF16 && kv_dtype != PKV_FP8_E5M2) return PKV_ERR_UNSUPPORTED;
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
  a.src = src;
  a.dst = dst;
  a.status = device_status;
  a.chunks_per_block = static_cast<long long>(cache->num_kv_heads) * kBlockSize * cache->head_size *
                       kv_elem_bytes(static_cast<int>(kv_dtype)) / 16;
  a.num_blocks = cache->num_blocks;
  a.n = n;
  const long long total = 2ll * n * a.chunks_per_block;
  long long blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  copy_blocks_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  return PKV_OK;
}
