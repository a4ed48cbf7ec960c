// Cache write: scatter new tokens into their physical slots ("kernel1" of the
// KVCache Quant section of "AI大模型推理速度翻倍，Colossal-Inference开源发布":
// when the cache is FP8 E5M2, the writer casts fp16 to fp8).
//
// One thread moves one 16-byte chunk (8 elements) of one token's key or value
// row; consecutive threads cover consecutive chunks of a row, so both the read
// of key/value and the write of the cache row are coalesced.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {

// fp16 bit pattern -> E5M2 byte. E5M2 keeps fp16's sign, exponent field and
// bias and the top two mantissa bits, so rounding the 16-bit magnitude at bit 8
// (round half to even: add 0x7F plus the bit that will become the last kept
// mantissa bit) yields the E5M2 magnitude directly; a carry moves into the
// exponent as it should. Results beyond the largest finite code 0x7B (57344),
// including infinities, saturate to it; NaN becomes 0x7E; the sign is kept.
__device__ __forceinline__ uint32_t e5m2_of_fp16(uint32_t h) {
  const uint32_t mag = h & 0x7FFFu;
  uint32_t r = (mag + 0x7Fu + ((mag >> 8) & 1u)) >> 8;
  r = r > 0x7Bu ? 0x7Bu : r;
  r = mag > 0x7C00u ? 0x7Eu : r;
  return ((h >> 8) & 0x80u) | r;
}

__device__ __forceinline__ uint32_t e5m2x4(uint32_t lo_pair, uint32_t hi_pair) {
  return e5m2_of_fp16(lo_pair & 0xFFFFu) | (e5m2_of_fp16(lo_pair >> 16) << 8) |
         (e5m2_of_fp16(hi_pair & 0xFFFFu) << 16) | (e5m2_of_fp16(hi_pair >> 16) << 24);
}

__global__ void __launch_bounds__(256) kv_cache_write_kernel(const CacheWriteArgs a) {
  pdl_wait_prior_grid();
  const int chunks_per_row = a.head_size / 8;
  const long long per_tensor = static_cast<long long>(a.num_tokens) * a.num_kv_heads * chunks_per_row;
  const long long total = 2 * per_tensor;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const bool is_v = idx >= per_tensor;
    const long long rem = is_v ? idx - per_tensor : idx;
    const int t = static_cast<int>(rem / (static_cast<long long>(a.num_kv_heads) * chunks_per_row));
    const int hc = static_cast<int>(rem - static_cast<long long>(t) * a.num_kv_heads * chunks_per_row);
    const int h = hc / chunks_per_row, ch = hc - h * chunks_per_row;
    const long long slot = a.slot_mapping[t];
    if (slot == -1) continue;
    if (slot < 0 || slot >= a.num_slots) {
      if (a.status) atomicOr(a.status, kDevBadSlot);
      continue;
    }
    const long long blk = slot / kBlockSize, off = slot - blk * kBlockSize;
    const long long dst = ((blk * a.num_kv_heads + h) * kBlockSize + off) * a.head_size + ch * 8;
    const uint4 v = (is_v ? a.value : a.key)[rem];
    void* cache = is_v ? a.v_cache : a.k_cache;
    if (a.kv == kKvE5m2) {
      uint2 o;
      o.x = e5m2x4(v.x, v.y);
      o.y = e5m2x4(v.z, v.w);
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(cache) + dst) = o;
    } else {
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(cache) + dst) = v;
    }
  }
  pdl_launch_dependents();
}

const void* kv_cache_write_kernel_ptr() { return reinterpret_cast<const void*>(&kv_cache_write_kernel); }

// INT8 cache write (the "KV Cache INT8 量化" the inference-framework survey lists
// for LMDeploy; the codec is ours): one warp quantises one (token, head) row of
// K or V. scale = max|x| / 127 rounded up to the nearest fp16 value (so that the
// decode can fold it into an fp16 weight exactly) and code = round-half-even(x /
// scale) clamped to [-127, 127]; both divisions are IEEE fp32 (__fdiv_rn), so the
// codes do not depend on compiler flags. An all-zero row gets scale 0 and codes 0. Codes are
// stored in offset binary (byte = code + 128), which the decode kernel widens
// to fp16 with a single byte permute.
__global__ void __launch_bounds__(256) kv_cache_write_int8_kernel(const CacheWriteArgs a) {
  pdl_wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int per_lane = a.head_size / 32;   // 4 (head 128) or 2 (head 64) elements
  const long long rows = 2ll * a.num_tokens * a.num_kv_heads;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long w = warp0; w < rows; w += nwarps) {
    const bool is_v = w >= static_cast<long long>(a.num_tokens) * a.num_kv_heads;
    const long long th = is_v ? w - static_cast<long long>(a.num_tokens) * a.num_kv_heads : w;
    const int t = static_cast<int>(th / a.num_kv_heads), h = static_cast<int>(th - static_cast<long long>(t) * a.num_kv_heads);
    const long long slot = a.slot_mapping[t];
    if (slot == -1) continue;
    if (slot < 0 || slot >= a.num_slots) {
      if (lane == 0 && !is_v && a.status) atomicOr(a.status, kDevBadSlot);
      continue;
    }
    const __half* src = reinterpret_cast<const __half*>(is_v ? a.value : a.key) + th * a.head_size + lane * per_lane;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (i < per_lane) {
        x[i] = __half2float(src[i]);
        amax = fmaxf(amax, fabsf(x[i]));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = __half2float(__float2half_ru(__fdiv_rn(amax, 127.0f)));
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (i >= per_lane) break;
      float qv = 0.f;
      if (scale != 0.f) {
        qv = rintf(__fdiv_rn(x[i], scale));
        qv = fmaxf(qv, -127.0f);
        qv = fminf(qv, 127.0f);
      }
      packed |= static_cast<uint32_t>(static_cast<int>(qv) + 128) << (8 * i);
    }
    const long long blk = slot / kBlockSize, off = slot - blk * kBlockSize;
    const long long row = (blk * a.num_kv_heads + h) * kBlockSize + off;
    uint8_t* dst = static_cast<uint8_t*>(is_v ? a.v_cache : a.k_cache) + row * a.head_size + lane * per_lane;
    if (per_lane == 4) {
      *reinterpret_cast<uint32_t*>(dst) = packed;
    } else {
      *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(packed);
    }
    // [block][head][K, V][16]: row = (block * Hkv + head) * 16 + token
    if (lane == 0) a.scales[(row >> 4) * 32 + (is_v ? 16 : 0) + (row & 15)] = scale;
  }
  pdl_launch_dependents();
}

const void* kv_cache_write_int8_kernel_ptr() {
  return reinterpret_cast<const void*>(&kv_cache_write_int8_kernel);
}

}  // namespace pkv
