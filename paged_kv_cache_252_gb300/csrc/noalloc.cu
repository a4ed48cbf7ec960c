// Allocation-free entry point for paged decode attention.
//
// Some callers cannot allocate device memory at the moment they run attention:
// code that runs inside a custom allocator's own callbacks, engines that reserve
// every byte of the device for the KV pool up front and forbid later
// cudaMalloc calls, or runtimes that only hand out fixed buffers for inputs and
// outputs. They can still run decode attention through
// pkv_paged_attention_decode_noalloc, which takes its split-KV scratch from a
// buffer built into this library instead of a caller-provided workspace.
//
// The scratch is a file-scope device array of PKV_NOALLOC_SCRATCH_BYTES. The
// driver places it in device memory when this file's module is loaded on a
// device, and it stays there until the process exits. Host code cannot use the
// array's name as a device address (on the host it is only a stand-in), so the
// first call on each device looks up its device address with
// cudaGetSymbolAddress while that device is current, and later calls reuse it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace {

constexpr size_t kScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevicesNoAlloc = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevicesNoAlloc] = {};

// Device address of the scratch array on the current device (set up once per
// device). Returns PKV_OK or an error code.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevicesNoAlloc) return PKV_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" int pkv_paged_attention_decode_noalloc(void* out, const void* q, int32_t num_seqs,
                                                  int32_t num_q_heads, int32_t q_per_seq,
                                                  const void* k_cache, const void* v_cache,
                                                  pkv_dtype kv_dtype, const pkv_cache_desc* cache,
                                                  const int32_t* block_tables,
                                                  int32_t max_blocks_per_seq,
                                                  const int32_t* context_lens, float scale,
                                                  int32_t* device_status, void* stream) {
  if (num_seqs == 0) {
    return pkv_paged_attention_decode(out, q, num_seqs, num_q_heads, q_per_seq, k_cache, v_cache,
                                      kv_dtype, cache, block_tables, max_blocks_per_seq,
                                      context_lens, scale, nullptr, 0, device_status, stream);
  }
  const size_t need = pkv_decode_workspace_bytes(num_seqs, num_q_heads, q_per_seq, cache);
  if (need == 0) {
    // The shape was refused (invalid, unsupported, or no device). Let the regular
    // entry point's host checks pick the status it would return: it is given a
    // workspace of 0 bytes, so it returns before any launch whatever the outcome
    // (the stand-in pointer is never dereferenced).
    return pkv_paged_attention_decode(out, q, num_seqs, num_q_heads, q_per_seq, k_cache, v_cache,
                                      kv_dtype, cache, block_tables, max_blocks_per_seq, context_lens,
                                      scale, reinterpret_cast<void*>(static_cast<uintptr_t>(256)), 0,
                                      device_status, stream);
  }
  // The problem needs more scratch than the built-in buffer holds.
  if (need > kScratchBytes) return PKV_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if (int rc = scratch_for_current_device(&scratch)) return rc;
  // Partial results are written before they are read. The split-KV piece
  // counters are not: they are read and bumped with atomics, and stay correct
  // because each is tagged with the call's epoch (a counter left by an earlier
  // call reads as zero), the array starts zeroed when the module loads, and the
  // CTA that completes a unit puts its counter back to zero.
  return pkv_paged_attention_decode(out, q, num_seqs, num_q_heads, q_per_seq, k_cache, v_cache,
                                    kv_dtype, cache, block_tables, max_blocks_per_seq, context_lens,
                                    scale, scratch, kScratchBytes, device_status, stream);
}
