// Device-side self-test of the bounded waits every decode kernel uses: failure
// detection exercised on the GPU without a fault, on an mbarrier phase that nothing
// completes.
#include <cuda_runtime.h>

#include "decode_common.cuh"
#include "pagedkv.h"

namespace pkv {

// Thread 0 of warp 0 waits with limit_ns, thread 0 of warp 1 with the decode
// kernels' own limit; each on a barrier phase no one completes. The first gives up
// after limit_ns, raises the CTA's abort flag and sets kDevTimeout; the second
// leaves when it sees the flag. elapsed[w] = wait w's duration in ns.
__global__ void bounded_wait_probe_kernel(int32_t* status, unsigned long long limit_ns,
                                          unsigned long long* elapsed) {
  __shared__ alignas(8) unsigned long long bars[2];
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bars[0]), 1);
    mbar_init(smem_addr(&bars[1]), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (lane == 0 && warp < 2) {
    const uint64_t t0 = global_timer_ns();
    const bool ok = wait_or_abort_for(smem_addr(&bars[warp]), 0u, abort_flag, warp == 0 ? limit_ns : kWaitLimitNs);
    if (!ok) {
      *abort_flag = 1;
      atomicOr(status, kDevTimeout);
    }
    elapsed[warp] = global_timer_ns() - t0;
  }
}

}  // namespace pkv

extern "C" int pkv_selftest_bounded_wait(int32_t* device_status, uint64_t limit_ns,
                                         unsigned long long* device_elapsed_ns, void* stream) {
  if (!device_status || !device_elapsed_ns || (reinterpret_cast<uintptr_t>(device_status) & 3u) ||
      (reinterpret_cast<uintptr_t>(device_elapsed_ns) & 7u) || limit_ns == 0 || limit_ns > pkv::kWaitLimitNs)
    return PKV_ERR_INVALID_ARGUMENT;
  pkv::bounded_wait_probe_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(device_status, limit_ns,
                                                                               device_elapsed_ns);
  if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  return PKV_OK;
}
