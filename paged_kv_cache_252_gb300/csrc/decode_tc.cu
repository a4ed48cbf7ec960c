// Instantiations of the tcgen05 decode kernel (E5M2 cache, head size 128) for
// units of up to 32 (rc = 1) and up to 64 (rc = 2) query rows.
#include "decode_tc_kernel.cuh"

namespace pkv {

const void* decode_tc_kernel_ptr(int kv, int rc) {
  if (kv == kKvE5m2 && rc == 1) return reinterpret_cast<const void*>(&decode_tc_kernel<1>);
  if (kv == kKvE5m2 && rc == 2) return reinterpret_cast<const void*>(&decode_tc_kernel<2>);
  return nullptr;
}

}  // namespace pkv
