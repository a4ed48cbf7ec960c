// Instantiations of the decode kernel for the f16 KV cache.
#include "decode_kernel.cuh"

namespace pkv {

const void* decode_kernel_ptr_f16(int d, int ntw) {
  if (d == 64 && ntw == 1) return reinterpret_cast<const void*>(&decode_kernel<0, 64, 1>);
  if (d == 64 && ntw == 2) return reinterpret_cast<const void*>(&decode_kernel<0, 64, 2>);
  if (d == 128 && ntw == 1) return reinterpret_cast<const void*>(&decode_kernel<0, 128, 1>);
  if (d == 128 && ntw == 2) return reinterpret_cast<const void*>(&decode_kernel<0, 128, 2>);
  return nullptr;
}

}  // namespace pkv
