// Instantiations of the decode kernel for the bf16 KV cache.
#include "decode_kernel.cuh"

namespace pkv {

const void* decode_kernel_ptr_bf16(int d, int ntw) {
  if (d == 64 && ntw == 1) return reinterpret_cast<const void*>(&decode_kernel<1, 64, 1>);
  if (d == 64 && ntw == 2) return reinterpret_cast<const void*>(&decode_kernel<1, 64, 2>);
  if (d == 128 && ntw == 1) return reinterpret_cast<const void*>(&decode_kernel<1, 128, 1>);
  if (d == 128 && ntw == 2) return reinterpret_cast<const void*>(&decode_kernel<1, 128, 2>);
  return nullptr;
}

// Units of at most 8 rows: the 96-thread kernel with 144 registers.
const void* decode_kernel_narrow_ptr_bf16(int d) {
  if (d == 64) return reinterpret_cast<const void*>(&decode_kernel_narrow<1, 64, 144>);
  if (d == 128) return reinterpret_cast<const void*>(&decode_kernel_narrow<1, 128, 144>);
  return nullptr;
}

}  // namespace pkv
