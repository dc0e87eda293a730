// The decode kernel's instantiations for attention head dim 128.
#include "decode_kernel.cuh"

namespace q35 {

DecodeKernel decode_kernel_d128(uint32_t hpw, uint32_t Dk, bool batched) {
  return decode_kernel_for<128>(hpw, Dk, batched);
}

}  // namespace q35
