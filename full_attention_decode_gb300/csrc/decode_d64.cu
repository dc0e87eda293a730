// The decode kernel's instantiations for attention head dim 64.
#include "decode_kernel.cuh"

namespace q35 {

DecodeKernel decode_kernel_d64(uint32_t hpw, uint32_t Dk, bool batched) {
  return decode_kernel_for<64>(hpw, Dk, batched);
}

}  // namespace q35
