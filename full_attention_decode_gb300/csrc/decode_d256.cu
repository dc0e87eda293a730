// The decode kernel's instantiations for attention head dim 256.
#include "decode_kernel.cuh"

namespace q35 {

DecodeKernel decode_kernel_d256(uint32_t hpw, uint32_t Dk, bool batched) {
  return decode_kernel_for<256>(hpw, Dk, batched);
}

}  // namespace q35
