// Dequantised export of one int8 group-64 affine matrix (a check of the code,
// scale and bias indexing the decode kernel's GEMV phases use).
#include "common.cuh"
#include "decode.h"

namespace q35 {
namespace {

__global__ void dequant_kernel(const uint8_t* codes, const uint16_t* scales, const uint16_t* biases,
                               uint32_t n, uint32_t k, uint32_t gstride, float* out) {
  const uint64_t total = (uint64_t)n * k;
  for (uint64_t e = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; e < total;
       e += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t r = (uint32_t)(e / k), c = (uint32_t)(e % k);
    const float s = bf16f(scales[(size_t)r * gstride + c / 64]);
    const float b = bf16f(biases[(size_t)r * gstride + c / 64]);
    out[e] = fmaf(s, (float)codes[e], b);
  }
}

}  // namespace

cudaError_t dequant_launch(const uint8_t* codes, const uint16_t* scales, const uint16_t* biases, uint32_t n,
                           uint32_t k, uint32_t gstride, float* out, cudaStream_t stream) {
  const uint64_t total = (uint64_t)n * k;
  uint64_t blocks = (total + 255) / 256;
  if (blocks > 65535) blocks = 65535;
  dequant_kernel<<<(unsigned)blocks, 256, 0, stream>>>(codes, scales, biases, n, k, gstride, out);
  return cudaGetLastError();
}

}  // namespace q35
