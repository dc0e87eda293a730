// Greedy token choice over the output head's bf16 logits: the index of the largest
// value, the lowest index among equal ones. NaN logits are never chosen (if every
// logit is NaN the result is -1).
#include <cstdint>

#include "decode.h"

namespace q35 {
namespace {

constexpr uint32_t kArgmaxThreads = 1024;

// (v, i) replaces the best so far (bv, bi): a larger value, or an equal value at a
// lower index.
__device__ __forceinline__ void take_better(float v, uint32_t i, float& bv, uint32_t& bi) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void warp_best(float& bv, uint32_t& bi) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const uint32_t oi = __shfl_xor_sync(0xffffffffu, bi, o);
    take_better(ov, oi, bv, bi);
  }
}

// One block: each thread scans 8-value chunks (16-byte loads) j = tid, tid + 1024, ...
// in increasing index order, then the tail; a warp and then a block reduction.
__global__ void __launch_bounds__(kArgmaxThreads) argmax_bf16_kernel(const uint16_t* __restrict__ v, uint32_t n,
                                                                     int32_t* __restrict__ out) {
  float bv = -__int_as_float(0x7f800000);  // -inf
  uint32_t bi = 0xffffffffu;
  const uint32_t n8 = n / 8;
  const uint4* v8 = reinterpret_cast<const uint4*>(v);
#pragma unroll 8
  for (uint32_t j = threadIdx.x; j < n8; j += kArgmaxThreads) {
    const uint4 u = v8[j];
    const uint32_t b = 8 * j;
    take_better(bf16_lo(u.x), b + 0, bv, bi);
    take_better(bf16_hi(u.x), b + 1, bv, bi);
    take_better(bf16_lo(u.y), b + 2, bv, bi);
    take_better(bf16_hi(u.y), b + 3, bv, bi);
    take_better(bf16_lo(u.z), b + 4, bv, bi);
    take_better(bf16_hi(u.z), b + 5, bv, bi);
    take_better(bf16_lo(u.w), b + 6, bv, bi);
    take_better(bf16_hi(u.w), b + 7, bv, bi);
  }
  for (uint32_t i = 8 * n8 + threadIdx.x; i < n; i += kArgmaxThreads) take_better(bf16_lo(v[i]), i, bv, bi);
  warp_best(bv, bi);
  __shared__ float sv[kArgmaxThreads / 32];
  __shared__ uint32_t si[kArgmaxThreads / 32];
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    bv = sv[lane];
    bi = si[lane];
    warp_best(bv, bi);
    if (lane == 0) *out = bi == 0xffffffffu ? -1 : (int32_t)bi;
  }
}

}  // namespace

cudaError_t argmax_bf16_launch(const uint16_t* v, uint32_t n, int32_t* out, cudaStream_t stream) {
  argmax_bf16_kernel<<<1, kArgmaxThreads, 0, stream>>>(v, n, out);
  return cudaGetLastError();
}

}  // namespace q35
