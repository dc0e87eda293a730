// Gated DeltaNet decode step ("linear_attention.rs", forward_linear_attention:
// causal_conv1d_update_l2norm, gdn_compute_gate, sigmoid_bf16_to_f32 and
// gated_delta_rule_decode in one kernel), on sm_103a.
//
// CTA (h, j) owns v-head h and the 32 state columns [32j, 32j+32). Given the
// head's q, k, gate and beta, state columns are independent:
//   u_v = sum_i (g S[i][v]) k_i,   S[i][v] <- g S[i][v] + k_i beta (v_v - u_v),
//   y_v = sum_i S[i][v] q_i / sqrt(Dk),
// so the [Dk][32] fp32 slice is read once into registers, updated, and written
// once (the state is [Hv][Dk][Dv], contiguous in v: each warp moves 128-byte rows).
// The slice and the conv state are loaded before the kernel waits on the
// projections that precede it. Each CTA recomputes the conv + SiLU + L2 norm of
// its head's q and k channels (2*Dk channels, cheap) and of its 32 v channels.
// The CTAs that share a k-head form one thread-block cluster: a cluster barrier
// separates their reads of the q/k conv state from the one CTA that writes it
// back; every CTA writes its own v channels.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace q35 {
namespace {

constexpr int kGdnThreads = 256;
constexpr int kGdnCols = 32;
constexpr int kMaxKc = 8;

template <int DK>
__global__ void __launch_bounds__(kGdnThreads) gdn_kernel(const __grid_constant__ GdnArgs a) {
  constexpr int RPT = DK / 8;  // state rows per thread (8 warps cover Dk rows)
  constexpr int NCH = 2 * DK + kGdnCols;
  __shared__ float act[NCH];   // conv + SiLU output of this CTA's channels
  __shared__ float red[2][8][kGdnCols];
  __shared__ float stat[4];    // |q|^2, |k|^2, gate, beta

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t h = blockIdx.x, j = blockIdx.y;
  const uint32_t grp = a.Hv / a.Hk, hk = h / grp;
  const uint32_t Dv = a.Dv, Kc = a.Kc;
  const uint32_t v0 = j * kGdnCols;

  // ---- before the dependency: state slice and conv state (not written by the predecessor)
  float st[RPT];
  float* sp = a.ssm + ((size_t)h * DK + warp * RPT) * Dv + v0 + lane;
#pragma unroll
  for (int r = 0; r < RPT; ++r) st[r] = sp[(size_t)r * Dv];

  // channel of local index c: q of k-head hk, k of k-head hk, or v of this slice
  auto channel = [&](uint32_t c) -> uint32_t {
    if (c < DK) return hk * DK + c;
    if (c < 2 * DK) return a.Hk * DK + hk * DK + (c - DK);
    return 2 * a.Hk * DK + h * Dv + v0 + (c - 2 * DK);
  };
  constexpr int CPT = (NCH + kGdnThreads - 1) / kGdnThreads;  // channels per thread
  float cst[CPT][kMaxKc], cw[CPT][kMaxKc];
#pragma unroll
  for (int q = 0; q < CPT; ++q) {
    const uint32_t c = threadIdx.x + q * kGdnThreads;
    if (c < (uint32_t)NCH) {
      const uint32_t ch = channel(c);
#pragma unroll
      for (int t = 0; t < kMaxKc; ++t) {
        cst[q][t] = t < (int)Kc ? a.conv_state[(size_t)ch * Kc + t] : 0.f;
        cw[q][t] = t < (int)Kc ? bf16f(a.conv_w[(size_t)ch * Kc + t]) : 0.f;
      }
    }
  }
  const float alog = a.a_log[h], dtb = bf16f(a.dt_bias[h]);

  pdl_wait();
  pdl_launch();

  // ---- causal conv update + SiLU; conv state written back once per channel
  const bool own_qk = (h % grp) == 0 && j == 0;
#pragma unroll
  for (int q = 0; q < CPT; ++q) {
    const uint32_t c = threadIdx.x + q * kGdnThreads;
    if (c < (uint32_t)NCH) {
      const uint32_t ch = channel(c);
      const float x = bf16f(a.qkv[ch]);
      float o = 0.f;
#pragma unroll
      for (int t = 0; t < kMaxKc; ++t) {
        if (t < (int)Kc) {
          const float sv = (t + 1 < (int)Kc) ? cst[q][t + 1] : x;  // shift left, newest last
          cst[q][t] = sv;
          o = fmaf(cw[q][t], sv, o);
        }
      }
      act[c] = siluf_(o);
      if (c >= 2 * DK) {
#pragma unroll
        for (int t = 0; t < kMaxKc; ++t)
          if (t < (int)Kc) a.conv_state[(size_t)ch * Kc + t] = cst[q][t];
      }
    }
  }
  // every CTA of the k-head has read the old q/k conv state: one of them writes it
  cooperative_groups::this_cluster().sync();
  if (own_qk) {
#pragma unroll
    for (int q = 0; q < CPT; ++q) {
      const uint32_t c = threadIdx.x + q * kGdnThreads;
      if (c < 2u * DK) {
        const uint32_t ch = channel(c);
#pragma unroll
        for (int t = 0; t < kMaxKc; ++t)
          if (t < (int)Kc) a.conv_state[(size_t)ch * Kc + t] = cst[q][t];
      }
    }
  }
  if (threadIdx.x == 0) {
    // gate = exp(softplus(dt + dt_bias) * -exp(A_log)); beta = sigmoid(b)
    const float x = bf16f(a.dt_raw[h]) + dtb;
    const float sp_ = x > 20.f ? x : log1pf(expf(x));
    stat[2] = expf(sp_ * -expf(alog));
    stat[3] = sigmoidf_(bf16f(a.b_raw[h]));
  }
  __syncthreads();

  // ---- per-head L2 norm of q and k (eps 1e-6), then bf16 like qkv_smooth
  {
    float sq = 0.f, sk = 0.f;
    for (uint32_t i = threadIdx.x; i < DK; i += kGdnThreads) {
      sq = fmaf(act[i], act[i], sq);
      sk = fmaf(act[DK + i], act[DK + i], sk);
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    if (lane == 0) {
      red[0][warp][0] = sq;
      red[1][warp][0] = sk;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float tq = 0.f, tk = 0.f;
      for (int w = 0; w < 8; ++w) {
        tq += red[0][w][0];
        tk += red[1][w][0];
      }
      stat[0] = rsqrtf(tq + a.l2_eps);
      stat[1] = rsqrtf(tk + a.l2_eps);
    }
    __syncthreads();
    const float iq = stat[0], ik = stat[1];
    for (uint32_t i = threadIdx.x; i < (uint32_t)NCH; i += kGdnThreads) {
      const float v = act[i];
      act[i] = round_bf16(i < DK ? v * iq : (i < 2 * DK ? v * ik : v));
    }
    __syncthreads();
  }

  // ---- delta rule on the slice: thread (warp, lane) holds rows warp*RPT + r of column lane
  const float g = stat[2], beta = stat[3];
  const float* qv = act;
  const float* kv = act + DK;
  float u = 0.f;
#pragma unroll
  for (int r = 0; r < RPT; ++r) {
    st[r] *= g;
    u = fmaf(st[r], kv[warp * RPT + r], u);
  }
  red[0][warp][lane] = u;
  __syncthreads();
  u = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) u += red[0][w][lane];
  const float delta = beta * (act[2 * DK + lane] - u);
  float y = 0.f;
#pragma unroll
  for (int r = 0; r < RPT; ++r) {
    st[r] = fmaf(kv[warp * RPT + r], delta, st[r]);
    y = fmaf(st[r], qv[warp * RPT + r], y);
  }
  red[1][warp][lane] = y;
#pragma unroll
  for (int r = 0; r < RPT; ++r) sp[(size_t)r * Dv] = st[r];
  __syncthreads();
  if (warp == 0) {
    y = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) y += red[1][w][lane];
    a.y[(size_t)h * Dv + v0 + lane] = to_bf16(y * a.out_scale);
  }
}

}  // namespace

cudaError_t gdn_launch(const GdnArgs& a, cudaStream_t stream, bool pdl) {
  if (a.Dv % kGdnCols || a.Kc == 0 || a.Kc > (uint32_t)kMaxKc || a.Hk == 0 || a.Hv % a.Hk ||
      (a.Hv / a.Hk) * (a.Dv / kGdnCols) > 8)
    return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.Hv / a.Hk;  // the v-heads of one k-head ...
  attr[0].val.clusterDim.y = a.Dv / kGdnCols;  // ... and all their column slices
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hv, a.Dv / kGdnCols);
  cfg.blockDim = dim3(kGdnThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  switch (a.Dk) {
    case 32: return cudaLaunchKernelEx(&cfg, gdn_kernel<32>, a);
    case 64: return cudaLaunchKernelEx(&cfg, gdn_kernel<64>, a);
    case 128: return cudaLaunchKernelEx(&cfg, gdn_kernel<128>, a);
  }
  return cudaErrorInvalidValue;
}

__global__ void advance_pos_kernel(int32_t* d_pos) {
  pdl_wait();
  pdl_launch();
  if (threadIdx.x == 0) *d_pos += 1;
}

cudaError_t advance_pos_launch(int32_t* d_pos, cudaStream_t stream, bool pdl) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, advance_pos_kernel, d_pos);
}

}  // namespace q35
