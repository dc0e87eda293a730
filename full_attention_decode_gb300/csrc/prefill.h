// Multi-token prefill of Qwen3.5 decoder layers: the launchers of prefill.cu,
// called by the C ABI (abi.cu). A prompt of T tokens runs layer by layer, each
// step over all T tokens at once: the projections as tensor-core GEMMs
// (tcgen05, int8 group-64 weights dequantised to bf16 in shared memory), the
// causal attention over the prompt and the cache, and the Gated DeltaNet
// recurrence token after token with each state block held on chip for the whole
// prompt. Token t computes what the single-token forward computes for it after
// tokens 0 .. t-1.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace q35pf {

// Y[t][n] = bf16(sum_k X[t][k] W[n][k] (+ R[t][n])) for t < T, n < N, with
// w = scales[n][k/64] * codes[n][k] + biases[n][k/64] taken as W = bf16(w) + bf16(w -
// bf16(w)) (w to 2^-16 relative) when exact, else as W = bf16(w).
// X bf16 [T][ldx] (ldx % 8 == 0), Y and R bf16 [T][ldy]; K % 64 == 0.
struct Gemm {
  const uint16_t* X;
  const uint8_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
  uint16_t* Y;
  const uint16_t* R;  // residual added in the epilogue, or null
  uint32_t ldx, ldy, gstride, N, K, T;
  int* status;
  unsigned long long wait_ns;
  bool exact;
  float* ws;  // split-K partial sums (kGemmWorkspace bytes), or null: no split
};
// Workspace for a GEMM whose tiles leave SMs idle: K is split so that tiles x
// splits fill the GPU, each split's fp32 partial sums land here and a second
// kernel adds them in split order (deterministic). splits x T x N <= 152 x 128 x
// 256, so the bound does not depend on the shape.
constexpr size_t kGemmWorkspace = (size_t)152 * 128 * 256 * 4;
cudaError_t gemm(const Gemm& g, cudaStream_t st);

// out[t] = bf16(RMSNorm(v[t]) * w) over E values, v = a (b null) or
// v = bf16(a + b), which is also stored in resid (when not null).
cudaError_t rmsnorm(const uint16_t* a, const uint16_t* b, uint16_t* resid, const uint16_t* w, uint16_t* out,
                    uint32_t T, uint32_t E, float eps, cudaStream_t st);

// h[i] = bf16(SiLU(g[i]) * u[i]), i < n.
cudaError_t silu_mul(const uint16_t* g, const uint16_t* u, uint16_t* h, size_t n, cudaStream_t st);

// Full attention: per token t (position p0 + t) the per-head q/k RMSNorm, RoPE on
// the first R dims, the KV append at row p0 + t, then the causal attention of every
// q-head over rows [0, p0 + t] gated by sigmoid(gate).
struct Attn {
  const uint16_t* qf;  // q_proj outputs [T][H][2D] ([Q_h | gate_h])
  const uint16_t* k;   // k_proj outputs [T][Hkv*D]
  const uint16_t* v;   // v_proj outputs [T][Hkv*D]
  const uint16_t *q_norm, *k_norm;
  uint16_t* qr;        // roped q [T][H][D] (written)
  uint16_t *kc, *vc;   // bf16 caches [capacity][Hkv][D], or pools of 2^bt_shift-row blocks;
                       // Turbo8: E4M3 codes, u8 [capacity][Hkv][D]
  uint16_t *ks, *vs;   // Turbo8: bf16 scales [capacity][sstride], one per 16 elements
  const int32_t* btab; // paged: logical token t in row t % 2^bt_shift of block btab[t >> bt_shift]
  uint16_t* ga;        // gated attention [T][H*D] (written)
  uint32_t T, p0, H, Hkv, D, R, bt_shift;
  uint32_t turbo8, sstride;  // Turbo8 cache (rows rotated by the normalised WHT, quantised)
  float eps;
  float inv_freq[128];
};
cudaError_t attention(const Attn& a, cudaStream_t st);

// Gated DeltaNet: the conv1d update of every channel over the T tokens (state
// advanced), SiLU, per-head L2 norm on the Q/K channels, the decay gate and beta,
// the delta-rule recurrence of every state block over the T tokens, then the
// per-head output RMSNorm gated by SiLU(z).
struct Gdn {
  const uint16_t* qkv;     // in_proj_qkv outputs [T][C]
  const uint16_t* z;       // in_proj_z outputs [T][Z]
  const uint16_t* dt_raw;  // in_proj_a outputs [T][Hv]
  const uint16_t* b_raw;   // in_proj_b outputs [T][Hv]
  const uint16_t* conv_w;  // [C][Kc]
  const float* a_log;      // [Hv]
  const uint16_t* dt_bias; // [Hv]
  const uint16_t* norm_w;  // [Dv]
  float* conv_state;       // [C][Kc]
  float* ssm;              // [Hv][Dv/32][Dk][32]
  uint16_t* qs;            // qkv_smooth [T][C] (written)
  float* act;              // conv outputs after SiLU [T][C] (work buffer)
  float* gb;               // gate, beta [T][Hv][2] (written)
  uint16_t* y;             // readout [T][Z] (written)
  uint16_t* yin;           // out_proj input SiLU(z) * y_norm [T][Z] (written)
  uint32_t T, Hk, Hv, Dk, Dv, Kc, C;
  float eps;
};
cudaError_t gdn(const Gdn& g, cudaStream_t st);

}  // namespace q35pf
