// Argument blocks and host-side launchers of the decode kernels (internal to the
// library; the public boundary is include/qwen35_decode.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace q35 {

// ------------------------------------------------------------ quantised GEMV

constexpr int kGemvConsumerWarps = 8;
constexpr int kGemvThreads = (kGemvConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kGemvMaxSegs = 4;
constexpr int kGemvCplMax = 5;      // 16-byte code chunks per lane and row
constexpr int kGemvMaxK = 12288;    // x in registers: at most 8 warps x 32 lanes x 5 chunks x 16
constexpr int kGemvSmemBudget = 96 * 1024;  // pipeline stages per CTA

// How the GEMV input vector x is formed from the preceding kernel's outputs.
enum GemvPrologue : int {
  kProPlain = 0,       // x = a (bf16)
  kProRmsNorm = 1,     // x = bf16(a * rsqrt(mean(a^2) + eps) * nw)
  kProAddRmsNorm = 2,  // r = bf16(a + b); x = bf16(r * rsqrt(mean(r^2) + eps) * nw); CTA 0 stores r
  kProSiluMul = 3,     // x = silu(a) * b (fp32, unrounded)
  kProHeadNormSilu = 4 // x = silu(b) * bf16(a * rsqrt(mean_head(a^2) + eps) * nw[k % head_dim])
};
enum GemvEpilogue : int {
  kEpiStore = 0,  // out = bf16(W x)
  kEpiResid = 1   // out = bf16(resid + W x)
};

struct GemvSeg {
  const uint8_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
  uint16_t* out;
  uint32_t rows;
  uint32_t row0;  // first row of this segment in the concatenated row space
};

struct GemvArgs {
  GemvSeg seg[kGemvMaxSegs];
  uint32_t nseg, total_rows;
  uint32_t K, gstride;     // input length; bf16 stride of a scale/bias row
  uint32_t W;              // warps per row (1, 2, 4 or 8)
  uint32_t cpl;            // code chunks per lane per row
  uint32_t nstage, stage_stride, stage_scale_off, stage_bias_off, bar_off;
  const uint16_t* a;       // prologue inputs (see GemvPrologue)
  const uint16_t* b;
  const uint16_t* nw;
  float eps;
  uint32_t head_dim;
  uint16_t* resid_out;
  const uint16_t* resid_in;
  int* status;
};

struct GemvPlan {
  GemvArgs args;
  int prologue, epilogue;
  uint32_t grid, smem;
};

// Fill stage geometry for K and the segment list; false if K is unsupported.
bool gemv_plan(GemvPlan& p, int num_sms);
cudaError_t gemv_launch(const GemvPlan& p, cudaStream_t stream, bool pdl);
cudaError_t gemv_set_attributes();

// Dequantise one matrix to fp32 (bit-exact check of the GEMV's indexing).
cudaError_t dequant_launch(const uint8_t* codes, const uint16_t* scales, const uint16_t* biases,
                           uint32_t n, uint32_t k, uint32_t gstride, float* out, cudaStream_t stream);

// ------------------------------------------------------------ full attention

constexpr int kAttnConsumerWarps = 8;
constexpr int kAttnThreads = (kAttnConsumerWarps + 1) * 32;
constexpr int kAttnMaxSplits = 512;
constexpr int kAttnMaxHalfRot = 128;
constexpr int kAttnSmemBudget = 96 * 1024;
constexpr int kAttnTile = 8;  // tokens per pipeline stage

struct AttnArgs {
  const uint16_t* q_full;  // [H][2D]: [Q_h | gate_h]
  const uint16_t* k_new;   // [Hkv][D] raw k_proj output
  const uint16_t* v_new;   // [Hkv][D]
  const uint16_t* q_norm;  // [D]
  const uint16_t* k_norm;  // [D]
  uint16_t* kc;            // [capacity][Hkv][D]
  uint16_t* vc;
  uint32_t capacity;
  uint32_t H, Hkv, D, R;
  float eps, scale_log2;   // rms eps; softmax scale * log2(e)
  uint32_t cache_pos, S;   // host position (d_pos == nullptr)
  const int32_t* d_pos;    // device position (seq_len = *d_pos + 1)
  uint32_t max_seq;        // bound of a device position
  uint32_t P;              // number of sequence splits (grid size)
  uint32_t TS, nstage, stage_stride, bar_off, q_off, fresh_off;
  float* part_o;           // [P][H][D] unnormalised outputs
  float* part_ml;          // [P][H][2] running max (log2 domain) and sum
  uint16_t* ga;            // combine output [H*D]: bf16(bf16(attn) * sigmoid(gate))
  int* status;
  float inv_freq[kAttnMaxHalfRot];
};

struct AttnPlan {
  AttnArgs args;
  uint32_t smem;
};
bool attn_plan(AttnPlan& p);
cudaError_t attn_launch(const AttnPlan& p, cudaStream_t stream, bool pdl);
cudaError_t attn_set_attributes();

// ------------------------------------------------------------ Gated DeltaNet

struct GdnArgs {
  const uint16_t* qkv;     // [C] raw in_proj_qkv output, channels [Q | K | V]
  const uint16_t* dt_raw;  // [Hv]
  const uint16_t* b_raw;   // [Hv]
  const float* a_log;      // [Hv]
  const uint16_t* dt_bias; // [Hv]
  const uint16_t* conv_w;  // [C][Kc]
  float* conv_state;       // [C][Kc]
  float* ssm;              // [Hv][Dk][Dv]
  uint16_t* y;             // [Hv*Dv]
  uint32_t Hk, Hv, Dk, Dv, Kc;
  float l2_eps, out_scale;
  int* status;
};
cudaError_t gdn_launch(const GdnArgs& a, cudaStream_t stream, bool pdl);

// ------------------------------------------------------------ misc

cudaError_t advance_pos_launch(int32_t* d_pos, cudaStream_t stream, bool pdl);

}  // namespace q35
