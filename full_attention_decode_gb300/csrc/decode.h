// The persistent decode kernel: one launch runs a program of layers (one layer
// for the per-layer forwards, the whole stack for a decode step).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace q35 {

constexpr int kMaxLayers = 64;
constexpr int kMaxBatch = 8;  // sequences decoded together (their own caches, shared weights)
constexpr int kTraceSlots = 16;  // timeline entries per CTA and phase
constexpr int kDecMaxSplits = 512;  // split-KV partials the scratch holds

// One quantised matrix: codes [n][k] u8, scales/biases [n][gstride] bf16.
struct QMat {
  const uint8_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
  uint32_t n, pad;
};

// kLayerGemv: a single GEMV phase, x_out = bf16(m[0] x_in) (the component entry point).
// kLayerHead: the output head's GEMV, x_out = bf16(m[0] bf16(RMSNorm(x_in) * input_ln))
// (input_ln holds the final norm's weights; x_out receives the logits).
enum LayerKind : int32_t { kLayerFA = 0, kLayerGDN = 1, kLayerGemv = 2, kLayerHead = 3 };

// Matrix slots of a layer.
//   full attention:   0 q_proj, 1 k_proj, 2 v_proj, 3 o_proj, 4 gate, 5 up, 6 down
//   linear attention: 0 in_proj_a, 1 in_proj_b, 2 in_proj_qkv, 3 in_proj_z, 4 gate,
//                     5 up, 6 down, 7 out_proj
struct LayerDesc {
  int32_t kind;
  uint32_t capacity;  // KV rows (full attention)
  QMat m[8];
  const uint16_t *input_ln, *post_ln, *q_norm, *k_norm, *norm_weight, *dt_bias, *conv_w;
  const float* a_log;
  uint16_t *kc, *vc;
  float *conv_state, *ssm;
};

// Byte offsets of the intermediates inside the scratch buffer.
struct ScratchMap {
  uint32_t q_full, k, v, ga, o, part_o, part_ml;  // full attention
  uint32_t dt_raw, b_raw, qkv, z, y, out;         // linear attention
  uint32_t x_resid, g, u;                         // both
};

struct Program {
  // dims
  uint32_t E, I, H, Hkv, D, R, Hk, Hv, Dk, Dv, Kc, C, Z;
  float eps, scale_log2, gdn_out_scale, l2_eps;
  uint32_t n_layers;
  const uint16_t* x_in;
  uint16_t* x_out;
  uint8_t* scratch;
  ScratchMap sm;
  int* status;
  uint32_t* barrier;  // grid-barrier counter, zero at launch
  // position: host values, or d_pos[b] (seq_len = d_pos[b] + 1) bounded by max_seq
  uint32_t pos, S, max_seq, P;
  const int32_t* d_pos;
  int32_t* advance;  // advance[b] incremented by one after the last layer, or null
  // batch: sequence b's intermediates at scratch + b * seq_stride, vectors at
  // x_in/x_out + b * E, caches at the layer's pointers + b * (one sequence's size)
  uint32_t batch, seq_stride;
  float inv_freq[128];
  // optional phase timeline: trace[(cta * trace_phases + phase) * kTraceSlots + k],
  // k = 0 barrier arrival, 1 barrier release, 2 phase end, 3 GEMV input formed,
  // 4 first tile in shared memory, 5 last tile in shared memory, 6 rows done
  // (globaltimer ns, thread 0), 7 first tile issued (the producer), 8 input loads
  // landed, 9 input stored, 10 row loop entered, 11 tile loop entered, 12 rows
  // reduced; null = off
  unsigned long long* trace;
  uint32_t trace_phases;
  // shared memory split of this launch: the tile ring's bytes and the per-phase
  // buffer's (ring_bytes + union_bytes + kDecFixed = kDecSmem)
  uint32_t ring_bytes, union_bytes;
  LayerDesc layers[kMaxLayers];
};

// Launch geometry and attributes.
constexpr int kDecConsumerWarps = 12;
constexpr int kDecThreads = (kDecConsumerWarps + 1) * 32;
// The tile ring: tiles of any size up to kDecTileMax sit at increasing offsets of
// one circular buffer, at most kDecSlots in flight (one full/empty barrier pair
// and one offset word per slot).
// Two splits of the same dynamic shared memory between the ring and the per-phase
// buffer (x chunks + partial sums / attention / GDN work area): a batch's
// tensor-core passes stage several sequences' inputs in the larger buffer; a single
// sequence needs at most about 28 KiB there and takes the larger ring (six 4B-shape
// 12-row tiles of 2560 columns, ten 2-row tiles of 9216).
constexpr int kDecRing = 174080;    // 170 KiB
constexpr int kDecTileMax = 45056;  // 44 KiB
constexpr int kDecSlots = 16;
constexpr int kDecUnion = 53248;
constexpr int kDecFixed = 2 * kDecSlots * 8 + 16 + 2 * kDecSlots * 4 + 1024;  // barriers, slot words, misc
constexpr int kDecSmem = kDecRing + kDecFixed + kDecUnion;
constexpr int kDecRingLarge = 195840;
constexpr int kDecUnionSmall = kDecSmem - kDecFixed - kDecRingLarge;

cudaError_t decode_set_attributes();
// Dequantise one matrix to fp32 [n][k]: fmaf(scale, code, bias), one rounding.
cudaError_t dequant_launch(const uint8_t* codes, const uint16_t* scales, const uint16_t* biases,
                           uint32_t n, uint32_t k, uint32_t gstride, float* out, cudaStream_t stream);
// Index of the largest of n bf16 values (the lowest index among equal ones) into
// *out: one block of 1024 threads.
cudaError_t argmax_bf16_launch(const uint16_t* v, uint32_t n, int32_t* out, cudaStream_t stream);
// Zeroes the barrier counter, then launches the program (cooperative, one CTA per SM).
cudaError_t decode_launch(const Program& p, int num_sms, cudaStream_t stream);
// Host check of the dims the kernel supports on a grid of num_sms CTAs; false if
// unsupported.
bool decode_dims_ok(const Program& p, bool has_fa, bool has_gdn, int num_sms);
// Picks the launch's shared-memory split (the larger ring when every phase fits the
// smaller buffer), then checks the dims; false if unsupported.
bool decode_pick_split(Program& p, bool has_fa, bool has_gdn, int num_sms);

}  // namespace q35
