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
// KV formats (qwen35_kv_dtype): bf16 rows, or Turbo8 (E4M3 codes + bf16 scales per
// 16, rotated basis).
enum KvDtype : uint32_t { kKvBf16 = 0, kKvTurbo8 = 1 };

struct LayerDesc {
  int32_t kind;
  uint32_t capacity;  // KV rows (full attention)
  QMat m[8];
  const uint16_t *input_ln, *post_ln, *q_norm, *k_norm, *norm_weight, *dt_bias, *conv_w;
  const float* a_log;
  uint8_t *kc, *vc;     // bf16 rows or Turbo8 codes (paged: the block pools)
  uint16_t *ks, *vs;    // Turbo8 scales [capacity][sstride]
  uint32_t kv_dtype, pad;
  // paged KV: token t in row t & (2^bt_shift - 1) of pool block btab[t >> bt_shift];
  // null: contiguous rows
  const int32_t* btab;
  uint32_t bt_shift, pad2;
  float *conv_state, *ssm;
};

// Byte offsets of the intermediates inside the scratch buffer (from the start of
// a sequence's block). The ones other CTAs read are tagged words: one 32-bit word
// per element, the bf16 value in the high half and, in the low half, the tag of
// the phase that wrote it (the launch's phase index + 1); the launch starts with
// these words zeroed (tag 0: not written yet). They sit first in the block,
// [tag_begin, tag_end); the attention partials (fp32, released by a per-split
// flag word, also tagged) and the debug stage dumps (plain bf16) follow.
struct ScratchMap {
  uint32_t q_full, k, v, ga, o, flags;        // full attention (tagged)
  uint32_t dt_raw, b_raw, qkv, z, y, out;     // linear attention (tagged)
  uint32_t x_resid, g, u, xa;                 // both (tagged); xa: a layer's output inside a stack
  // a single sequence's SiLU(gate) * up, formed by the gate|up phase and quantised
  // as the down projection's input (tagged): 16-bit codes [I], chunk exponents [I/16]
  uint32_t hq, he;
  uint32_t tag_begin, tag_end;
  uint32_t part_o, part_ml;                   // split-KV partials (fp32)
  uint32_t x_norm, x_norm2, qkv_smooth, y_norm;  // debug stage dumps (bf16)
  uint32_t k_rot, v_rot;                         // debug: a Turbo8 layer's rotated new k, v (bf16)
};

// The split of a GEMV phase's work that depends only on its shape (the layer kind
// and phase), computed once per launch on the host: K-parts per row W, chunks per
// lane cpl, rows per tile R, a batch's sequences per pass bs and passes npass. It
// travels in the program header, which every CTA keeps in shared memory.
struct GemvShape {
  uint8_t W, cpl, R, bs, npass, pad[3];
};
constexpr int kShapeKinds = 4, kShapePhases = 6;

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
  // bounded waits give up after wait_ns; wait_probe (debug) is a word that thread
  // 0 of every CTA waits on at the start (bounded) until it is nonzero
  unsigned long long wait_ns;
  const uint32_t* wait_probe;
  uint32_t dump;  // debug: the fused steps also store x_norm, x_norm2, qkv_smooth, y_norm
  // position: host values, or d_pos[b] (seq_len = d_pos[b] + 1) bounded by max_seq
  uint32_t pos, S, max_seq, P;
  const int32_t* d_pos;
  int32_t* advance;  // advance[b] incremented by one after the last layer, or null
  // batch: sequence b's intermediates at scratch + b * seq_stride, vectors at
  // x_in/x_out + b * E, caches at the layer's pointers + b * (one sequence's size)
  uint32_t batch, seq_stride;
  float inv_freq[128];
  // optional phase timeline: trace[(cta * trace_phases + phase) * kTraceSlots + k],
  // k = 0 previous phase done, 1 phase entered, 2 phase end, 3 GEMV input formed,
  // 4 first tile in shared memory, 5 last tile in shared memory, 6 rows done
  // (globaltimer ns, thread 0), 7 first tile issued (the producer), 8 input loads
  // landed, 9 input stored, 10 row loop entered, 11 tile loop entered, 12 rows
  // reduced, 13 the previous phase done in every warp, 14 the phase's descriptions
  // formed, 15 the GEMV input loads issued; null = off
  unsigned long long* trace;
  uint32_t trace_phases;
  // shared memory split of this launch: the tile ring's bytes and the per-phase
  // buffer's (ring_bytes + union_bytes + kDecFixed = kDecSmem)
  uint32_t ring_bytes, union_bytes;
  // GEMV shapes by [layer kind][phase], filled by decode_pick_split
  GemvShape shapes[kShapeKinds][kShapePhases];
  LayerDesc layers[kMaxLayers];
};

// Launch geometry and attributes.
constexpr int kDecConsumerWarps = 12;
// consumers, then the producer warp, then the helper warp
constexpr int kDecThreads = (kDecConsumerWarps + 2) * 32;
// The tile ring: tiles of any size up to kDecTileMax sit at increasing offsets of
// one circular buffer, at most kDecSlots in flight (one full/empty barrier pair
// and one offset word per slot).
// Two splits of the same dynamic shared memory between the ring and the per-phase
// buffer (x chunks + partial sums / attention / GDN work area): a batch's
// tensor-core passes stage several sequences' inputs in a 90 KiB buffer beside a
// 130 KiB ring (at 4B dims 8, 8 and 4 sequences per pass at K = 2560, 4096, 9216;
// fewer passes over the down projection measured faster than a larger ring); a
// single sequence needs at most about 28 KiB there and takes the larger ring (six
// 4B-shape 12-row tiles of 2560 columns, ten 2-row tiles of 9216).
constexpr int kDecRing = 133120;    // 130 KiB
constexpr int kDecTileMax = 45056;  // 44 KiB
constexpr int kDecSlots = 16;
constexpr int kDecUnion = 92160;
constexpr int kDecFixed = 2 * kDecSlots * 8 + 16 + 2 * kDecSlots * 4 + 1024;  // barriers, slot words, misc
constexpr int kDecSmem = kDecRing + kDecFixed + kDecUnion;
constexpr int kDecRingLarge = 195840;
constexpr int kDecUnionSmall = kDecSmem - kDecFixed - kDecRingLarge;

// The decode kernel for a program's dims: attention head dim (one function per
// supported D, each in its own translation unit), q-heads per attention warp, GDN
// key head dim, batched or not; nullptr for an unsupported combination.
using DecodeKernel = void (*)(Program);
DecodeKernel decode_kernel_d64(uint32_t hpw, uint32_t Dk, bool batched);
DecodeKernel decode_kernel_d128(uint32_t hpw, uint32_t Dk, bool batched);
DecodeKernel decode_kernel_d256(uint32_t hpw, uint32_t Dk, bool batched);

cudaError_t decode_set_attributes();
// Dequantise one matrix to fp32 [n][k]: fmaf(scale, code, bias), one rounding.
cudaError_t dequant_launch(const uint8_t* codes, const uint16_t* scales, const uint16_t* biases,
                           uint32_t n, uint32_t k, uint32_t gstride, float* out, cudaStream_t stream);
// Index of the largest of n bf16 values (the lowest index among equal ones) into
// *out: one block of 1024 threads.
cudaError_t argmax_bf16_launch(const uint16_t* v, uint32_t n, int32_t* out, cudaStream_t stream);
// Zeroes the tagged words of every sequence's block, then launches the program
// (cooperative, one CTA per SM).
cudaError_t decode_launch(const Program& p, int num_sms, cudaStream_t stream);
// Host check of the dims the kernel supports on a grid of num_sms CTAs; false if
// unsupported.
bool decode_dims_ok(const Program& p, bool has_fa, bool has_gdn, int num_sms);
// Picks the launch's shared-memory split (the larger ring when every phase fits the
// smaller buffer), checks the dims and fills the GEMV shapes; false if unsupported.
bool decode_pick_split(Program& p, bool has_fa, bool has_gdn, int num_sms);

}  // namespace q35
