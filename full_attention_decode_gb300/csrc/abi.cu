// C ABI of the decode library (include/qwen35_decode.h): argument validation,
// scratch layout, and the kernel sequence of each layer kind.
//
// Full-attention layer ("full_attention.rs", forward_full_attention), 6 launches:
//   1 GEMV  [q_proj | k_proj | v_proj] with the input RMSNorm in its prologue
//   2 attention partials (q/k RMSNorm, RoPE, KV append, split-KV softmax)
//   3 combine + sigmoid(gate)
//   4 GEMV  o_proj
//   5 GEMV  [gate_proj | up_proj] with residual add + post RMSNorm in its prologue
//   6 GEMV  down_proj with silu(gate) * up in its prologue and the residual add
// Linear-attention layer ("linear_attention.rs", forward_linear_attention), 5:
//   1 GEMV  [in_proj_a | in_proj_b | in_proj_qkv | in_proj_z] + input RMSNorm
//   2 Gated DeltaNet step (conv1d + SiLU + L2 norm, gate, beta, delta rule)
//   3 GEMV  out_proj with per-head RMSNorm and silu(z) gating in its prologue
//   4, 5 as 5, 6 above.
// Every launch after the first of a call is a programmatic dependent launch, so
// each kernel's weight stream starts while its predecessor finishes.
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "../../include/qwen35_decode.h"
#include "kernels.h"

using namespace q35;

namespace {

constexpr int kMaxDevices = 64;
int g_num_sms[kMaxDevices] = {0};

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return g_num_sms[dev];
}

bool aligned16(const void* p) { return p && ((uintptr_t)p % 16) == 0; }
uint32_t gstride_of(uint32_t k) { return ((k / 64 + 7) / 8) * 8; }

struct Dims {
  uint32_t E, I, H, Hkv, D, R, Hk, Hv, Dk, Dv, Kc, C, Z;
};

int check_config(const qwen35_config* c, Dims& d) {
  if (!c) return QWEN35_ERR_INVALID_ARGUMENT;
  d.E = c->hidden; d.I = c->intermediate;
  d.H = c->num_heads; d.Hkv = c->num_kv_heads; d.D = c->head_dim; d.R = c->rotary_dim;
  d.Hk = c->num_k_heads_lin; d.Hv = c->num_v_heads_lin;
  d.Dk = c->k_head_dim_lin; d.Dv = c->v_head_dim_lin; d.Kc = c->conv_kernel_size;
  d.C = 2 * d.Hk * d.Dk + d.Hv * d.Dv;
  d.Z = d.Hv * d.Dv;
  if (c->group_size != 64) return QWEN35_ERR_INVALID_ARGUMENT;
  if (!(c->rms_eps >= 0.f) || !std::isfinite(c->rms_eps)) return QWEN35_ERR_INVALID_ARGUMENT;
  if (d.E == 0 || d.I == 0 || d.E % 64 || d.I % 64) return QWEN35_ERR_INVALID_ARGUMENT;
  if (d.E > (uint32_t)kGemvMaxK || d.I > (uint32_t)kGemvMaxK) return QWEN35_ERR_UNSUPPORTED;
  return QWEN35_OK;
}

int check_fa_dims(const qwen35_config* c, const Dims& d) {
  if (d.H == 0 || d.Hkv == 0 || d.H % d.Hkv) return QWEN35_ERR_INVALID_ARGUMENT;
  if (d.R % 2 || d.R > d.D || d.R == 0) return QWEN35_ERR_INVALID_ARGUMENT;
  if (d.D != 64 && d.D != 128 && d.D != 256) return QWEN35_ERR_UNSUPPORTED;
  if (d.Hkv > 8 || (d.H > 8 && d.H % 8) || (d.H > 8 && d.H / 8 > 4) ||
      (d.H > 8 && d.H / 8 > d.H / d.Hkv))
    return QWEN35_ERR_UNSUPPORTED;
  if (d.H * d.D > (uint32_t)kGemvMaxK) return QWEN35_ERR_UNSUPPORTED;
  if (!(c->rope_theta > 0.f)) return QWEN35_ERR_INVALID_ARGUMENT;
  return QWEN35_OK;
}

int check_gdn_dims(const Dims& d) {
  if (d.Hk == 0 || d.Hv == 0 || d.Hv % d.Hk) return QWEN35_ERR_INVALID_ARGUMENT;
  if ((d.Dk != 32 && d.Dk != 64 && d.Dk != 128) || (d.Dv != 32 && d.Dv != 64 && d.Dv != 128))
    return QWEN35_ERR_UNSUPPORTED;
  if (d.Kc == 0 || d.Kc > 8) return QWEN35_ERR_UNSUPPORTED;
  if ((d.Hv / d.Hk) * (d.Dv / 32) > 8) return QWEN35_ERR_UNSUPPORTED;  // one cluster per k-head
  if (d.Z > (uint32_t)kGemvMaxK || d.Z / d.Dv > 128) return QWEN35_ERR_UNSUPPORTED;
  return QWEN35_OK;
}

bool qw_ok(const qwen35_qweight& w, uint32_t n, uint32_t k) {
  return w.n == n && w.k == k && aligned16(w.codes) && aligned16(w.scales) && aligned16(w.biases);
}

// ---------------------------------------------------------------- scratch layout

struct Layout {
  size_t q_full, k, v, ga, o, part_o, part_ml;      // full attention
  size_t dt_raw, b_raw, qkv, z, y, out;             // linear attention
  size_t x_resid, g, u;                             // both (MLP)
  size_t total;
};

struct Bump {
  size_t off = 256;  // [0, 4): device status word
  size_t take(size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  }
};

Layout layout(const Dims& d, int kind) {
  Layout L = {};
  Bump b;
  L.x_resid = b.take(d.E * 2);
  L.g = b.take(d.I * 2);
  L.u = b.take(d.I * 2);
  if (kind == QWEN35_LAYER_FULL_ATTENTION) {
    L.q_full = b.take((size_t)2 * d.H * d.D * 2);
    L.k = b.take((size_t)d.Hkv * d.D * 2);
    L.v = b.take((size_t)d.Hkv * d.D * 2);
    L.ga = b.take((size_t)d.H * d.D * 2);
    L.o = b.take((size_t)d.E * 2);
    L.part_o = b.take((size_t)kAttnMaxSplits * d.H * d.D * 4);
    L.part_ml = b.take((size_t)kAttnMaxSplits * d.H * 2 * 4);
  } else {
    L.dt_raw = b.take(d.Hv * 2);
    L.b_raw = b.take(d.Hv * 2);
    L.qkv = b.take((size_t)d.C * 2);
    L.z = b.take((size_t)d.Z * 2);
    L.y = b.take((size_t)d.Z * 2);
    L.out = b.take((size_t)d.E * 2);
  }
  L.total = b.off;
  return L;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(base) + off);
}

GemvSeg seg_of(const qwen35_qweight& w, uint16_t* out) {
  GemvSeg s = {};
  s.codes = w.codes;
  s.scales = w.scales;
  s.biases = w.biases;
  s.out = out;
  s.rows = w.n;
  return s;
}

int launch_gemv(GemvPlan& p, cudaStream_t st, bool pdl) {
  if (!gemv_plan(p, num_sms())) return QWEN35_ERR_UNSUPPORTED;
  return gemv_launch(p, st, pdl) == cudaSuccess ? QWEN35_OK : QWEN35_ERR_CUDA;
}

// MLP tail shared by both layer kinds: [gate | up] with residual + post norm, then down.
int mlp(const Dims& d, float eps, const uint16_t* post_ln, const qwen35_qweight& gate_w,
        const qwen35_qweight& up_w, const qwen35_qweight& down_w, const uint16_t* x_in, const uint16_t* delta,
        const Layout& L, void* scratch, uint16_t* x_out, cudaStream_t st) {
  int* status = at<int>(scratch, 0);
  GemvPlan p = {};
  p.prologue = kProAddRmsNorm;
  p.epilogue = kEpiStore;
  p.args.nseg = 2;
  p.args.seg[0] = seg_of(gate_w, at<uint16_t>(scratch, L.g));
  p.args.seg[1] = seg_of(up_w, at<uint16_t>(scratch, L.u));
  p.args.K = d.E;
  p.args.a = x_in;
  p.args.b = delta;
  p.args.nw = post_ln;
  p.args.eps = eps;
  p.args.resid_out = at<uint16_t>(scratch, L.x_resid);
  p.args.status = status;
  int r = launch_gemv(p, st, true);
  if (r) return r;
  GemvPlan q = {};
  q.prologue = kProSiluMul;
  q.epilogue = kEpiResid;
  q.args.nseg = 1;
  q.args.seg[0] = seg_of(down_w, x_out);
  q.args.K = d.I;
  q.args.a = at<uint16_t>(scratch, L.g);
  q.args.b = at<uint16_t>(scratch, L.u);
  q.args.resid_in = at<uint16_t>(scratch, L.x_resid);
  q.args.status = status;
  return launch_gemv(q, st, true);
}

int check_fa_layer(const qwen35_fa_layer* l, const Dims& d) {
  if (!l) return QWEN35_ERR_INVALID_ARGUMENT;
  if (!aligned16(l->input_ln) || !aligned16(l->q_norm) || !aligned16(l->k_norm) || !aligned16(l->post_ln))
    return QWEN35_ERR_INVALID_ARGUMENT;
  const uint32_t HD = d.H * d.D, KV = d.Hkv * d.D;
  if (!qw_ok(l->q_proj, 2 * HD, d.E) || !qw_ok(l->k_proj, KV, d.E) || !qw_ok(l->v_proj, KV, d.E) ||
      !qw_ok(l->o_proj, d.E, HD) || !qw_ok(l->gate_proj, d.I, d.E) || !qw_ok(l->up_proj, d.I, d.E) ||
      !qw_ok(l->down_proj, d.E, d.I))
    return QWEN35_ERR_INVALID_ARGUMENT;
  return QWEN35_OK;
}

int check_gdn_layer(const qwen35_gdn_layer* l, const Dims& d) {
  if (!l) return QWEN35_ERR_INVALID_ARGUMENT;
  if (!aligned16(l->input_ln) || !aligned16(l->post_ln) || !aligned16(l->norm_weight) || !l->a_log ||
      !l->dt_bias || !l->conv1d_weight || ((uintptr_t)l->a_log % 4) || ((uintptr_t)l->dt_bias % 2) ||
      ((uintptr_t)l->conv1d_weight % 2))
    return QWEN35_ERR_INVALID_ARGUMENT;
  if (!qw_ok(l->in_proj_a, d.Hv, d.E) || !qw_ok(l->in_proj_b, d.Hv, d.E) ||
      !qw_ok(l->in_proj_qkv, d.C, d.E) || !qw_ok(l->in_proj_z, d.Z, d.E) || !qw_ok(l->out_proj, d.E, d.Z) ||
      !qw_ok(l->gate_proj, d.I, d.E) || !qw_ok(l->up_proj, d.I, d.E) || !qw_ok(l->down_proj, d.E, d.I))
    return QWEN35_ERR_INVALID_ARGUMENT;
  return QWEN35_OK;
}

// The full-attention sequence; d_pos == nullptr selects the host position.
int fa_forward(const qwen35_config* cfg, const qwen35_fa_layer* layer, void* scratch, size_t scratch_bytes,
               const qwen35_kv_cache* kv, const uint16_t* x_in, uint16_t* x_out, uint32_t cache_pos,
               uint32_t seq_len, const int32_t* d_pos, uint32_t max_seq, cudaStream_t st) {
  Dims d;
  int r = check_config(cfg, d);
  if (r) return r;
  if ((r = check_fa_dims(cfg, d))) return r;
  if ((r = check_fa_layer(layer, d))) return r;
  if (!kv || !aligned16(kv->k) || !aligned16(kv->v) || kv->capacity == 0) return QWEN35_ERR_INVALID_ARGUMENT;
  if (!aligned16(x_in) || !aligned16(x_out) || !aligned16(scratch)) return QWEN35_ERR_INVALID_ARGUMENT;
  const Layout L = layout(d, QWEN35_LAYER_FULL_ATTENTION);
  if (scratch_bytes < L.total) return QWEN35_ERR_INVALID_ARGUMENT;
  if (d_pos) {
    if (max_seq == 0) return QWEN35_ERR_INVALID_ARGUMENT;
  } else if (cache_pos >= kv->capacity || seq_len == 0 || seq_len > cache_pos + 1) {
    return QWEN35_ERR_OUT_OF_RANGE;
  }
  if (num_sms() <= 0) return QWEN35_ERR_CUDA;
  int* status = at<int>(scratch, 0);

  GemvPlan p = {};
  p.prologue = kProRmsNorm;
  p.epilogue = kEpiStore;
  p.args.nseg = 3;
  p.args.seg[0] = seg_of(layer->q_proj, at<uint16_t>(scratch, L.q_full));
  p.args.seg[1] = seg_of(layer->k_proj, at<uint16_t>(scratch, L.k));
  p.args.seg[2] = seg_of(layer->v_proj, at<uint16_t>(scratch, L.v));
  p.args.K = d.E;
  p.args.a = x_in;
  p.args.nw = layer->input_ln;
  p.args.eps = cfg->rms_eps;
  p.args.status = status;
  if ((r = launch_gemv(p, st, true))) return r;

  AttnPlan ap = {};
  AttnArgs& a = ap.args;
  a.q_full = at<uint16_t>(scratch, L.q_full);
  a.k_new = at<uint16_t>(scratch, L.k);
  a.v_new = at<uint16_t>(scratch, L.v);
  a.q_norm = layer->q_norm;
  a.k_norm = layer->k_norm;
  a.kc = kv->k;
  a.vc = kv->v;
  a.capacity = kv->capacity;
  a.H = d.H; a.Hkv = d.Hkv; a.D = d.D; a.R = d.R;
  a.eps = cfg->rms_eps;
  a.scale_log2 = (float)(1.0 / std::sqrt((double)d.D) * 1.4426950408889634);
  a.cache_pos = cache_pos;
  a.S = seq_len;
  a.d_pos = d_pos;
  a.max_seq = max_seq;
  const uint32_t span = d_pos ? max_seq : seq_len;
  uint32_t P = (span + 31) / 32;
  if (P > (uint32_t)num_sms()) P = num_sms();
  if (P > (uint32_t)kAttnMaxSplits) P = kAttnMaxSplits;
  if (P == 0) P = 1;
  a.P = P;
  a.part_o = at<float>(scratch, L.part_o);
  a.part_ml = at<float>(scratch, L.part_ml);
  a.ga = at<uint16_t>(scratch, L.ga);
  a.status = status;
  // inv_freq[i] = theta^(-2i/R), computed in double and kept as fp32
  for (uint32_t i = 0; i < d.R / 2; ++i)
    a.inv_freq[i] = (float)std::pow((double)cfg->rope_theta, -2.0 * (double)i / (double)d.R);
  if (!attn_plan(ap)) return QWEN35_ERR_UNSUPPORTED;
  if (attn_launch(ap, st, true) != cudaSuccess) return QWEN35_ERR_CUDA;

  GemvPlan o = {};
  o.prologue = kProPlain;
  o.epilogue = kEpiStore;
  o.args.nseg = 1;
  o.args.seg[0] = seg_of(layer->o_proj, at<uint16_t>(scratch, L.o));
  o.args.K = d.H * d.D;
  o.args.a = at<uint16_t>(scratch, L.ga);
  o.args.status = status;
  if ((r = launch_gemv(o, st, true))) return r;

  return mlp(d, cfg->rms_eps, layer->post_ln, layer->gate_proj, layer->up_proj, layer->down_proj, x_in,
             at<uint16_t>(scratch, L.o), L, scratch, x_out, st);
}

int gdn_forward(const qwen35_config* cfg, const qwen35_gdn_layer* layer, void* scratch, size_t scratch_bytes,
                const qwen35_gdn_state* state, const uint16_t* x_in, uint16_t* x_out, cudaStream_t st) {
  Dims d;
  int r = check_config(cfg, d);
  if (r) return r;
  if ((r = check_gdn_dims(d))) return r;
  if ((r = check_gdn_layer(layer, d))) return r;
  if (!state || !aligned16(state->conv_state) || !aligned16(state->gdn_state)) return QWEN35_ERR_INVALID_ARGUMENT;
  if (!aligned16(x_in) || !aligned16(x_out) || !aligned16(scratch)) return QWEN35_ERR_INVALID_ARGUMENT;
  const Layout L = layout(d, QWEN35_LAYER_LINEAR_ATTENTION);
  if (scratch_bytes < L.total) return QWEN35_ERR_INVALID_ARGUMENT;
  if (num_sms() <= 0) return QWEN35_ERR_CUDA;
  int* status = at<int>(scratch, 0);

  GemvPlan p = {};
  p.prologue = kProRmsNorm;
  p.epilogue = kEpiStore;
  p.args.nseg = 4;
  p.args.seg[0] = seg_of(layer->in_proj_a, at<uint16_t>(scratch, L.dt_raw));
  p.args.seg[1] = seg_of(layer->in_proj_b, at<uint16_t>(scratch, L.b_raw));
  p.args.seg[2] = seg_of(layer->in_proj_qkv, at<uint16_t>(scratch, L.qkv));
  p.args.seg[3] = seg_of(layer->in_proj_z, at<uint16_t>(scratch, L.z));
  p.args.K = d.E;
  p.args.a = x_in;
  p.args.nw = layer->input_ln;
  p.args.eps = cfg->rms_eps;
  p.args.status = status;
  if ((r = launch_gemv(p, st, true))) return r;

  GdnArgs g = {};
  g.qkv = at<uint16_t>(scratch, L.qkv);
  g.dt_raw = at<uint16_t>(scratch, L.dt_raw);
  g.b_raw = at<uint16_t>(scratch, L.b_raw);
  g.a_log = layer->a_log;
  g.dt_bias = layer->dt_bias;
  g.conv_w = layer->conv1d_weight;
  g.conv_state = state->conv_state;
  g.ssm = state->gdn_state;
  g.y = at<uint16_t>(scratch, L.y);
  g.Hk = d.Hk; g.Hv = d.Hv; g.Dk = d.Dk; g.Dv = d.Dv; g.Kc = d.Kc;
  g.l2_eps = 1e-6f;
  g.out_scale = (float)(1.0 / std::sqrt((double)d.Dk));
  g.status = status;
  if (gdn_launch(g, st, true) != cudaSuccess) return QWEN35_ERR_CUDA;

  GemvPlan o = {};
  o.prologue = kProHeadNormSilu;
  o.epilogue = kEpiStore;
  o.args.nseg = 1;
  o.args.seg[0] = seg_of(layer->out_proj, at<uint16_t>(scratch, L.out));
  o.args.K = d.Z;
  o.args.a = at<uint16_t>(scratch, L.y);
  o.args.b = at<uint16_t>(scratch, L.z);
  o.args.nw = layer->norm_weight;
  o.args.eps = cfg->rms_eps;
  o.args.head_dim = d.Dv;
  o.args.status = status;
  if ((r = launch_gemv(o, st, true))) return r;

  return mlp(d, cfg->rms_eps, layer->post_ln, layer->gate_proj, layer->up_proj, layer->down_proj, x_in,
             at<uint16_t>(scratch, L.out), L, scratch, x_out, st);
}

}  // namespace

// Scratch of qwen35_forward_linear_attention_static: one array per device that
// loads the library. Host code must not use the symbol as an address; the device
// address is looked up per device and cached below.
static __device__ __align__(256) uint8_t g_static_scratch[QWEN35_STATIC_SCRATCH_BYTES];
static void* g_static_scratch_ptr[kMaxDevices] = {nullptr};

extern "C" {

int qwen35_init(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QWEN35_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return QWEN35_ERR_CUDA;
  if (major != 10 || minor != 3) return QWEN35_ERR_CUDA;  // built for sm_103a only
  if (gemv_set_attributes() != cudaSuccess || attn_set_attributes() != cudaSuccess) return QWEN35_ERR_CUDA;
  g_num_sms[dev] = sms;
  return QWEN35_OK;
}

const char* qwen35_status_string(int s) {
  switch (s) {
    case QWEN35_OK: return "ok";
    case QWEN35_ERR_INVALID_ARGUMENT: return "invalid argument";
    case QWEN35_ERR_OUT_OF_RANGE: return "position out of range";
    case QWEN35_ERR_UNSUPPORTED: return "unsupported dimensions";
    case QWEN35_ERR_CUDA: return "CUDA error";
    case QWEN35_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case QWEN35_ERR_DEVICE_RANGE: return "device position out of range";
  }
  return "unknown status";
}

size_t qwen35_scratch_bytes(const qwen35_config* cfg, int kind) {
  Dims d;
  if (check_config(cfg, d)) return 0;
  if (kind == QWEN35_LAYER_FULL_ATTENTION) {
    if (check_fa_dims(cfg, d)) return 0;
  } else if (kind == QWEN35_LAYER_LINEAR_ATTENTION) {
    if (check_gdn_dims(d)) return 0;
  } else {
    return 0;
  }
  return layout(d, kind).total;
}

size_t qwen35_stack_scratch_bytes(const qwen35_config* cfg) {
  const size_t a = qwen35_scratch_bytes(cfg, QWEN35_LAYER_FULL_ATTENTION);
  const size_t b = qwen35_scratch_bytes(cfg, QWEN35_LAYER_LINEAR_ATTENTION);
  if (a == 0 || b == 0) return 0;
  return a > b ? a : b;
}

int qwen35_scratch_init(void* scratch, size_t scratch_bytes, void* stream) {
  if (!aligned16(scratch) || scratch_bytes < 256) return QWEN35_ERR_INVALID_ARGUMENT;
  return cudaMemsetAsync(scratch, 0, 256, (cudaStream_t)stream) == cudaSuccess ? QWEN35_OK : QWEN35_ERR_CUDA;
}

int qwen35_read_device_status(const void* scratch, int32_t* host_status, void* stream) {
  if (!aligned16(scratch) || !host_status) return QWEN35_ERR_INVALID_ARGUMENT;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return QWEN35_ERR_CUDA;
  return cudaMemcpy(host_status, scratch, 4, cudaMemcpyDeviceToHost) == cudaSuccess ? QWEN35_OK
                                                                                     : QWEN35_ERR_CUDA;
}

int qwen35_forward_full_attention(const qwen35_config* cfg, const qwen35_fa_layer* layer, void* scratch,
                                  size_t scratch_bytes, const qwen35_kv_cache* kv, const qwen35_bf16* x_in,
                                  qwen35_bf16* x_out, uint32_t cache_pos, uint32_t seq_len_attn, void* stream) {
  return fa_forward(cfg, layer, scratch, scratch_bytes, kv, x_in, x_out, cache_pos, seq_len_attn, nullptr, 0,
                    (cudaStream_t)stream);
}

int qwen35_forward_full_attention_dpos(const qwen35_config* cfg, const qwen35_fa_layer* layer, void* scratch,
                                       size_t scratch_bytes, const qwen35_kv_cache* kv,
                                       const qwen35_bf16* x_in, qwen35_bf16* x_out, const int32_t* d_cache_pos,
                                       uint32_t max_seq_len, void* stream) {
  if (!d_cache_pos || ((uintptr_t)d_cache_pos % 4)) return QWEN35_ERR_INVALID_ARGUMENT;
  return fa_forward(cfg, layer, scratch, scratch_bytes, kv, x_in, x_out, 0, 0, d_cache_pos, max_seq_len,
                    (cudaStream_t)stream);
}

int qwen35_forward_linear_attention(const qwen35_config* cfg, const qwen35_gdn_layer* layer, void* scratch,
                                    size_t scratch_bytes, const qwen35_gdn_state* state, const qwen35_bf16* x_in,
                                    qwen35_bf16* x_out, void* stream) {
  return gdn_forward(cfg, layer, scratch, scratch_bytes, state, x_in, x_out, (cudaStream_t)stream);
}

int qwen35_forward_linear_attention_static(const qwen35_config* cfg, const qwen35_gdn_layer* layer,
                                           const qwen35_gdn_state* state, const qwen35_bf16* x_in,
                                           qwen35_bf16* x_out, void* stream) {
  const size_t need = qwen35_scratch_bytes(cfg, QWEN35_LAYER_LINEAR_ATTENTION);
  if (need == 0) return QWEN35_ERR_INVALID_ARGUMENT;
  if (need > QWEN35_STATIC_SCRATCH_BYTES) return QWEN35_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QWEN35_ERR_CUDA;
  if (!g_static_scratch_ptr[dev]) {  // once per device, with that device current
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return QWEN35_ERR_CUDA;
    g_static_scratch_ptr[dev] = p;
  }
  void* scratch = g_static_scratch_ptr[dev];
  cudaStream_t st = (cudaStream_t)stream;
  // the array keeps the previous call's contents: the status word must start at zero
  if (cudaMemsetAsync(scratch, 0, 256, st) != cudaSuccess) return QWEN35_ERR_CUDA;
  return gdn_forward(cfg, layer, scratch, QWEN35_STATIC_SCRATCH_BYTES, state, x_in, x_out, st);
}

int qwen35_decode_step(const qwen35_config* cfg, const qwen35_layer* layers, uint32_t num_layers, void* scratch,
                       size_t scratch_bytes, const qwen35_bf16* x_in, qwen35_bf16* x_out, int32_t* d_cache_pos,
                       uint32_t max_seq_len, void* stream) {
  if (!layers || num_layers == 0 || !d_cache_pos || ((uintptr_t)d_cache_pos % 4)) return QWEN35_ERR_INVALID_ARGUMENT;
  for (uint32_t i = 0; i < num_layers; ++i) {
    const qwen35_layer& l = layers[i];
    if (l.kind == QWEN35_LAYER_FULL_ATTENTION) {
      if (!l.fa || !l.kv) return QWEN35_ERR_INVALID_ARGUMENT;
    } else if (l.kind == QWEN35_LAYER_LINEAR_ATTENTION) {
      if (!l.gdn || !l.state) return QWEN35_ERR_INVALID_ARGUMENT;
    } else {
      return QWEN35_ERR_INVALID_ARGUMENT;
    }
  }
  cudaStream_t st = (cudaStream_t)stream;
  for (uint32_t i = 0; i < num_layers; ++i) {
    const qwen35_layer& l = layers[i];
    const qwen35_bf16* src = i == 0 ? x_in : x_out;
    int r = l.kind == QWEN35_LAYER_FULL_ATTENTION
                ? fa_forward(cfg, l.fa, scratch, scratch_bytes, l.kv, src, x_out, 0, 0, d_cache_pos, max_seq_len, st)
                : gdn_forward(cfg, l.gdn, scratch, scratch_bytes, l.state, src, x_out, st);
    if (r) return r;
  }
  return advance_pos_launch(d_cache_pos, st, true) == cudaSuccess ? QWEN35_OK : QWEN35_ERR_CUDA;
}

struct qwen35_graph {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

int qwen35_graph_create(const qwen35_config* cfg, const qwen35_layer* layers, uint32_t num_layers, void* scratch,
                        size_t scratch_bytes, const qwen35_bf16* x_in, qwen35_bf16* x_out, int32_t* d_cache_pos,
                        uint32_t max_seq_len, void* stream, qwen35_graph** out_graph) {
  if (!out_graph) return QWEN35_ERR_INVALID_ARGUMENT;
  *out_graph = nullptr;
  cudaStream_t st = (cudaStream_t)stream;
  if (st == nullptr) return QWEN35_ERR_INVALID_ARGUMENT;  // the legacy stream cannot be captured
  if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return QWEN35_ERR_CUDA;
  int r = qwen35_decode_step(cfg, layers, num_layers, scratch, scratch_bytes, x_in, x_out, d_cache_pos,
                             max_seq_len, stream);
  cudaGraph_t g = nullptr;
  cudaError_t e = cudaStreamEndCapture(st, &g);
  if (r != QWEN35_OK) {
    if (g) cudaGraphDestroy(g);
    return r;
  }
  if (e != cudaSuccess || !g) return QWEN35_ERR_CUDA;
  cudaGraphExec_t ex = nullptr;
  if (cudaGraphInstantiate(&ex, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    return QWEN35_ERR_CUDA;
  }
  qwen35_graph* out = new qwen35_graph{g, ex};
  *out_graph = out;
  return QWEN35_OK;
}

int qwen35_graph_launch(qwen35_graph* graph, void* stream) {
  if (!graph) return QWEN35_ERR_INVALID_ARGUMENT;
  return cudaGraphLaunch(graph->exec, (cudaStream_t)stream) == cudaSuccess ? QWEN35_OK : QWEN35_ERR_CUDA;
}

int qwen35_graph_destroy(qwen35_graph* graph) {
  if (!graph) return QWEN35_ERR_INVALID_ARGUMENT;
  cudaGraphExecDestroy(graph->exec);
  cudaGraphDestroy(graph->graph);
  delete graph;
  return QWEN35_OK;
}

size_t qwen35_debug_scratch_offset(const qwen35_config* cfg, int kind, const char* name) {
  const size_t none = (size_t)-1;
  if (!name || qwen35_scratch_bytes(cfg, kind) == 0) return none;
  Dims d;
  check_config(cfg, d);
  const Layout L = layout(d, kind);
  struct Named {
    const char* n;
    size_t off;
    int kind;
  };
  const int F = QWEN35_LAYER_FULL_ATTENTION, G = QWEN35_LAYER_LINEAR_ATTENTION;
  const Named tab[] = {{"q_full", L.q_full, F}, {"k", L.k, F},         {"v", L.v, F},
                       {"gated_attn", L.ga, F}, {"o", L.o, F},         {"dt_raw", L.dt_raw, G},
                       {"b_raw", L.b_raw, G},   {"qkv", L.qkv, G},     {"z", L.z, G},
                       {"y", L.y, G},           {"out", L.out, G},     {"x_resid", L.x_resid, -1},
                       {"gate_act", L.g, -1},   {"up_act", L.u, -1}};
  for (const Named& e : tab)
    if ((e.kind == kind || e.kind == -1) && std::strcmp(e.n, name) == 0) return e.off;
  return none;
}

int qwen35_gemv(const qwen35_qweight* w, const qwen35_bf16* x, qwen35_bf16* y, void* scratch, size_t scratch_bytes,
                void* stream) {
  if (!w || !aligned16(x) || !y || !aligned16(scratch) || scratch_bytes < 256) return QWEN35_ERR_INVALID_ARGUMENT;
  if (!qw_ok(*w, w->n, w->k) || w->n == 0 || w->k == 0 || w->k % 64) return QWEN35_ERR_INVALID_ARGUMENT;
  if (w->k > (uint32_t)kGemvMaxK) return QWEN35_ERR_UNSUPPORTED;
  if (num_sms() <= 0) return QWEN35_ERR_CUDA;
  GemvPlan p = {};
  p.prologue = kProPlain;
  p.epilogue = kEpiStore;
  p.args.nseg = 1;
  p.args.seg[0] = seg_of(*w, y);
  p.args.K = w->k;
  p.args.a = x;
  p.args.status = at<int>(scratch, 0);
  return launch_gemv(p, (cudaStream_t)stream, true);
}

int qwen35_dequant(const qwen35_qweight* w, float* out, void* stream) {
  if (!w || !out || !qw_ok(*w, w->n, w->k) || w->n == 0 || w->k == 0 || w->k % 64)
    return QWEN35_ERR_INVALID_ARGUMENT;
  return dequant_launch(w->codes, w->scales, w->biases, w->n, w->k, gstride_of(w->k), out,
                        (cudaStream_t)stream) == cudaSuccess
             ? QWEN35_OK
             : QWEN35_ERR_CUDA;
}

}  // extern "C"
