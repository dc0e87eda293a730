// C ABI of the decode library (include/qwen35_decode.h): argument validation,
// scratch layout, and the programs the persistent decode kernel runs.
//
// Every forward is one launch of decode_kernel (decode.cu) over a program of
// layers: one layer for qwen35_forward_full_attention / _dpos /
// qwen35_forward_linear_attention, every layer of the stack for
// qwen35_decode_step. A launch is preceded by a memset of the scratch's tagged
// words (the results CTAs hand each other), so a captured decode step is two graph
// nodes.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>

#include "qwen35_decode.h"  // include/ (on the include path)
#include "common.cuh"
#include "decode.h"
#include "prefill.h"

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
  if (d.E > 12288 || d.I > 12288) return QWEN35_ERR_UNSUPPORTED;
  return QWEN35_OK;
}

int check_fa_dims(const qwen35_config* c, const Dims& d) {
  if (d.H == 0 || d.Hkv == 0 || d.H % d.Hkv) return QWEN35_ERR_INVALID_ARGUMENT;
  if (d.R % 2 || d.R > d.D || d.R == 0) return QWEN35_ERR_INVALID_ARGUMENT;
  if (!(c->rope_theta > 0.f)) return QWEN35_ERR_INVALID_ARGUMENT;
  if (d.D != 64 && d.D != 128 && d.D != 256) return QWEN35_ERR_UNSUPPORTED;
  if (d.Hkv > 8 || d.H * d.D > 12288 || d.H * d.D % 64) return QWEN35_ERR_UNSUPPORTED;
  if (d.R / 2 > 128) return QWEN35_ERR_UNSUPPORTED;
  // attention warps: the consumer warps hold the q-heads in groups of 1 or 2
  const bool two = (d.H / d.Hkv) % 2 == 0 && d.H / 2 <= (uint32_t)kDecConsumerWarps;
  const bool one = d.H <= (uint32_t)kDecConsumerWarps;
  if (!two && !one) return QWEN35_ERR_UNSUPPORTED;
  return QWEN35_OK;
}

int check_gdn_dims(const Dims& d) {
  if (d.Hk == 0 || d.Hv == 0 || d.Hv % d.Hk) return QWEN35_ERR_INVALID_ARGUMENT;
  if ((d.Dk != 32 && d.Dk != 64 && d.Dk != 128) || (d.Dv != 32 && d.Dv != 64 && d.Dv != 128))
    return QWEN35_ERR_UNSUPPORTED;
  if (d.Kc == 0 || d.Kc > 8) return QWEN35_ERR_UNSUPPORTED;
  if (d.Z > 12288) return QWEN35_ERR_UNSUPPORTED;
  return QWEN35_OK;
}

bool qw_ok(const qwen35_qweight& w, uint32_t n, uint32_t k) {
  return w.n == n && w.k == k && aligned16(w.codes) && aligned16(w.scales) && aligned16(w.biases);
}

// ---------------------------------------------------------------- scratch layout

// [0, 4) device status word; a sequence's block from 256: the tagged words other
// CTAs read (32-bit words, zeroed before each launch), then the split-KV partials,
// then the debug stage dumps (bf16).
struct Layout {
  ScratchMap m;
  size_t total;
};

struct Bump {
  size_t off = 256;
  uint32_t take(size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return (uint32_t)o;
  }
};

// Which layer kinds a layout serves (a stack of both kinds keeps both sets apart).
constexpr int kHasFa = 1, kHasGdn = 2;

Layout layout(const Dims& d, int kinds) {
  Layout L = {};
  Bump b;
  auto words = [&](size_t n) { return b.take(n * 4); };
  L.m.tag_begin = (uint32_t)b.off;
  L.m.x_resid = words(d.E);
  L.m.g = words(d.I);
  L.m.u = words(d.I);
  L.m.xa = words(d.E);
  L.m.hq = words(d.I);
  L.m.he = words(d.I / 16);
  if (kinds & kHasFa) {
    L.m.q_full = words((size_t)2 * d.H * d.D);
    L.m.k = words((size_t)d.Hkv * d.D);
    L.m.v = words((size_t)d.Hkv * d.D);
    L.m.ga = words((size_t)d.H * d.D);
    L.m.o = words(d.E);
    L.m.flags = words(kDecMaxSplits);
  }
  if (kinds & kHasGdn) {
    L.m.dt_raw = words(d.Hv);
    L.m.b_raw = words(d.Hv);
    L.m.qkv = words(d.C);
    L.m.z = words(d.Z);
    L.m.y = words(d.Z);
    L.m.out = words(d.E);
  }
  L.m.tag_end = (uint32_t)b.off;
  if (kinds & kHasFa) {
    L.m.part_o = b.take((size_t)kDecMaxSplits * d.H * d.D * 4);
    L.m.part_ml = b.take((size_t)kDecMaxSplits * d.H * 2 * 4);
  }
  L.m.x_norm = b.take((size_t)d.E * 2);
  L.m.x_norm2 = b.take((size_t)d.E * 2);
  if (kinds & kHasFa) {
    L.m.k_rot = b.take((size_t)d.Hkv * d.D * 2);
    L.m.v_rot = b.take((size_t)d.Hkv * d.D * 2);
  }
  if (kinds & kHasGdn) {
    L.m.qkv_smooth = b.take((size_t)d.C * 2);
    L.m.y_norm = b.take((size_t)d.Z * 2);
  }
  L.total = b.off;
  return L;
}
int kinds_of(int layer_kind) { return layer_kind == QWEN35_LAYER_FULL_ATTENTION ? kHasFa : kHasGdn; }

QMat qm(const qwen35_qweight& w) {
  QMat m;
  m.codes = w.codes;
  m.scales = w.scales;
  m.biases = w.biases;
  m.n = w.n;
  m.pad = 0;
  return m;
}

// The cache of a full-attention layer: aligned pointers, a known format (Turbo8:
// scale arrays too).
bool kv_ok(const qwen35_kv_cache* kv) {
  if (!kv || !aligned16(kv->k) || !aligned16(kv->v) || kv->capacity == 0) return false;
  if (kv->block_table) {  // paged: bf16 blocks of a power of two >= 8 rows dividing the capacity
    const uint32_t bt = kv->block_tokens;
    if (kv->dtype != QWEN35_KV_BF16 || ((uintptr_t)kv->block_table % 4) || bt < 8 || (bt & (bt - 1)) ||
        kv->capacity % bt)
      return false;
    return true;
  }
  if (kv->dtype == QWEN35_KV_BF16) return true;
  if (kv->dtype == QWEN35_KV_TURBO8) return aligned16(kv->k_scales) && aligned16(kv->v_scales);
  return false;
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
      !l->dt_bias || !aligned16(l->conv1d_weight) || ((uintptr_t)l->a_log % 4) || ((uintptr_t)l->dt_bias % 2))
    return QWEN35_ERR_INVALID_ARGUMENT;
  if (!qw_ok(l->in_proj_a, d.Hv, d.E) || !qw_ok(l->in_proj_b, d.Hv, d.E) ||
      !qw_ok(l->in_proj_qkv, d.C, d.E) || !qw_ok(l->in_proj_z, d.Z, d.E) || !qw_ok(l->out_proj, d.E, d.Z) ||
      !qw_ok(l->gate_proj, d.I, d.E) || !qw_ok(l->up_proj, d.I, d.E) || !qw_ok(l->down_proj, d.E, d.I))
    return QWEN35_ERR_INVALID_ARGUMENT;
  return QWEN35_OK;
}

void fill_fa(LayerDesc& L, const qwen35_fa_layer* l, const qwen35_kv_cache* kv) {
  L.kind = kLayerFA;
  L.capacity = kv->capacity;
  L.m[0] = qm(l->q_proj);
  L.m[1] = qm(l->k_proj);
  L.m[2] = qm(l->v_proj);
  L.m[3] = qm(l->o_proj);
  L.m[4] = qm(l->gate_proj);
  L.m[5] = qm(l->up_proj);
  L.m[6] = qm(l->down_proj);
  L.input_ln = l->input_ln;
  L.post_ln = l->post_ln;
  L.q_norm = l->q_norm;
  L.k_norm = l->k_norm;
  L.kc = static_cast<uint8_t*>(kv->k);
  L.vc = static_cast<uint8_t*>(kv->v);
  L.kv_dtype = kv->dtype;
  L.ks = kv->k_scales;
  L.vs = kv->v_scales;
  L.btab = kv->block_table;
  L.bt_shift = 0;
  if (kv->block_table)
    while ((1u << L.bt_shift) < kv->block_tokens) ++L.bt_shift;
}

void fill_gdn(LayerDesc& L, const qwen35_gdn_layer* l, const qwen35_gdn_state* st) {
  L.kind = kLayerGDN;
  L.m[0] = qm(l->in_proj_a);
  L.m[1] = qm(l->in_proj_b);
  L.m[2] = qm(l->in_proj_qkv);
  L.m[3] = qm(l->in_proj_z);
  L.m[4] = qm(l->gate_proj);
  L.m[5] = qm(l->up_proj);
  L.m[6] = qm(l->down_proj);
  L.m[7] = qm(l->out_proj);
  L.input_ln = l->input_ln;
  L.post_ln = l->post_ln;
  L.norm_weight = l->norm_weight;
  L.dt_bias = l->dt_bias;
  L.conv_w = l->conv1d_weight;
  L.a_log = l->a_log;
  L.conv_state = st->conv_state;
  L.ssm = st->gdn_state;
}

// Debug settings of the next launches (qwen35_debug_*).
unsigned long long g_wait_ns = kWaitNs;
const uint32_t* g_wait_probe = nullptr;
uint32_t g_dump = 0;

// The program header shared by every call; the caller fills the scratch map and
// the layers.
Program* new_program(const qwen35_config* cfg, const Dims& d, void* scratch) {
  Program* p = new (std::nothrow) Program();
  if (!p) return nullptr;
  p->E = d.E; p->I = d.I; p->H = d.H; p->Hkv = d.Hkv; p->D = d.D; p->R = d.R;
  p->Hk = d.Hk; p->Hv = d.Hv; p->Dk = d.Dk; p->Dv = d.Dv; p->Kc = d.Kc; p->C = d.C; p->Z = d.Z;
  p->eps = cfg->rms_eps;
  p->scale_log2 = d.D ? (float)(1.0 / std::sqrt((double)d.D) * 1.4426950408889634) : 0.f;
  p->gdn_out_scale = d.Dk ? (float)(1.0 / std::sqrt((double)d.Dk)) : 0.f;
  p->l2_eps = 1e-6f;
  p->scratch = static_cast<uint8_t*>(scratch);
  p->status = reinterpret_cast<int*>(scratch);
  p->wait_ns = g_wait_ns;
  p->wait_probe = g_wait_probe;
  p->dump = g_dump;
  p->batch = 1;
  p->seq_stride = 0;
  // inv_freq[i] = theta^(-2i/R), computed in double and kept as fp32
  for (uint32_t i = 0; i < d.R / 2 && i < 128; ++i)
    p->inv_freq[i] = (float)std::pow((double)cfg->rope_theta, -2.0 * (double)i / (double)d.R);
  return p;
}

// Phase timeline of the next launches (qwen35_debug_trace); off when null.
unsigned long long* g_trace = nullptr;
uint32_t g_trace_phases = 0;

uint32_t splits_for(uint32_t span) {
  uint32_t P = (span + 31) / 32;
  if (P > (uint32_t)num_sms()) P = num_sms();
  if (P > (uint32_t)kDecMaxSplits) P = kDecMaxSplits;
  return P == 0 ? 1 : P;
}

int launch(Program* p, bool has_fa, bool has_gdn, cudaStream_t st) {
  p->trace = g_trace;
  p->trace_phases = g_trace_phases;
  int r = QWEN35_OK;
  if (!decode_pick_split(*p, has_fa, has_gdn, num_sms())) r = QWEN35_ERR_UNSUPPORTED;
  else if (decode_launch(*p, num_sms(), st) != cudaSuccess) r = QWEN35_ERR_CUDA;
  delete p;
  return r;
}

int fa_forward(const qwen35_config* cfg, const qwen35_fa_layer* layer, void* scratch, size_t scratch_bytes,
               const qwen35_kv_cache* kv, const uint16_t* x_in, uint16_t* x_out, uint32_t cache_pos,
               uint32_t seq_len, const int32_t* d_pos, uint32_t max_seq, cudaStream_t st) {
  Dims d;
  int r = check_config(cfg, d);
  if (r) return r;
  if ((r = check_fa_dims(cfg, d))) return r;
  if ((r = check_fa_layer(layer, d))) return r;
  if (!kv_ok(kv)) return QWEN35_ERR_INVALID_ARGUMENT;
  if (!aligned16(x_in) || !aligned16(x_out) || !aligned16(scratch)) return QWEN35_ERR_INVALID_ARGUMENT;
  const Layout lay = layout(d, kHasFa);
  if (scratch_bytes < lay.total) return QWEN35_ERR_INVALID_ARGUMENT;
  if (d_pos) {
    if (max_seq == 0) return QWEN35_ERR_INVALID_ARGUMENT;
  } else if (cache_pos >= kv->capacity || seq_len == 0 || seq_len > cache_pos + 1) {
    return QWEN35_ERR_OUT_OF_RANGE;
  }
  if (num_sms() <= 0) return QWEN35_ERR_CUDA;
  Program* p = new_program(cfg, d, scratch);
  if (!p) return QWEN35_ERR_CUDA;
  p->sm = lay.m;
  p->n_layers = 1;
  p->x_in = x_in;
  p->x_out = x_out;
  p->pos = cache_pos;
  p->S = seq_len;
  p->d_pos = d_pos;
  p->max_seq = max_seq;
  p->P = splits_for(d_pos ? max_seq : seq_len);
  fill_fa(p->layers[0], layer, kv);
  return launch(p, true, false, st);
}

// The linear-attention forward's checks of everything but the scratch.
int gdn_check(const qwen35_config* cfg, const qwen35_gdn_layer* layer, const qwen35_gdn_state* state,
              const uint16_t* x_in, const uint16_t* x_out, Dims& d) {
  int r = check_config(cfg, d);
  if (r) return r;
  if ((r = check_gdn_dims(d))) return r;
  if ((r = check_gdn_layer(layer, d))) return r;
  if (!state || !aligned16(state->conv_state) || !aligned16(state->gdn_state)) return QWEN35_ERR_INVALID_ARGUMENT;
  if (!aligned16(x_in) || !aligned16(x_out)) return QWEN35_ERR_INVALID_ARGUMENT;
  return QWEN35_OK;
}

int gdn_forward(const qwen35_config* cfg, const qwen35_gdn_layer* layer, void* scratch, size_t scratch_bytes,
                const qwen35_gdn_state* state, const uint16_t* x_in, uint16_t* x_out, cudaStream_t st) {
  Dims d;
  const int r = gdn_check(cfg, layer, state, x_in, x_out, d);
  if (r) return r;
  if (!aligned16(scratch)) return QWEN35_ERR_INVALID_ARGUMENT;
  const Layout lay = layout(d, kHasGdn);
  if (scratch_bytes < lay.total) return QWEN35_ERR_INVALID_ARGUMENT;
  if (num_sms() <= 0) return QWEN35_ERR_CUDA;
  Program* p = new_program(cfg, d, scratch);
  if (!p) return QWEN35_ERR_CUDA;
  p->sm = lay.m;
  p->n_layers = 1;
  p->x_in = x_in;
  p->x_out = x_out;
  fill_gdn(p->layers[0], layer, state);
  return launch(p, false, true, st);
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
  int major = 0, minor = 0, sms = 0, coop = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
    return QWEN35_ERR_CUDA;
  if (major != 10 || minor != 3 || !coop) return QWEN35_ERR_CUDA;  // built for sm_103a only
  if (decode_set_attributes() != cudaSuccess) return QWEN35_ERR_CUDA;
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
  return layout(d, kinds_of(kind)).total;
}

size_t qwen35_stack_scratch_bytes(const qwen35_config* cfg) {
  if (qwen35_scratch_bytes(cfg, QWEN35_LAYER_FULL_ATTENTION) == 0 ||
      qwen35_scratch_bytes(cfg, QWEN35_LAYER_LINEAR_ATTENTION) == 0)
    return 0;
  Dims d;
  check_config(cfg, d);
  return layout(d, kHasFa | kHasGdn).total;
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

namespace {
// The device address of the static array on the current device, looked up once per
// device (with that device current) and cached; null on failure.
void* static_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (!g_static_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return nullptr;
    g_static_scratch_ptr[dev] = p;
  }
  return g_static_scratch_ptr[dev];
}
}  // namespace

int qwen35_forward_linear_attention_static(const qwen35_config* cfg, const qwen35_gdn_layer* layer,
                                           const qwen35_gdn_state* state, const qwen35_bf16* x_in,
                                           qwen35_bf16* x_out, void* stream) {
  // every argument is checked before the device is touched: a rejected call leaves
  // the array (and the previous call's status word) as it was. The config first:
  // one that needs more scratch than the array is unsupported whatever the pointers.
  Dims d;
  int r = check_config(cfg, d);
  if (r) return r;
  if ((r = check_gdn_dims(d))) return r;
  if (layout(d, kHasGdn).total > QWEN35_STATIC_SCRATCH_BYTES) return QWEN35_ERR_UNSUPPORTED;
  if ((r = gdn_check(cfg, layer, state, x_in, x_out, d))) return r;
  void* scratch = static_scratch();
  if (!scratch) return QWEN35_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  // the array keeps the previous call's contents: the status word must start at zero
  if (cudaMemsetAsync(scratch, 0, 256, st) != cudaSuccess) return QWEN35_ERR_CUDA;
  return gdn_forward(cfg, layer, scratch, QWEN35_STATIC_SCRATCH_BYTES, state, x_in, x_out, st);
}

int qwen35_read_static_status(int32_t* host_status, void* stream) {
  if (!host_status) return QWEN35_ERR_INVALID_ARGUMENT;
  void* scratch = static_scratch();
  if (!scratch) return QWEN35_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return QWEN35_ERR_CUDA;
  return cudaMemcpy(host_status, scratch, 4, cudaMemcpyDeviceToHost) == cudaSuccess ? QWEN35_OK : QWEN35_ERR_CUDA;
}

namespace {

// Scratch of one sequence's intermediates in a stack program (both layer kinds'
// maps share it), and of a batch: the status word and barrier counter, then one
// block per sequence.
Layout stack_layout(const Dims& d, bool has_fa, bool has_gdn) {
  return layout(d, (has_fa ? kHasFa : 0) | (has_gdn ? kHasGdn : 0));
}
size_t batch_need(size_t one, uint32_t batch) { return 256 + (size_t)batch * (one - 256); }

// A program of layers over a batch of sequences. `advance`: the kernel advances
// every sequence's device position after the last layer (a decode step); the
// per-layer batched forwards leave the positions alone, and a program without a
// full-attention layer reads none (d_cache_pos may then be null). `check_only`:
// return after the argument checks, before any CUDA call.
int decode_step(const qwen35_config* cfg, const qwen35_layer* layers, uint32_t num_layers, uint32_t batch,
                void* scratch, size_t scratch_bytes, const qwen35_bf16* x_in, qwen35_bf16* x_out,
                int32_t* d_cache_pos, uint32_t max_seq_len, cudaStream_t stream, bool advance = true,
                bool check_only = false) {
  if (!layers || num_layers == 0 || num_layers > (uint32_t)kMaxLayers || batch == 0 ||
      batch > (uint32_t)kMaxBatch)
    return QWEN35_ERR_INVALID_ARGUMENT;
  bool any_fa = false;
  for (uint32_t i = 0; i < num_layers; ++i) any_fa |= layers[i].kind == QWEN35_LAYER_FULL_ATTENTION;
  if (advance || any_fa) {
    if (!d_cache_pos || ((uintptr_t)d_cache_pos % 4) || max_seq_len == 0) return QWEN35_ERR_INVALID_ARGUMENT;
  } else if (d_cache_pos && ((uintptr_t)d_cache_pos % 4)) {
    return QWEN35_ERR_INVALID_ARGUMENT;
  }
  Dims d;
  int r = check_config(cfg, d);
  if (r) return r;
  bool has_fa = false, has_gdn = false;
  for (uint32_t i = 0; i < num_layers; ++i) {
    const qwen35_layer& l = layers[i];
    if (l.kind == QWEN35_LAYER_FULL_ATTENTION) {
      if (!l.fa || !kv_ok(l.kv)) return QWEN35_ERR_INVALID_ARGUMENT;
      if ((r = check_fa_dims(cfg, d)) || (r = check_fa_layer(l.fa, d))) return r;
      has_fa = true;
    } else if (l.kind == QWEN35_LAYER_LINEAR_ATTENTION) {
      if (!l.gdn || !l.state || !aligned16(l.state->conv_state) || !aligned16(l.state->gdn_state))
        return QWEN35_ERR_INVALID_ARGUMENT;
      if ((r = check_gdn_dims(d)) || (r = check_gdn_layer(l.gdn, d))) return r;
      has_gdn = true;
    } else {
      return QWEN35_ERR_INVALID_ARGUMENT;
    }
  }
  if (!aligned16(x_in) || !aligned16(x_out) || !aligned16(scratch)) return QWEN35_ERR_INVALID_ARGUMENT;
  const Layout lay = stack_layout(d, has_fa, has_gdn);
  const size_t one = lay.total;
  if (scratch_bytes < batch_need(one, batch)) return QWEN35_ERR_INVALID_ARGUMENT;
  if (check_only) return QWEN35_OK;
  if (num_sms() <= 0) return QWEN35_ERR_CUDA;
  Program* p = new_program(cfg, d, scratch);
  if (!p) return QWEN35_ERR_CUDA;
  p->sm = lay.m;
  p->n_layers = num_layers;
  p->x_in = x_in;
  p->x_out = x_out;
  p->d_pos = any_fa ? d_cache_pos : nullptr;
  p->max_seq = max_seq_len ? max_seq_len : 1;
  p->P = splits_for(p->max_seq);
  p->advance = advance ? d_cache_pos : nullptr;
  p->batch = batch;
  p->seq_stride = (uint32_t)(one - 256);
  for (uint32_t i = 0; i < num_layers; ++i) {
    if (layers[i].kind == QWEN35_LAYER_FULL_ATTENTION) fill_fa(p->layers[i], layers[i].fa, layers[i].kv);
    else fill_gdn(p->layers[i], layers[i].gdn, layers[i].state);
  }
  return launch(p, has_fa, has_gdn, stream);
}

}  // namespace

int qwen35_decode_step(const qwen35_config* cfg, const qwen35_layer* layers, uint32_t num_layers, void* scratch,
                       size_t scratch_bytes, const qwen35_bf16* x_in, qwen35_bf16* x_out, int32_t* d_cache_pos,
                       uint32_t max_seq_len, void* stream) {
  return decode_step(cfg, layers, num_layers, 1, scratch, scratch_bytes, x_in, x_out, d_cache_pos, max_seq_len,
                     (cudaStream_t)stream);
}

int qwen35_decode_step_batched(const qwen35_config* cfg, const qwen35_layer* layers, uint32_t num_layers,
                               uint32_t batch, void* scratch, size_t scratch_bytes, const qwen35_bf16* x_in,
                               qwen35_bf16* x_out, int32_t* d_cache_pos, uint32_t max_seq_len, void* stream) {
  return decode_step(cfg, layers, num_layers, batch, scratch, scratch_bytes, x_in, x_out, d_cache_pos, max_seq_len,
                     (cudaStream_t)stream);
}

int qwen35_forward_full_attention_batched(const qwen35_config* cfg, const qwen35_fa_layer* layer, uint32_t batch,
                                          void* scratch, size_t scratch_bytes, const qwen35_kv_cache* kv,
                                          const qwen35_bf16* x_in, qwen35_bf16* x_out, const int32_t* d_cache_pos,
                                          uint32_t max_seq_len, void* stream) {
  if (!layer || !kv || !d_cache_pos) return QWEN35_ERR_INVALID_ARGUMENT;
  qwen35_layer l = {QWEN35_LAYER_FULL_ATTENTION, layer, kv, nullptr, nullptr};
  return decode_step(cfg, &l, 1, batch, scratch, scratch_bytes, x_in, x_out, const_cast<int32_t*>(d_cache_pos),
                     max_seq_len, (cudaStream_t)stream, false);
}

int qwen35_forward_linear_attention_batched(const qwen35_config* cfg, const qwen35_gdn_layer* layer, uint32_t batch,
                                            void* scratch, size_t scratch_bytes, const qwen35_gdn_state* state,
                                            const qwen35_bf16* x_in, qwen35_bf16* x_out, void* stream) {
  if (!layer || !state) return QWEN35_ERR_INVALID_ARGUMENT;
  qwen35_layer l = {QWEN35_LAYER_LINEAR_ATTENTION, nullptr, nullptr, layer, state};
  return decode_step(cfg, &l, 1, batch, scratch, scratch_bytes, x_in, x_out, nullptr, 0, (cudaStream_t)stream, false);
}

size_t qwen35_stack_scratch_bytes_batched(const qwen35_config* cfg, uint32_t batch) {
  Dims d;
  if (!cfg || batch == 0 || batch > (uint32_t)kMaxBatch || check_config(cfg, d) != QWEN35_OK) return 0;
  return batch_need(stack_layout(d, true, true).total, batch);
}

struct qwen35_graph {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

namespace {
int graph_create(const qwen35_config* cfg, const qwen35_layer* layers, uint32_t num_layers, uint32_t batch,
                 void* scratch, size_t scratch_bytes, const qwen35_bf16* x_in, qwen35_bf16* x_out,
                 int32_t* d_cache_pos, uint32_t max_seq_len, void* stream, qwen35_graph** out_graph) {
  if (!out_graph) return QWEN35_ERR_INVALID_ARGUMENT;
  *out_graph = nullptr;
  cudaStream_t st = (cudaStream_t)stream;
  if (st == nullptr) return QWEN35_ERR_INVALID_ARGUMENT;  // the legacy stream cannot be captured
  // argument errors before the capture begins: the caller's stream is left alone
  int r = decode_step(cfg, layers, num_layers, batch, scratch, scratch_bytes, x_in, x_out, d_cache_pos, max_seq_len,
                      st, true, true);
  if (r != QWEN35_OK) return r;
  if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return QWEN35_ERR_CUDA;
  r = decode_step(cfg, layers, num_layers, batch, scratch, scratch_bytes, x_in, x_out, d_cache_pos, max_seq_len, st);
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
  qwen35_graph* out = new (std::nothrow) qwen35_graph{g, ex};
  if (!out) {
    cudaGraphExecDestroy(ex);
    cudaGraphDestroy(g);
    return QWEN35_ERR_CUDA;
  }
  *out_graph = out;
  return QWEN35_OK;
}
}  // namespace

int qwen35_graph_create(const qwen35_config* cfg, const qwen35_layer* layers, uint32_t num_layers, void* scratch,
                        size_t scratch_bytes, const qwen35_bf16* x_in, qwen35_bf16* x_out, int32_t* d_cache_pos,
                        uint32_t max_seq_len, void* stream, qwen35_graph** out_graph) {
  return graph_create(cfg, layers, num_layers, 1, scratch, scratch_bytes, x_in, x_out, d_cache_pos, max_seq_len,
                      stream, out_graph);
}

int qwen35_graph_create_batched(const qwen35_config* cfg, const qwen35_layer* layers, uint32_t num_layers,
                                uint32_t batch, void* scratch, size_t scratch_bytes, const qwen35_bf16* x_in,
                                qwen35_bf16* x_out, int32_t* d_cache_pos, uint32_t max_seq_len, void* stream,
                                qwen35_graph** out_graph) {
  return graph_create(cfg, layers, num_layers, batch, scratch, scratch_bytes, x_in, x_out, d_cache_pos, max_seq_len,
                      stream, out_graph);
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

namespace {
// A named intermediate's offset in map m; kind -1 accepts either kind's names.
size_t named_offset(const ScratchMap& m, int kind, const char* name) {
  struct Named {
    const char* n;
    uint32_t off;
    int kind;
  };
  const int F = QWEN35_LAYER_FULL_ATTENTION, G = QWEN35_LAYER_LINEAR_ATTENTION;
  const Named tab[] = {{"q_full", m.q_full, F},    {"k", m.k, F},          {"v", m.v, F},
                       {"gated_attn", m.ga, F},    {"o", m.o, F},          {"dt_raw", m.dt_raw, G},
                       {"b_raw", m.b_raw, G},      {"qkv", m.qkv, G},      {"z", m.z, G},
                       {"y", m.y, G},              {"out", m.out, G},      {"x_resid", m.x_resid, -1},
                       {"gate_act", m.g, -1},      {"up_act", m.u, -1},    {"x_norm", m.x_norm, -1},
                       {"x_norm2", m.x_norm2, -1}, {"qkv_smooth", m.qkv_smooth, G}, {"y_norm", m.y_norm, G},
                       {"k_rot", m.k_rot, F},      {"v_rot", m.v_rot, F}};
  for (const Named& e : tab)
    if ((kind == -1 || e.kind == kind || e.kind == -1) && std::strcmp(e.n, name) == 0) return e.off;
  return (size_t)-1;
}
}  // namespace

size_t qwen35_debug_scratch_offset(const qwen35_config* cfg, int kind, const char* name) {
  if (!name || qwen35_scratch_bytes(cfg, kind) == 0) return (size_t)-1;
  Dims d;
  check_config(cfg, d);
  return named_offset(layout(d, kinds_of(kind)).m, kind, name);
}

size_t qwen35_debug_stack_scratch_offset(const qwen35_config* cfg, const char* name) {
  if (!name || qwen35_stack_scratch_bytes(cfg) == 0) return (size_t)-1;
  Dims d;
  check_config(cfg, d);
  return named_offset(layout(d, kHasFa | kHasGdn).m, -1, name);
}

int qwen35_debug_stage_dump(int on) {
  g_dump = on ? 1u : 0u;
  return QWEN35_OK;
}

int qwen35_debug_set_wait_limit(unsigned long long limit_ns) {
  g_wait_ns = limit_ns ? limit_ns : kWaitNs;
  return QWEN35_OK;
}

int qwen35_debug_wait_probe(const uint32_t* d_flag) {
  if (d_flag && ((uintptr_t)d_flag % 4)) return QWEN35_ERR_INVALID_ARGUMENT;
  g_wait_probe = d_flag;
  return QWEN35_OK;
}

int qwen35_gemv(const qwen35_qweight* w, const qwen35_bf16* x, qwen35_bf16* y, void* scratch, size_t scratch_bytes,
                void* stream) {
  if (!w || !aligned16(x) || !aligned16(y) || !aligned16(scratch) || scratch_bytes < 256)
    return QWEN35_ERR_INVALID_ARGUMENT;
  if (!qw_ok(*w, w->n, w->k) || w->n == 0 || w->k == 0 || w->k % 64) return QWEN35_ERR_INVALID_ARGUMENT;
  if (w->k > 12288) return QWEN35_ERR_UNSUPPORTED;
  if (num_sms() <= 0) return QWEN35_ERR_CUDA;
  qwen35_config cfg = {};
  cfg.group_size = 64;
  Dims d = {};
  d.E = w->k;
  d.I = w->k;
  Program* p = new_program(&cfg, d, scratch);
  if (!p) return QWEN35_ERR_CUDA;
  p->n_layers = 1;
  p->x_in = x;
  p->x_out = y;
  p->layers[0].kind = kLayerGemv;
  p->layers[0].m[0] = qm(*w);
  return launch(p, false, false, (cudaStream_t)stream);
}

int qwen35_debug_trace(unsigned long long* d_trace, uint32_t max_phases) {
  if ((d_trace == nullptr) != (max_phases == 0)) return QWEN35_ERR_INVALID_ARGUMENT;
  g_trace = d_trace;
  g_trace_phases = max_phases;
  return QWEN35_OK;
}

int qwen35_lm_head_greedy(const qwen35_config* cfg, const qwen35_bf16* final_norm, const qwen35_qweight* lm_head,
                          const qwen35_bf16* x, qwen35_bf16* logits, int32_t* token, void* scratch,
                          size_t scratch_bytes, void* stream) {
  if (!cfg || !lm_head || !aligned16(final_norm) || !aligned16(x) || !aligned16(logits) || !token ||
      ((uintptr_t)token % 4) || !aligned16(scratch) || scratch_bytes < 256)
    return QWEN35_ERR_INVALID_ARGUMENT;
  const uint32_t E = cfg->hidden;
  if (E == 0 || E % 64 || cfg->group_size != 64 || !(cfg->rms_eps >= 0.f)) return QWEN35_ERR_INVALID_ARGUMENT;
  if (lm_head->n == 0 || !qw_ok(*lm_head, lm_head->n, E)) return QWEN35_ERR_INVALID_ARGUMENT;
  if (E > 12288) return QWEN35_ERR_UNSUPPORTED;
  if (num_sms() <= 0) return QWEN35_ERR_CUDA;
  Dims d = {};
  d.E = E;
  d.I = E;
  Program* p = new_program(cfg, d, scratch);
  if (!p) return QWEN35_ERR_CUDA;
  p->n_layers = 1;
  p->x_in = x;
  p->x_out = logits;
  p->layers[0].kind = kLayerHead;
  p->layers[0].m[0] = qm(*lm_head);
  p->layers[0].input_ln = final_norm;
  const cudaStream_t st = (cudaStream_t)stream;
  const int r = launch(p, false, false, st);
  if (r != QWEN35_OK) return r;
  return argmax_bf16_launch(logits, lm_head->n, token, st) == cudaSuccess ? QWEN35_OK : QWEN35_ERR_CUDA;
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

// ---------------------------------------------------------------- prefill

namespace {

// Scratch of a prefill of up to T tokens after the status word: per-token buffers
// (bf16 unless noted), each 256-byte aligned; both layer kinds' buffers, so one
// scratch serves a stack.
struct PfLayout {
  size_t xn, xr, o, g, u;                                // [T][E] x3, [T][I] x2
  size_t qf, k, v, qr, ga;                               // full attention
  size_t dt, bb, qkv, z, qs, gb, act, y, yin;            // linear attention (gb, act fp32)
  size_t ws;                                             // split-K partial sums (fp32)
  size_t total;
};
PfLayout pf_layout(const Dims& d, uint32_t T) {
  PfLayout L = {};
  size_t off = 256;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  };
  const size_t t = T;
  L.xn = take(t * d.E * 2);
  L.xr = take(t * d.E * 2);
  L.o = take(t * d.E * 2);
  L.g = take(t * d.I * 2);
  L.u = take(t * d.I * 2);
  L.qf = take(t * 2 * d.H * d.D * 2);
  L.k = take(t * d.Hkv * d.D * 2);
  L.v = take(t * d.Hkv * d.D * 2);
  L.qr = take(t * d.H * d.D * 2);
  L.ga = take(t * d.H * d.D * 2);
  L.dt = take(t * d.Hv * 2);
  L.bb = take(t * d.Hv * 2);
  L.qkv = take(t * d.C * 2);
  L.z = take(t * d.Z * 2);
  L.qs = take(t * d.C * 2);
  L.gb = take(t * d.Hv * 2 * 4);
  L.act = take(t * d.C * 4);
  L.y = take(t * d.Z * 2);
  L.yin = take(t * d.Z * 2);
  L.ws = take(q35pf::kGemmWorkspace);
  L.total = off;
  return L;
}

constexpr uint32_t kMaxPrefillTokens = 65536;

struct PfCtx {
  const qwen35_config* cfg;
  Dims d;
  uint8_t* s;  // scratch
  PfLayout L;
  uint32_t T;
  cudaStream_t st;
  float* ws;  // split-K workspace, or null
  uint16_t* b16(size_t off) const { return reinterpret_cast<uint16_t*>(s + off); }
  float* f32(size_t off) const { return reinterpret_cast<float*>(s + off); }
  int* status() const { return reinterpret_cast<int*>(s); }
};

// The checks every prefill entry shares: config, scratch size, token count, x.
int pf_begin(PfCtx& c, const qwen35_config* cfg, void* scratch, size_t scratch_bytes, const void* x_in,
             const void* x_out, uint32_t T, cudaStream_t st) {
  int r = check_config(cfg, c.d);
  if (r) return r;
  if (T == 0 || T > kMaxPrefillTokens || !aligned16(scratch) || !aligned16(x_in) || !aligned16(x_out))
    return QWEN35_ERR_INVALID_ARGUMENT;
  c.cfg = cfg;
  c.L = pf_layout(c.d, T);
  if (scratch_bytes < c.L.total) return QWEN35_ERR_INVALID_ARGUMENT;
  c.s = static_cast<uint8_t*>(scratch);
  c.T = T;
  c.st = st;
  c.ws = c.f32(c.L.ws);
  return QWEN35_OK;
}

int cu(cudaError_t e) { return e == cudaSuccess ? QWEN35_OK : QWEN35_ERR_CUDA; }

// A prefill projection. exact: the weights to 2^-16 (the projections whose outputs
// are kept: k_proj and v_proj fill the KV cache, in_proj_qkv/a/b drive the conv and
// delta-rule states); otherwise bf16-rounded weights.
int pf_gemm(const PfCtx& c, const qwen35_qweight& w, const uint16_t* X, uint16_t* Y, const uint16_t* R,
            bool exact) {
  q35pf::Gemm g;
  g.X = X;
  g.codes = w.codes;
  g.scales = w.scales;
  g.biases = w.biases;
  g.Y = Y;
  g.R = R;
  g.ldx = w.k;
  g.ldy = w.n;
  g.gstride = gstride_of(w.k);
  g.N = w.n;
  g.K = w.k;
  g.T = c.T;
  g.status = c.status();
  g.wait_ns = g_wait_ns;
  g.exact = exact;
  g.ws = c.ws;
  return cu(q35pf::gemm(g, c.st));
}

// x_out = x_resid + down(SiLU(gate) * up) with x_resid = bf16(x_in + delta) and
// the MLP input RMSNorm(x_resid) * post_ln. x_in is last read before x_out is
// written, so the two may be one buffer.
int pf_mlp(const PfCtx& c, const uint16_t* x_in, const uint16_t* delta, const uint16_t* post_ln,
           const qwen35_qweight& gate, const qwen35_qweight& up, const qwen35_qweight& down, uint16_t* x_out) {
  const Dims& d = c.d;
  uint16_t *xn = c.b16(c.L.xn), *xr = c.b16(c.L.xr), *g = c.b16(c.L.g), *u = c.b16(c.L.u);
  int r = cu(q35pf::rmsnorm(x_in, delta, xr, post_ln, xn, c.T, d.E, c.cfg->rms_eps, c.st));
  if (!r) r = pf_gemm(c, gate, xn, g, nullptr, false);
  if (!r) r = pf_gemm(c, up, xn, u, nullptr, false);
  if (!r) r = cu(q35pf::silu_mul(g, u, g, (size_t)c.T * d.I, c.st));
  if (!r) r = pf_gemm(c, down, g, x_out, xr, false);
  return r;
}

int pf_fa(const PfCtx& c, const qwen35_fa_layer* l, const qwen35_kv_cache* kv, const uint16_t* x_in,
          uint16_t* x_out, uint32_t p0) {
  const Dims& d = c.d;
  uint16_t *xn = c.b16(c.L.xn), *qf = c.b16(c.L.qf), *k = c.b16(c.L.k), *v = c.b16(c.L.v);
  int r = cu(q35pf::rmsnorm(x_in, nullptr, nullptr, l->input_ln, xn, c.T, d.E, c.cfg->rms_eps, c.st));
  if (!r) r = pf_gemm(c, l->q_proj, xn, qf, nullptr, false);
  if (!r) r = pf_gemm(c, l->k_proj, xn, k, nullptr, true);
  if (!r) r = pf_gemm(c, l->v_proj, xn, v, nullptr, true);
  if (r) return r;
  q35pf::Attn a = {};
  a.qf = qf;
  a.k = k;
  a.v = v;
  a.q_norm = l->q_norm;
  a.k_norm = l->k_norm;
  a.qr = c.b16(c.L.qr);
  a.kc = static_cast<uint16_t*>(kv->k);
  a.vc = static_cast<uint16_t*>(kv->v);
  a.turbo8 = kv->dtype == QWEN35_KV_TURBO8;
  a.ks = kv->k_scales;
  a.vs = kv->v_scales;
  a.sstride = (d.Hkv * d.D / 16 + 7) / 8 * 8;  // scale rows padded to 16 bytes
  a.btab = kv->block_table;
  a.bt_shift = 0;
  if (kv->block_table)
    while ((1u << a.bt_shift) < kv->block_tokens) ++a.bt_shift;
  a.ga = c.b16(c.L.ga);
  a.T = c.T;
  a.p0 = p0;
  a.H = d.H;
  a.Hkv = d.Hkv;
  a.D = d.D;
  a.R = d.R;
  a.eps = c.cfg->rms_eps;
  for (uint32_t i = 0; i < d.R / 2 && i < 128; ++i)  // theta^(-2i/R) in double, kept fp32
    a.inv_freq[i] = (float)std::pow((double)c.cfg->rope_theta, -2.0 * (double)i / (double)d.R);
  r = cu(q35pf::attention(a, c.st));
  if (!r) r = pf_gemm(c, l->o_proj, a.ga, c.b16(c.L.o), nullptr, false);
  if (!r) r = pf_mlp(c, x_in, c.b16(c.L.o), l->post_ln, l->gate_proj, l->up_proj, l->down_proj, x_out);
  return r;
}

int pf_gdn(const PfCtx& c, const qwen35_gdn_layer* l, const qwen35_gdn_state* st, const uint16_t* x_in,
           uint16_t* x_out) {
  const Dims& d = c.d;
  uint16_t* xn = c.b16(c.L.xn);
  q35pf::Gdn g = {};
  g.qkv = c.b16(c.L.qkv);
  g.z = c.b16(c.L.z);
  g.dt_raw = c.b16(c.L.dt);
  g.b_raw = c.b16(c.L.bb);
  int r = cu(q35pf::rmsnorm(x_in, nullptr, nullptr, l->input_ln, xn, c.T, d.E, c.cfg->rms_eps, c.st));
  if (!r) r = pf_gemm(c, l->in_proj_a, xn, c.b16(c.L.dt), nullptr, true);
  if (!r) r = pf_gemm(c, l->in_proj_b, xn, c.b16(c.L.bb), nullptr, true);
  if (!r) r = pf_gemm(c, l->in_proj_qkv, xn, c.b16(c.L.qkv), nullptr, true);
  if (!r) r = pf_gemm(c, l->in_proj_z, xn, c.b16(c.L.z), nullptr, false);
  if (r) return r;
  g.conv_w = l->conv1d_weight;
  g.a_log = l->a_log;
  g.dt_bias = l->dt_bias;
  g.norm_w = l->norm_weight;
  g.conv_state = st->conv_state;
  g.ssm = st->gdn_state;
  g.qs = c.b16(c.L.qs);
  g.act = c.f32(c.L.act);
  g.gb = c.f32(c.L.gb);
  g.y = c.b16(c.L.y);
  g.yin = c.b16(c.L.yin);
  g.T = c.T;
  g.Hk = d.Hk;
  g.Hv = d.Hv;
  g.Dk = d.Dk;
  g.Dv = d.Dv;
  g.Kc = d.Kc;
  g.C = d.C;
  g.eps = c.cfg->rms_eps;
  r = cu(q35pf::gdn(g, c.st));
  if (!r) r = pf_gemm(c, l->out_proj, g.yin, c.b16(c.L.o), nullptr, false);
  if (!r) r = pf_mlp(c, x_in, c.b16(c.L.o), l->post_ln, l->gate_proj, l->up_proj, l->down_proj, x_out);
  return r;
}

// The prefill's causal attention holds one kv-head's group of q-heads per CTA, in
// groups of 1, 2, 4 or 8 q-heads (the single-token forward takes any group).
int pf_fa_dims(const qwen35_config* cfg, const Dims& d) {
  const int r = check_fa_dims(cfg, d);
  if (r) return r;
  const uint32_t g = d.H / d.Hkv;
  return g == 1 || g == 2 || g == 4 || g == 8 ? QWEN35_OK : QWEN35_ERR_UNSUPPORTED;
}

// A prefill's KV cache: bf16 (contiguous or paged) or Turbo8, room for positions
// [p0, p0 + T).
int pf_kv_ok(const qwen35_kv_cache* kv, uint32_t p0, uint32_t T) {
  if (!kv_ok(kv)) return QWEN35_ERR_INVALID_ARGUMENT;
  if ((uint64_t)p0 + T > kv->capacity) return QWEN35_ERR_OUT_OF_RANGE;
  return QWEN35_OK;
}

}  // namespace

extern "C" {

int qwen35_prefill_gemm(const qwen35_qweight* w, const qwen35_bf16* X, qwen35_bf16* Y, uint32_t n_tokens,
                        int exact, void* scratch, size_t scratch_bytes, void* stream) {
  if (!w || !aligned16(X) || !aligned16(Y) || !aligned16(scratch) || scratch_bytes < 256)
    return QWEN35_ERR_INVALID_ARGUMENT;
  if (!qw_ok(*w, w->n, w->k) || w->n == 0 || w->k == 0 || w->k % 64 || n_tokens == 0 ||
      n_tokens > kMaxPrefillTokens)
    return QWEN35_ERR_INVALID_ARGUMENT;
  if (num_sms() <= 0) return QWEN35_ERR_CUDA;
  PfCtx c = {};
  c.s = static_cast<uint8_t*>(scratch);
  c.T = n_tokens;
  c.st = (cudaStream_t)stream;
  // a scratch with room for the split-K workspace after its first 256 bytes lets a
  // GEMM of few tiles split K
  c.ws = scratch_bytes >= 256 + q35pf::kGemmWorkspace ? reinterpret_cast<float*>(c.s + 256) : nullptr;
  return pf_gemm(c, *w, X, Y, nullptr, exact != 0);
}

size_t qwen35_prefill_scratch_bytes(const qwen35_config* cfg, uint32_t max_tokens) {
  Dims d;
  if (check_config(cfg, d) || max_tokens == 0 || max_tokens > kMaxPrefillTokens) return 0;
  return pf_layout(d, max_tokens).total;
}

int qwen35_prefill_full_attention(const qwen35_config* cfg, const qwen35_fa_layer* layer, void* scratch,
                                  size_t scratch_bytes, const qwen35_kv_cache* kv, const qwen35_bf16* x_in,
                                  qwen35_bf16* x_out, uint32_t cache_pos, uint32_t n_tokens, void* stream) {
  PfCtx c;
  int r = pf_begin(c, cfg, scratch, scratch_bytes, x_in, x_out, n_tokens, (cudaStream_t)stream);
  if (!r) r = pf_fa_dims(cfg, c.d);
  if (!r) r = check_fa_layer(layer, c.d);
  if (!r) r = pf_kv_ok(kv, cache_pos, n_tokens);
  if (r) return r;
  if (num_sms() <= 0) return QWEN35_ERR_CUDA;
  return pf_fa(c, layer, kv, x_in, x_out, cache_pos);
}

int qwen35_prefill_linear_attention(const qwen35_config* cfg, const qwen35_gdn_layer* layer, void* scratch,
                                    size_t scratch_bytes, const qwen35_gdn_state* state, const qwen35_bf16* x_in,
                                    qwen35_bf16* x_out, uint32_t n_tokens, void* stream) {
  PfCtx c;
  int r = pf_begin(c, cfg, scratch, scratch_bytes, x_in, x_out, n_tokens, (cudaStream_t)stream);
  if (!r) r = check_gdn_dims(c.d);
  if (!r) r = check_gdn_layer(layer, c.d);
  if (!r && (!state || !aligned16(state->conv_state) || !aligned16(state->gdn_state)))
    r = QWEN35_ERR_INVALID_ARGUMENT;
  if (r) return r;
  if (num_sms() <= 0) return QWEN35_ERR_CUDA;
  return pf_gdn(c, layer, state, x_in, x_out);
}

int qwen35_prefill_step(const qwen35_config* cfg, const qwen35_layer* layers, uint32_t num_layers, void* scratch,
                        size_t scratch_bytes, const qwen35_bf16* x_in, qwen35_bf16* x_out, uint32_t cache_pos,
                        uint32_t n_tokens, void* stream) {
  PfCtx c;
  int r = pf_begin(c, cfg, scratch, scratch_bytes, x_in, x_out, n_tokens, (cudaStream_t)stream);
  if (r) return r;
  if (!layers || num_layers == 0) return QWEN35_ERR_INVALID_ARGUMENT;
  for (uint32_t i = 0; i < num_layers && !r; ++i) {  // every layer checked before anything is enqueued
    const qwen35_layer& L = layers[i];
    if (L.kind == QWEN35_LAYER_FULL_ATTENTION) {
      r = pf_fa_dims(cfg, c.d);
      if (!r) r = check_fa_layer(L.fa, c.d);
      if (!r) r = pf_kv_ok(L.kv, cache_pos, n_tokens);
    } else if (L.kind == QWEN35_LAYER_LINEAR_ATTENTION) {
      r = check_gdn_dims(c.d);
      if (!r) r = check_gdn_layer(L.gdn, c.d);
      if (!r && (!L.state || !aligned16(L.state->conv_state) || !aligned16(L.state->gdn_state)))
        r = QWEN35_ERR_INVALID_ARGUMENT;
    } else {
      r = QWEN35_ERR_INVALID_ARGUMENT;
    }
  }
  if (r) return r;
  if (num_sms() <= 0) return QWEN35_ERR_CUDA;
  for (uint32_t i = 0; i < num_layers && !r; ++i) {
    const uint16_t* xi = i == 0 ? x_in : x_out;
    const qwen35_layer& L = layers[i];
    r = L.kind == QWEN35_LAYER_FULL_ATTENTION ? pf_fa(c, L.fa, L.kv, xi, x_out, cache_pos)
                                              : pf_gdn(c, L.gdn, L.state, xi, x_out);
  }
  return r;
}

}  // extern "C"
