// Persistent single-token decode kernel for Qwen3.5 decoder layers on sm_103a.
//
// One launch runs a program of layers: a single layer for the per-layer forwards
// of the pages "full_attention.rs" (forward_full_attention) and
// "linear_attention.rs" (forward_linear_attention), or the whole stack for a
// decode step. Each layer is a sequence of phases:
//   full attention:   [q|k|v GEMV + input RMSNorm] [split-KV attention with q/k
//                     norm, partial RoPE, KV append] [combine + sigmoid gate]
//                     [o_proj] [gate|up GEMV + residual + post RMSNorm]
//                     [down GEMV + SiLU gate + residual]
//   linear attention: [a|b|qkv|z GEMV + input RMSNorm] [conv1d + SiLU + L2 norm,
//                     gate, beta, gated delta rule] [out_proj + per-head RMSNorm
//                     + SiLU(z) gate] [gate|up ...] [down ...]
//
// The grid is one CTA per SM (a cooperative launch, so all CTAs are resident):
// one producer warp and twelve consumer warps. The producer walks the CTA's
// whole schedule of the launch, every weight tile of every GEMV phase and every
// K/V tile of every attention phase, and streams them with bulk (TMA-engine)
// copies into a byte-addressed shared-memory ring, never waiting for a phase
// boundary: weights and old cache rows do not depend on the phases before them.
// It also stages each linear-attention layer's state block and conv inputs while
// that layer's input projection streams. Consumers run the phases in order; a
// phase's results reach the other CTAs as tagged words that the next phase polls
// (no grid barrier, see "hand-over between CTAs" below).
//
// Phase functions are kept out of line (one call per phase) and read the
// program header, the current layer and the current GEMV from static shared
// memory.
//
// GEMV phases (the int8 group-64 affine QuantWeights::gemv family): each CTA owns
// a balanced contiguous range of rows of the phase's concatenated matrices. The
// input vector is formed once per CTA (RMSNorm, residual add + RMSNorm, SiLU
// gating, per-head RMSNorm with SiLU(z) gating) and kept in shared memory as
// 16-bit fixed point per 16-element chunk (x ~= q 2^(e-15), q = 256 hi + lo, a
// power-of-two scale per chunk: exact for every element within 2^8 of its chunk's
// largest, since bf16 carries 8 significant bits). Each consumer lane holds its
// chunks in registers; a 16-code chunk costs eight dp4a giving sum (c - 128) q
// exactly in int32, and the group identity
//   sum_k (s c_k + b) x_k = s sum_k (c_k - 128) x_k + (b + 128 s) sum_k x_k
// applies scale and bias once per chunk (the -128 offset avoids cancelling two
// terms ~128x larger than the result when b is close to -128 s). Each tile's row
// is reduced across its warp into shared partial sums; one epilogue per phase
// stores the rows.
#pragma once

#include <algorithm>
#include <cstddef>

#include <cuda_fp16.h>

#include "common.cuh"
#include "decode.h"

namespace q35 {
namespace {

constexpr int NCW = kDecConsumerWarps;
constexpr int NCT = NCW * 32;
constexpr uint32_t FULLMASK = 0xffffffffu;
constexpr int kTS = 8;      // tokens per attention tile
constexpr int kMaxKc = 8;

enum PhaseType { kPhGemv = 0, kPhAttn = 1, kPhCombine = 2, kPhGdn = 3 };
// kWhtGate: a Turbo8 layer's o_proj input: the attention output, in the cache's
// rotated basis, rotated back per head (bf16), times sigmoid(gate) (bf16)
// kQuantized: the input arrives already quantised (16-bit codes and chunk exponents
// formed by the phase that produced it)
enum Pro { kPlain = 0, kRms = 1, kAddRms = 2, kSiluMul = 3, kHeadNormSilu = 4, kWhtGate = 5, kQuantized = 6 };

__device__ __forceinline__ int n_phases(int kind) { return kind == kLayerFA ? 6 : kind == kLayerGDN ? 5 : 1; }
__device__ __forceinline__ int phase_type(int kind, int p) {
  if (kind == kLayerFA) return p == 1 ? kPhAttn : p == 2 ? kPhCombine : kPhGemv;
  if (kind == kLayerGDN) return p == 1 ? kPhGdn : kPhGemv;
  return kPhGemv;
}

// ------------------------------------------------------------------ shared memory

extern __shared__ __align__(1024) uint8_t smem_raw[];

struct Smem {
  uint8_t* ring;
  uint64_t* full;
  uint64_t* empty;
  uint32_t* toff;    // ring offset of the tile in each slot (written before its copies)
  uint32_t* tmeta;  // GEMV tiles: first row | rows << 24
  float* misc;     // 256 floats (1 KiB): reductions, gate/beta
  uint8_t* uni;    // per-phase buffer (the launch's union_bytes)
};

__device__ __forceinline__ Smem smem_map(uint8_t* base, uint32_t ring_bytes) {
  Smem s;
  s.ring = base;
  s.full = reinterpret_cast<uint64_t*>(base + ring_bytes);
  s.empty = s.full + kDecSlots;
  s.toff = reinterpret_cast<uint32_t*>(s.empty + kDecSlots);
  s.tmeta = s.toff + kDecSlots;
  s.misc = reinterpret_cast<float*>(s.tmeta + kDecSlots);
  s.uni = reinterpret_cast<uint8_t*>(s.misc + 256);
  return s;
}
// The consumers' ring position travels through the phase functions by value: the
// count of tiles taken, with kDeadBit set once a wait has run out (a reference
// would put it in local memory).
constexpr uint32_t kDeadBit = 0x80000000u;
// The tile the consumers take as their it-th: its slot and the slot's phase parity.
__device__ __forceinline__ uint32_t slot_of(uint32_t it) { return it % kDecSlots; }
__device__ __forceinline__ uint32_t parity_of(uint32_t it) { return (it / kDecSlots) & 1; }

__device__ __forceinline__ void consumer_sync() { named_barrier(1, NCT); }

// Per-CTA state in static shared memory, addressed directly by every phase
// function (a shared-space address instead of a generic pointer parameter):
// the program's header (everything before the layer table, copied when the
// launch starts) and the current layer's description.
constexpr uint32_t kHeadBytes = (offsetof(Program, layers) + 3) / 4 * 4;
static_assert(offsetof(Program, layers) % 8 == 0, "layer table alignment");
static_assert(sizeof(Program) <= 32764, "kernel parameter block");
__shared__ __align__(16) uint8_t s_head[kHeadBytes];
// The descriptions the consumers work from, double-buffered so that the helper
// warp forms the next phase's while the consumers run the current one:
// the layer by layer parity (as the program gives it, s_lay0, and rebased to the
// current sequence of a batch, s_lay), the GEMV by phase parity (s_gv, below).
// s_sel: bit 0 the current phase's buffer, bit 1 the current layer's.
__shared__ LayerDesc s_lay[2];
__shared__ LayerDesc s_lay0[2];
__shared__ uint32_t s_sel;
__shared__ uint32_t s_dead_cta;  // a consumer wait on the helper ran out: no more ring reads
__device__ __forceinline__ const Program& prog() { return *reinterpret_cast<const Program*>(s_head); }
__device__ __forceinline__ LayerDesc& cur_layer() { return s_lay[(s_sel >> 1) & 1]; }
__device__ __forceinline__ LayerDesc& cur_layer0() { return s_lay0[(s_sel >> 1) & 1]; }
__device__ __forceinline__ Smem smem_map(uint8_t* base) { return smem_map(base, prog().ring_bytes); }

// The sequence the consumers are working on (a batch runs each phase for its
// sequences back to back): its scratch block, input and output vectors. The
// layer's cache pointers in s_layer are rebased to it as well.
struct SeqCtx {
  uint8_t* scratch;
  const uint16_t* x_in;
  uint16_t* x_out;
  uint32_t b;
};
__shared__ SeqCtx s_seq;
__shared__ int32_t s_pos[kMaxBatch];  // each sequence's device position, read at launch

// Row stride, in bf16 elements, of a Turbo8 cache's scales: one per 16 elements of
// a token's row, padded to 16 bytes.
__host__ __device__ inline uint32_t turbo8_sstride(uint32_t Hkv, uint32_t D) { return (Hkv * D / 16 + 7) / 8 * 8; }

// Sequence b's scratch block and its caches in layer L (the caller's [B][...] arrays).
__device__ __forceinline__ uint8_t* seq_scratch(const Program& P, uint32_t b) {
  return P.scratch + (size_t)b * P.seq_stride;
}
__device__ __forceinline__ void seq_caches(const Program& P, LayerDesc& L, uint32_t b) {
  if (L.kind == kLayerFA && L.btab) {  // paged: one shared pool, a table per sequence
    L.btab += (size_t)(L.capacity >> L.bt_shift) * b;
  } else if (L.kind == kLayerFA) {
    const bool t8 = L.kv_dtype == kKvTurbo8;
    const size_t kv = (size_t)L.capacity * P.Hkv * P.D * (t8 ? 1 : 2) * b;  // bytes
    L.kc += kv;
    L.vc += kv;
    if (t8) {
      const size_t sc = (size_t)L.capacity * turbo8_sstride(P.Hkv, P.D) * b;
      L.ks += sc;
      L.vs += sc;
    }
  } else if (L.kind == kLayerGDN) {
    L.conv_state += (size_t)P.C * P.Kc * b;
    L.ssm += (size_t)P.Hv * P.Dk * P.Dv * b;
  }
}

// The cache row holding logical token t: t itself, or for a paged cache its row in
// the pool block the table names.
__device__ __forceinline__ size_t kv_row(const LayerDesc& L, uint32_t t) {
  if (!L.btab) return t;
  const uint32_t mask = (1u << L.bt_shift) - 1u;
  return ((size_t)(uint32_t)__ldg(L.btab + (t >> L.bt_shift)) << L.bt_shift) | (t & mask);
}

// misc[255]: the device position, read once per CTA when the launch starts (every
// phase of the launch sees the same value although CTA 0 advances it at the end)
__device__ __forceinline__ int32_t launch_pos(uint32_t b) { return s_pos[b]; }

// ------------------------------------------------------------------ hand-over between CTAs
//
// No grid barrier separates the phases. A phase's results that other CTAs read are
// tagged words (common.cuh): each reader polls the words it needs until they carry
// the tag of the phase that writes them, so it starts as soon as its own inputs
// are in, one L2 round trip after they are stored. Every phase of a layer reads
// results of all CTAs of the phase before it (the full input vector of a
// projection, the partials of every split, every q-head's rows), so no CTA can be
// more than one phase ahead of another, and a buffer is rewritten only after every
// CTA has finished reading its previous contents: each phase's outputs are computed
// from the values its loads return, so those loads have completed before any of its
// stores is issued (no fence is needed for that order; one measured 0.4 us per
// phase). Tags are the launch's phase index + 1.

// The launch's limit for bounded waits (ns).
__device__ __forceinline__ uint64_t wait_limit() { return prog().wait_ns; }
// The limit for the producer's final drain of its copies in flight: at least the
// default, so that no copy into shared memory outlives the CTA.
__device__ __forceinline__ uint64_t drain_limit() { return prog().wait_ns > kWaitNs ? prog().wait_ns : kWaitNs; }

__device__ __forceinline__ uint32_t phase_tag(uint32_t ph) { return ph + 1u; }

// Poll N groups of 4 tagged words, w[i] loaded from p[i] and expected to carry
// tag t[i] (t[i] == 0: nothing to poll), until every group carries its tag. Each
// round re-loads all the groups still missing together, so a round costs one L2
// round trip however many are missing. False when the wait runs out.
template <int N>
__device__ __forceinline__ bool settle4(const uint32_t* const (&p)[N], const uint32_t (&t)[N], uint4 (&w)[N]) {
  uint32_t todo = 0;
#pragma unroll
  for (int i = 0; i < N; ++i)
    if (t[i] && !tags4_are(w[i], t[i])) todo |= 1u << i;
  if (!todo) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t n = 1;; ++n) {
    __nanosleep(64);
#pragma unroll
    for (int i = 0; i < N; ++i)
      if ((todo >> i) & 1u) w[i] = ld_tagged4(p[i]);
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (((todo >> i) & 1u) && tags4_are(w[i], t[i])) todo &= ~(1u << i);
    if (!todo) return true;
    if (global_ns() - t0 > wait_limit() || ((n & 15) == 0 && timed_out(prog().status))) return false;
  }
}
// The same for N single tagged words.
template <int N>
__device__ __forceinline__ bool settle1(const uint32_t* const (&p)[N], const uint32_t (&t)[N], uint32_t (&w)[N]) {
  uint32_t todo = 0;
#pragma unroll
  for (int i = 0; i < N; ++i)
    if (t[i] && !tag_is(w[i], t[i])) todo |= 1u << i;
  if (!todo) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t n = 1;; ++n) {
    __nanosleep(64);
#pragma unroll
    for (int i = 0; i < N; ++i)
      if ((todo >> i) & 1u) w[i] = ld_tagged(p[i]);
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (((todo >> i) & 1u) && tag_is(w[i], t[i])) todo &= ~(1u << i);
    if (!todo) return true;
    if (global_ns() - t0 > wait_limit() || ((n & 15) == 0 && timed_out(prog().status))) return false;
  }
}

// 16 input values of a chunk: tagged words (4 x uint4) or, for the caller's own
// bf16 vectors (tag 0), 16 bf16 (2 x uint4). Issue, settle (settle4 over the
// chunks' groups), then read out.
struct Chunk16 {
  uint4 w[4];
};
__device__ __forceinline__ void chunk_issue(const void* base, uint32_t tag, uint32_t c, Chunk16& ch) {
  if (tag) {
    const uint32_t* p = static_cast<const uint32_t*>(base) + (size_t)c * 16;
#pragma unroll
    for (int k = 0; k < 4; ++k) ch.w[k] = ld_tagged4(p + 4 * k);
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + (size_t)c * 16);
    ch.w[0] = p[0];
    ch.w[1] = p[1];
    ch.w[2] = ch.w[3] = make_uint4(0u, 0u, 0u, 0u);
  }
}
// The poll list entries of chunk c (tag 0 or inactive: none), at index i0..i0+3.
template <int N>
__device__ __forceinline__ void chunk_pend(const void* base, uint32_t tag, uint32_t c, bool active,
                                           const uint32_t* (&p)[N], uint32_t (&t)[N], int i0) {
  const uint32_t* q = static_cast<const uint32_t*>(base) + (size_t)c * 16;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    p[i0 + k] = q + 4 * k;
    t[i0 + k] = active ? tag : 0u;
  }
}
__device__ __forceinline__ void chunk_values(const Chunk16& ch, uint32_t tag, float* x) {
  if (tag) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[4 * k] = tag_value(ch.w[k].x);
      x[4 * k + 1] = tag_value(ch.w[k].y);
      x[4 * k + 2] = tag_value(ch.w[k].z);
      x[4 * k + 3] = tag_value(ch.w[k].w);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint4 u = ch.w[k];
      x[8 * k] = bf16lo(u.x); x[8 * k + 1] = bf16hi(u.x);
      x[8 * k + 2] = bf16lo(u.y); x[8 * k + 3] = bf16hi(u.y);
      x[8 * k + 4] = bf16lo(u.z); x[8 * k + 5] = bf16hi(u.z);
      x[8 * k + 6] = bf16lo(u.w); x[8 * k + 7] = bf16hi(u.w);
    }
  }
}
// One tagged value (polled); records a timeout in the status word.
__device__ __forceinline__ float tagged_value(const uint32_t* p, uint32_t tag) {
  uint32_t w;
  if (!ld_tagged_wait(p, tag, w, wait_limit(), prog().status)) set_status(prog().status, kStatusTimeout);
  return tag_value(w);
}
// Store 16 values of a chunk as tagged words (already rounded to bf16 or not).
__device__ __forceinline__ void chunk_store_tagged(uint32_t* dst, const float* v, uint32_t tag) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    st_tagged4(dst + 4 * k, make_uint4(tag_word(v[4 * k], tag), tag_word(v[4 * k + 1], tag),
                                       tag_word(v[4 * k + 2], tag), tag_word(v[4 * k + 3], tag)));
}
__device__ __forceinline__ void chunk_store_bf16(uint16_t* dst, const float* v) {
  uint32_t pk[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) pk[j] = (uint32_t)to_bf16(v[2 * j]) | ((uint32_t)to_bf16(v[2 * j + 1]) << 16);
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  d[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
}

// ------------------------------------------------------------------ bf16 helpers

// bf16 pair {lo, hi} (round to nearest).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ void unpack8(const uint4 u, float* x) {
  x[0] = bf16lo(u.x); x[1] = bf16hi(u.x);
  x[2] = bf16lo(u.y); x[3] = bf16hi(u.y);
  x[4] = bf16lo(u.z); x[5] = bf16hi(u.z);
  x[6] = bf16lo(u.w); x[7] = bf16hi(u.w);
}
template <int EPL>
__device__ __forceinline__ void load_row(const uint16_t* p, float* x) {
  if constexpr (EPL == 8) {
    unpack8(*reinterpret_cast<const uint4*>(p), x);
  } else if constexpr (EPL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    x[0] = bf16lo(u.x); x[1] = bf16hi(u.x); x[2] = bf16lo(u.y); x[3] = bf16hi(u.y);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    x[0] = bf16lo(u); x[1] = bf16hi(u);
  }
}

// Sum over the 32 lanes of v[0..NV-1] (NV a power of two up to 32), each step handing half of
// the remaining values to the partner lane; lane L ends with the total of
// v[L >> (5 - log2 NV)].
template <int NV>
__device__ __forceinline__ float reduce_transposed(float* v, uint32_t lane) {
  int n = NV;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    if (n > 1) {
      const bool up = lane & o;
      const int h = n / 2;
#pragma unroll
      for (int i = 0; i < NV / 2; ++i) {
        if (i < h) {
          const float keep = up ? v[i + h] : v[i];
          const float send = up ? v[i] : v[i + h];
          v[i] = keep + __shfl_xor_sync(FULLMASK, send, o);
        }
      }
      n = h;
    } else {
      v[0] += __shfl_xor_sync(FULLMASK, v[0], o);
    }
  }
  return v[0];
}

// ------------------------------------------------------------------ GEMV phases

struct XQ {
  uint32_t hi[4], lo[4];
  int qsum128;  // 128 * sum q
  float scale;  // 2^(e-15)
};

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ int sat16(float x) {  // round to nearest even, saturate to int16
  short r;
  asm("cvt.rni.sat.s16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void quantize16(const float* v, XQ& q) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  // amax = m 2^e, 0.5 <= m < 1, e = E - 126 for the biased exponent E; scale 2^(e-15).
  // A chunk whose largest element is below 2^-112 counts as zero.
  const uint32_t E = __float_as_uint(amax) >> 23;
  const bool nz = E >= 15;
  const float up = nz ? __uint_as_float((268u - E) << 23) : 0.f;  // 2^(15-e)
  q.scale = nz ? __uint_as_float((E - 14u) << 23) : 0.f;
  int qs = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    int t[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      t[j] = sat16(v[4 * w + j] * up);
      qs += t[j];
    }
    // byte j of lo / hi = the low / high byte of element 4w + j
    q.lo[w] = __byte_perm(__byte_perm(t[0], t[1], 0x0040), __byte_perm(t[2], t[3], 0x0040), 0x5410);
    q.hi[w] = __byte_perm(__byte_perm(t[0], t[1], 0x0051), __byte_perm(t[2], t[3], 0x0051), 0x5410);
  }
  q.qsum128 = 128 * qs;
}

// sum over the chunk of (c - 128) * q, exact: 256 * sum(c * hi) + sum(c * lo) - 128 * sum(q)
__device__ __forceinline__ int dot16i(const uint4 w, const XQ& q) {
  int ah = 0;
  uint32_t al = (uint32_t)(-q.qsum128);
  ah = dp4a_us(w.x, q.hi[0], ah);
  al = dp4a_uu(w.x, q.lo[0], al);
  ah = dp4a_us(w.y, q.hi[1], ah);
  al = dp4a_uu(w.y, q.lo[1], al);
  ah = dp4a_us(w.z, q.hi[2], ah);
  al = dp4a_uu(w.z, q.lo[2], al);
  ah = dp4a_us(w.w, q.hi[3], ah);
  al = dp4a_uu(w.w, q.lo[3], al);
  return ah * 256 + (int)al;
}


// Warps per row W (a divisor of the consumer warps) and 16-element chunks per lane
// (at most 5): the fewest wasted chunk slots, then the fewest warps per row.
__host__ __device__ inline void pick_split(uint32_t nch, uint32_t& W, uint32_t& cpl) {
  W = 0;
  cpl = 0;
  uint32_t best = 0xffffffffu;
  for (uint32_t w = 1; w <= (uint32_t)NCW; ++w) {
    if (NCW % w) continue;
    const uint32_t c = (nch + 32 * w - 1) / (32 * w);
    if (c > 5) continue;
    const uint32_t waste = c * 32 * w - nch;
    if (waste < best) {
      best = waste;
      W = w;
      cpl = c;
    }
  }
}

// A batch's projections run on the tensor cores as m16n8k16 f16 products with fp32
// sums: m = up to 16 weight rows of a tile (codes converted exactly to f16), n = the
// pass's sequences, each sequence's input staged in f16 with a power-of-two scale
// per 64-column group. Tiles hold up to kBatchRowsMax rows of the full K; rows of
// the staged inputs are padded by kXPadH elements (16 bytes: a quarter-warp's lanes
// then read distinct banks). Teams of warps take the tiles in turn: the warps of a
// team share a tile's column groups and add their row sums in a fixed order.
constexpr uint32_t kBatchRowsMax = 16;
constexpr uint32_t kXPadH = 8;
// each warp's 16 x 8 partial sums, then the down projection's residual rows of the
// pass's sequences ([CTA rows][bs], at most 1 KiB: rows <= 32)
constexpr uint32_t kBatchResid = 1024;
constexpr uint32_t kBatchPart = NCW * 128 * 4 + kBatchResid;
#ifndef QWEN35_TEAM_SLACK
#define QWEN35_TEAM_SLACK 1
#endif
__host__ __device__ inline uint32_t batch_rows(uint32_t K) {
  const uint32_t gs = ((K / 64 + 7) / 8) * 8;
  uint32_t r = kBatchRowsMax;
  while (r > 1 && (r * K + 15) / 16 * 16 + 4 * r * gs > (uint32_t)kDecTileMax) r /= 2;
  return r;
}
// Phase-buffer bytes per sequence of a pass: the staged f16 input and the group
// scales and sums.
__host__ __device__ inline uint32_t batch_seq_bytes(uint32_t K) { return 2 * (K + kXPadH) + 8 * (K / 64); }
// Teams per CTA: a divisor of the consumer warps, at most the tiles the ring holds at
// once less a slack (tiles in flight while every team computes), at most the tiles.
__host__ __device__ inline uint32_t batch_teams(uint32_t span, uint32_t ntiles, uint32_t ring_bytes) {
  const uint32_t fit = ring_bytes / span;
  uint32_t cap = fit > QWEN35_TEAM_SLACK ? fit - QWEN35_TEAM_SLACK : 1u;
  if (ntiles < cap) cap = ntiles > 0 ? ntiles : 1u;
  for (uint32_t d = cap; d > 1; --d)
    if (NCW % d == 0) return d;
  return 1;
}

struct Gemv {
  QMat seg[4];
  uint8_t* out[4];   // each segment's output: tagged words, or bf16 (out_tag 0)
  uint32_t row0[5];  // prefix sums of the segments' rows
  uint32_t nseg, K;
  int pro, epi;
  // inputs: tagged words expected to carry tag_a / tag_b / tag_r, or the caller's
  // bf16 vectors when the tag is 0 (a, b, resid_in); nw: norm weights (bf16)
  const void *a, *b, *resid_in;
  uint32_t tag_a, tag_b, tag_r;
  const uint16_t* nw;
  uint32_t* resid_out;  // x_resid (tagged, written by CTA 0 with tag out_tag)
  uint32_t out_tag;     // tag of the outputs; 0: bf16 into the caller's vector
  uint16_t* dump;       // debug: CTA 0 stores the formed input here (bf16), or null
  // the gate|up phase of a linear-attention layer also shifts the q/k channels' conv
  // state (of sequence 0; a batch's others follow at C * Kc strides), qkv tagged conv_tag
  float* conv_shift;
  uint32_t conv_tag;
  uint32_t head_dim;
  uint32_t W, cpl, R, gstride, scale_off, bias_off;
  uint32_t rb, re, ntiles;  // this CTA's rows [rb, re) and its tile count
  // a batch: sequence b's vectors at the pointers above + b * these strides
  // (elements), bs sequences per pass over the weights, npass passes
  uint32_t sa, sb, sres_in, sres_out, sout[4];
  uint32_t bs, npass, T;  // T: teams of warps per CTA (a batch)
  // epi 3 (a single sequence's gate|up): rows pr0 .. pr0 + pn - 1 of gate and of up
  // (whole 16-row chunks), partial sums [gate rows | up rows]
  uint32_t pr0, pn;
};

__shared__ Gemv s_gv[2];  // GEMV descriptions by phase parity
__device__ __forceinline__ Gemv& cur_gemv() { return s_gv[s_sel & 1]; }
// Per ring slot: where a GEMV tile's first row is stored, as an element offset
// from the phase's first output (a phase's outputs are consecutive buffers of one
// scratch block in segment order, or a single output), written by the producer with
// the tile's other words; the row loop stores whole rows without a segment lookup.
__shared__ uint32_t s_tout[kDecSlots];

__device__ __forceinline__ uint32_t out_esz(const Gemv& g) { return g.out_tag ? 4u : 2u; }

__device__ __forceinline__ void gemv_add(Gemv& g, const QMat& m, void* out, uint32_t stride) {
  g.seg[g.nseg] = m;
  g.out[g.nseg] = static_cast<uint8_t*>(out);
  g.sout[g.nseg] = stride;
  g.row0[g.nseg + 1] = g.row0[g.nseg] + m.n;
  ++g.nseg;
}

// Store output element i of segment sg (sequence b of a batch) as a tagged word or
// as bf16.
__device__ __forceinline__ void gemv_store(const Gemv& g, uint32_t sg, size_t i, float y) {
  if (g.out_tag) st_tagged(reinterpret_cast<uint32_t*>(g.out[sg]) + i, tag_word(y, g.out_tag));
  else reinterpret_cast<uint16_t*>(g.out[sg])[i] = to_bf16(y);
}

// The GEMV of phase p of layer l, written into g (shared memory: a returned struct
// would go through local memory). ph0 is the launch's phase index of the layer's
// phase 0 (for the tags); the last layer's down projection writes the caller's
// x_out, the others a stack's internal output vector. The program's shape table
// holds the split computed on the host, so this runs in a few hundred cycles on
// the thread that fills it.
__device__ __noinline__ void gemv_of(const Program& P, const LayerDesc& L, uint32_t l, int p, uint32_t sq,
                                     uint32_t ph0, Gemv& g) {
  g.nseg = 0;
  g.row0[0] = 0;
  g.b = nullptr;
  g.resid_in = nullptr;
  g.nw = nullptr;
  g.resid_out = nullptr;
  g.dump = nullptr;
  g.head_dim = 0;
  g.epi = 0;
  g.tag_a = g.tag_b = g.tag_r = 0;
  g.conv_shift = nullptr;
  g.conv_tag = 0;
  g.sa = g.sb = g.sres_in = g.sres_out = 0;
  uint8_t* S = seq_scratch(P, sq);
  const ScratchMap& m = P.sm;
  const uint16_t* x_in = P.x_in + (size_t)sq * P.E;
  uint16_t* x_out = P.x_out + (size_t)sq * P.E;
  auto tw = [&](uint32_t off) { return reinterpret_cast<uint32_t*>(S + off); };  // tagged words
  auto dmp = [&](uint32_t off) { return P.dump && blockIdx.x == 0 ? reinterpret_cast<uint16_t*>(S + off) : nullptr; };
  const uint32_t SS = P.seq_stride / 4, SX = P.E;  // per-sequence strides: scratch words, vectors
  const bool fa = L.kind == kLayerFA;
  const int mlp0 = fa ? 4 : 3;  // the gate|up phase
  const uint32_t tag_out = phase_tag(ph0 + p);
  // the layer's input: the caller's vector for layer 0, else the last layer's output
  const void* xin = l == 0 ? static_cast<const void*>(x_in) : static_cast<const void*>(tw(m.xa));
  const uint32_t tag_xin = l == 0 ? 0u : phase_tag(ph0 - 1);
  const uint32_t sxin = l == 0 ? SX : SS;
  g.out_tag = tag_out;
  if (L.kind == kLayerGemv || L.kind == kLayerHead) {
    g.K = P.E;
    g.pro = L.kind == kLayerHead ? kRms : kPlain;
    g.a = x_in;
    g.sa = SX;
    g.nw = L.input_ln;
    g.out_tag = 0;
    gemv_add(g, L.m[0], x_out, SX);
  } else if (p == 0) {
    g.K = P.E;
    g.pro = kRms;
    g.a = xin;
    g.tag_a = tag_xin;
    g.sa = sxin;
    g.nw = L.input_ln;
    g.dump = dmp(m.x_norm);
    if (fa) {
      gemv_add(g, L.m[0], tw(m.q_full), SS);
      gemv_add(g, L.m[1], tw(m.k), SS);
      gemv_add(g, L.m[2], tw(m.v), SS);
    } else {
      gemv_add(g, L.m[0], tw(m.dt_raw), SS);
      gemv_add(g, L.m[1], tw(m.b_raw), SS);
      gemv_add(g, L.m[2], tw(m.qkv), SS);
      gemv_add(g, L.m[3], tw(m.z), SS);
    }
  } else if (p == mlp0) {
    g.K = P.E;
    g.pro = kAddRms;
    g.a = xin;
    g.tag_a = tag_xin;
    g.sa = sxin;
    g.b = tw(fa ? m.o : m.out);
    g.tag_b = phase_tag(ph0 + p - 1);
    g.sb = SS;
    g.nw = L.post_ln;
    g.resid_out = tw(m.x_resid);
    g.sres_out = SS;
    g.dump = dmp(m.x_norm2);
    if (!fa) {  // the q/k conv state: every linear-attention CTA has read it two phases back
      g.conv_shift = L.conv_state;
      g.conv_tag = phase_tag(ph0);
    }
    if (P.batch <= 1) {  // matching gate and up rows per CTA; h = SiLU(gate) * up, quantised
      g.epi = 3;
      gemv_add(g, L.m[4], tw(m.hq), SS);
      gemv_add(g, L.m[5], tw(m.he), SS);
    } else {
      gemv_add(g, L.m[4], tw(m.g), SS);
      gemv_add(g, L.m[5], tw(m.u), SS);
    }
  } else if (p == mlp0 + 1) {
    g.K = P.I;
    g.pro = kSiluMul;
    g.epi = 1;
    g.a = tw(m.g);
    g.tag_a = phase_tag(ph0 + p - 1);
    g.sa = SS;
    g.b = tw(m.u);
    g.tag_b = g.tag_a;
    g.sb = SS;
    if (P.batch <= 1) {  // h's codes and chunk exponents from the gate|up phase
      g.pro = kQuantized;
      g.a = tw(m.hq);
      g.b = tw(m.he);
    }
    g.resid_in = tw(m.x_resid);
    g.tag_r = g.tag_a;
    g.sres_in = SS;
    if (l + 1 == P.n_layers) {
      g.out_tag = 0;
      gemv_add(g, L.m[6], x_out, SX);
    } else {
      gemv_add(g, L.m[6], tw(m.xa), SS);
    }
  } else if (fa) {  // p == 3: o_proj
    g.K = P.H * P.D;
    g.pro = kPlain;
    g.a = tw(m.ga);
    g.tag_a = phase_tag(ph0 + 2);
    g.sa = SS;
    if (L.kv_dtype == kKvTurbo8) {  // the attention output is still rotated: back, then the gate
      g.pro = kWhtGate;
      g.b = tw(m.q_full);  // head h's gate at q_full[h * 2D + D + d]
      g.tag_b = phase_tag(ph0);
      g.sb = SS;
      g.head_dim = P.D;
    }
    gemv_add(g, L.m[3], tw(m.o), SS);
  } else {  // p == 2: out_proj on silu(z) * RMSNorm_head(y)
    g.K = P.Z;
    g.pro = kHeadNormSilu;
    g.a = tw(m.y);
    g.tag_a = phase_tag(ph0 + 1);
    g.sa = SS;
    g.b = tw(m.z);
    g.tag_b = phase_tag(ph0);
    g.sb = SS;
    g.nw = L.norm_weight;
    g.head_dim = P.Dv;
    g.dump = dmp(m.y_norm);
    gemv_add(g, L.m[7], tw(m.out), SS);
  }
  const GemvShape sh = P.shapes[L.kind < kShapeKinds ? L.kind : 0][p];
  g.W = sh.W;
  g.cpl = sh.cpl;
  g.R = sh.R;
  g.gstride = ((g.K / 64 + 7) / 8) * 8;
  g.scale_off = (g.R * g.K + 15) / 16 * 16;
  g.bias_off = g.scale_off + g.R * g.gstride * 2;
  g.bs = sh.bs;
  g.npass = sh.npass;
  // a balanced contiguous range of rows per CTA (rows < 2^24, CTAs < 2^8: 32-bit
  // products), cut into R-row tiles per segment
  const uint32_t total = g.row0[g.nseg];
  g.rb = total * blockIdx.x / gridDim.x;
  g.re = total * (blockIdx.x + 1) / gridDim.x;
  g.ntiles = 0;
  g.pr0 = g.pn = 0;
  if (g.epi == 3) {  // a balanced range of whole 16-row chunks of gate, the same of up
    const uint32_t nch = g.seg[0].n / 16, c0 = nch * blockIdx.x / gridDim.x, c1 = nch * (blockIdx.x + 1) / gridDim.x;
    g.pr0 = 16 * c0;
    g.pn = 16 * (c1 - c0);
    g.rb = 0;
    g.re = 2 * g.pn;
    g.ntiles = 2 * ((g.pn + g.R - 1) / g.R);
  } else {
    for (uint32_t sg = 0; sg < g.nseg; ++sg) {
      const uint32_t lo = max(g.rb, g.row0[sg]), hi = min(g.re, g.row0[sg + 1]);
      if (hi > lo) g.ntiles += (hi - lo + g.R - 1) / g.R;
    }
  }
  g.T = P.batch > 1 ? batch_teams(g.bias_off + g.R * g.gstride * 2, g.ntiles, P.ring_bytes) : 1u;
}

// The shape-only part of every GEMV phase of the program (host).
void fill_shapes(Program& P) {
  for (int kind = 0; kind < kShapeKinds; ++kind)
    for (int p = 0; p < kShapePhases; ++p) {
      uint32_t K = 0;
      if (kind == kLayerFA) K = p == 0 || p == 4 ? P.E : p == 3 ? P.H * P.D : p == 5 ? P.I : 0;
      else if (kind == kLayerGDN) K = p == 0 || p == 3 ? P.E : p == 2 ? P.Z : p == 4 ? P.I : 0;
      else K = p == 0 ? P.E : 0;
      GemvShape& sh = P.shapes[kind][p];
      sh = GemvShape{};
      if (K == 0 || K % 64) continue;
      uint32_t W = 0, cpl = 0;
      pick_split(K / 16, W, cpl);
      if (W == 0) continue;
      const uint32_t R = P.batch > 1 ? batch_rows(K) : NCW / W;  // a batch: tensor-core tiles
      // a batch: as many sequences per pass over the weights as their staged inputs
      // fit in the phase buffer beside the teams' partial sums
      uint32_t bs = P.batch > 1 ? std::min(P.batch, (P.union_bytes - kBatchPart) / batch_seq_bytes(K)) : 1u;
      if (bs == 0) bs = 1;
      sh.W = (uint8_t)W;
      sh.cpl = (uint8_t)cpl;
      sh.R = (uint8_t)R;
      sh.bs = (uint8_t)bs;
      sh.npass = (uint8_t)((P.batch + bs - 1) / bs);
    }
}

// ------------------------------------------------------------------ phase descriptions

// Where the consumers are and what the helper warp has prepared: `entered` = the
// launch phase index the consumers are in + 1 (written by consumer thread 0 at the
// phase's entry), `prepped` = the phases whose descriptions are formed (the helper
// forms phase ph + 1's while the consumers run phase ph); the program's layer
// table (parameter space).
struct PhaseState {
  const LayerDesc* layers;
  uint32_t entered, prepped;
};
__shared__ PhaseState s_ph;

__device__ __forceinline__ uint32_t ld_volatile_shared(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_volatile_shared(uint32_t* p, uint32_t v) {
  asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}

// One warp: the descriptions of phase p of layer l (launch phase ph; the layer's
// first phase ph0) into the buffers of their parity: the layer's (copied from the
// parameter block at its first phase) and the GEMV's.
__device__ __noinline__ void form_phase(uint32_t l, uint32_t p, uint32_t ph, uint32_t ph0) {
  const Program& P = prog();
  const uint32_t lane = threadIdx.x & 31;
  if (p == 0) {  // a few words per lane
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&s_ph.layers[l]);
    uint32_t* d0 = reinterpret_cast<uint32_t*>(&s_lay0[l & 1]);
    uint32_t* d1 = reinterpret_cast<uint32_t*>(&s_lay[l & 1]);
    for (uint32_t i = lane; i < sizeof(LayerDesc) / 4; i += 32) {
      const uint32_t v = src[i];
      d0[i] = v;
      d1[i] = v;
    }
    __syncwarp();
  }
  if (lane == 0 && phase_type(s_lay0[l & 1].kind, p) == kPhGemv) gemv_of(P, s_lay0[l & 1], l, p, 0, ph0, s_gv[ph & 1]);
  __syncwarp();
}

// Forward declaration (defined with the linear-attention phase).
__device__ __noinline__ void conv_shift_qk(float* conv_state, const uint8_t* scratch, uint32_t tag);

// The CTA's partial row sums of a GEMV phase ([W][rows], one slice per K-part of
// a row) and, for the down projection, its residual rows ([rows]): shared memory
// after the input chunks.
__device__ __forceinline__ float* gemv_partials(const Smem& sh, uint32_t nch) {
  return reinterpret_cast<float*>(sh.uni + nch * 48);
}

// The down projection's input when the gate|up phase has already quantised it
// (kQuantized): chunk c's 16-bit codes are tagged words hq[16c .. 16c + 15] (code
// in the high half) and its exponent the tagged word he[c]; the chunks go into
// shared memory in the layout the row loop reads, with the same bits quantize16
// would have given (the gate|up phase ran it on the same values).
__device__ __noinline__ void gemv_prologue_quantized(unsigned long long* tr) {
  const Program& P = prog();
  const Gemv& g = cur_gemv();
  const Smem sh = smem_map(smem_raw);
  const uint32_t tid = threadIdx.x, nch = g.K / 16, tag = g.tag_a;
  uint4* qhi = reinterpret_cast<uint4*>(sh.uni);
  uint4* qlo = qhi + nch;
  float4* aux = reinterpret_cast<float4*>(qlo + nch);
  const uint32_t* hq = static_cast<const uint32_t*>(g.a);
  const uint32_t* he = static_cast<const uint32_t*>(g.b);
  Chunk16 ca[2];
  uint32_t ew[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint32_t c = tid + q * NCT;
    ca[q].w[0] = ca[q].w[1] = ca[q].w[2] = ca[q].w[3] = make_uint4(0u, 0u, 0u, 0u);
    ew[q] = 0u;
    if (c < nch) {
      chunk_issue(hq, tag, c, ca[q]);
      ew[q] = ld_tagged(he + c);
    }
  }
  if (tr && tid == 0) tr[15] = global_ns();  // loads issued
  const uint32_t rrows = g.re - g.rb;
  const bool has_r = g.epi == 1 && tid < rrows;
  const uint32_t* rin = static_cast<const uint32_t*>(g.resid_in) + g.rb + tid;
  const uint32_t rw0 = has_r ? ld_tagged(rin) : 0u;
  bool ok;
  {
    const uint32_t* pp[8];
    uint32_t pt[8];
    uint4 pw4[8];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t c = tid + q * NCT;
      chunk_pend(hq, tag, c < nch ? c : 0u, c < nch, pp, pt, 4 * q);
#pragma unroll
      for (int k = 0; k < 4; ++k) pw4[4 * q + k] = ca[q].w[k];
    }
    ok = settle4<8>(pp, pt, pw4);
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int k = 0; k < 4; ++k) ca[q].w[k] = pw4[4 * q + k];
    const uint32_t c1 = tid + NCT;
    const uint32_t* pp1[3] = {he + (tid < nch ? tid : 0u), he + (c1 < nch ? c1 : 0u), rin};
    const uint32_t pt1[3] = {tid < nch ? tag : 0u, c1 < nch ? tag : 0u, has_r ? g.tag_r : 0u};
    uint32_t w1[3] = {ew[0], ew[1], rw0};
    ok &= settle1<3>(pp1, pt1, w1);
    ew[0] = w1[0];
    ew[1] = w1[1];
    if (has_r) gemv_partials(sh, nch)[g.W * rrows + tid] = tag_value(w1[2]);
  }
  if (!ok) set_status(P.status, kStatusTimeout);
  if (tr && tid == 0 && ca[0].w[0].x != 0x12345678u) tr[8] = global_ns();
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint32_t c = tid + q * NCT;
    if (c >= nch) continue;
    uint4 h, l;
    int qs = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 w = ca[q].w[k];  // codes of elements 4k .. 4k + 3 in bytes 2 (low) and 3 (high)
      (&l.x)[k] = __byte_perm(__byte_perm(w.x, w.y, 0x0062), __byte_perm(w.z, w.w, 0x0062), 0x5410);
      (&h.x)[k] = __byte_perm(__byte_perm(w.x, w.y, 0x0073), __byte_perm(w.z, w.w, 0x0073), 0x5410);
      qs += (int)(int16_t)(w.x >> 16) + (int)(int16_t)(w.y >> 16) + (int)(int16_t)(w.z >> 16) +
            (int)(int16_t)(w.w >> 16);
    }
    const uint32_t E = ew[q] >> 16;
    qhi[c] = h;
    qlo[c] = l;
    aux[c] = make_float4(__int_as_float(128 * qs), E >= 15 ? __uint_as_float((E - 14u) << 23) : 0.f, 0.f, 0.f);
  }
  if (tr && tid == 0) tr[9] = global_ns();
  consumer_sync();
}

// Form the phase's input vector once per CTA and store it, quantised, in shared
// memory: chunk c at hi[c], lo[c] (uint4 each) and aux[c] = {qsum128, scale, sum x}.
// The inputs are polled until every word carries its expected tag. This form gives
// each thread whole 16-element chunks (a head's chunks on adjacent lanes for the
// per-head norm and the Turbo8 rotation); the RMSNorm inputs take the
// four-threads-per-chunk form below, which measured faster for them and slower
// for the wider inputs of the down and output projections.
__device__ __noinline__ void gemv_prologue_chunks(unsigned long long* tr) {
  const Program& P = prog();
  const Gemv& g = cur_gemv();
  const Smem sh = smem_map(smem_raw);
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t nch = g.K / 16;
  uint4* qhi = reinterpret_cast<uint4*>(sh.uni);
  uint4* qlo = qhi + nch;
  float4* aux = reinterpret_cast<float4*>(qlo + nch);
  const bool has_b = g.pro == kAddRms || g.pro == kSiluMul || g.pro == kHeadNormSilu || g.pro == kWhtGate;
  const bool has_w = g.pro == kAddRms || g.pro == kRms || g.pro == kHeadNormSilu;
  // chunk c of input b (kWhtGate: head h's gate chunk sits at q_full[h * 2D + D + ...])
  auto bchunk = [&](uint32_t c) {
    return g.pro == kWhtGate ? c + ((16 * c) / g.head_dim + 1) * (g.head_dim / 16) : c;
  };
  // every global load of the prologue is issued before any is used: one round trip
  Chunk16 ca[2], cb[2];
  uint4 pw[2][2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint32_t c = tid + q * NCT;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    ca[q].w[0] = ca[q].w[1] = ca[q].w[2] = ca[q].w[3] = z;
    cb[q] = ca[q];
    pw[q][0] = pw[q][1] = z;
    if (c < nch) {
      chunk_issue(g.a, g.tag_a, c, ca[q]);
      if (has_b) chunk_issue(g.b, g.tag_b, bchunk(c), cb[q]);
      if (has_w) {
        const uint32_t wi = g.pro == kHeadNormSilu ? (c * 16) % g.head_dim : c * 16;
        const uint4* wp = reinterpret_cast<const uint4*>(g.nw + wi);
        pw[q][0] = wp[0];
        pw[q][1] = wp[1];
      }
    }
  }
  if (tr && tid == 0) tr[15] = global_ns();  // loads issued
  // the down projection's residual rows (at most one per thread), for the epilogue:
  // loaded in the same round
  const uint32_t rrows = g.re - g.rb;
  const bool has_r = g.epi == 1 && tid < rrows;
  const uint32_t* rin = static_cast<const uint32_t*>(g.resid_in) + g.rb + tid;
  uint32_t rw = has_r ? ld_tagged(rin) : 0u;
  bool ok;
  {  // the tagged inputs not there yet, polled together
    const uint32_t* pp[16];
    uint32_t pt[16];
    uint4 pw4[16];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t c = tid + q * NCT;
      chunk_pend(g.a, g.tag_a, c < nch ? c : 0u, c < nch, pp, pt, 8 * q);
      chunk_pend(g.b, g.tag_b, c < nch ? bchunk(c) : 0u, c < nch && has_b, pp, pt, 8 * q + 4);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        pw4[8 * q + k] = ca[q].w[k];
        pw4[8 * q + 4 + k] = cb[q].w[k];
      }
    }
    ok = settle4<16>(pp, pt, pw4);
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        ca[q].w[k] = pw4[8 * q + k];
        cb[q].w[k] = pw4[8 * q + 4 + k];
      }
  }
  if (has_r) {
    const uint32_t* pp1[1] = {rin};
    const uint32_t pt1[1] = {g.tag_r};
    uint32_t w1[1] = {rw};
    ok &= settle1<1>(pp1, pt1, w1);
    gemv_partials(sh, nch)[g.W * rrows + tid] = tag_value(w1[0]);
  }
  if (!ok) set_status(P.status, kStatusTimeout);
  float raw[2][16];
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint32_t c = tid + q * NCT;
    chunk_values(ca[q], g.tag_a, raw[q]);
    if (g.pro == kAddRms) {
      float xb[16];
      chunk_values(cb[q], g.tag_b, xb);
#pragma unroll
      for (int j = 0; j < 16; ++j) raw[q][j] = round_bf16(raw[q][j] + xb[j]);
      if (blockIdx.x == 0 && c < nch)  // one CTA keeps x_resid for the down projection's residual
        chunk_store_tagged(g.resid_out + c * 16, raw[q], g.out_tag);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) ss = fmaf(raw[q][j], raw[q][j], ss);  // zero past the end
  }
  if (tr && tid == 0 && raw[0][0] != 12345.f) tr[8] = global_ns();  // thread 0's loads have landed
  float inv = 0.f;
  if (g.pro == kRms || g.pro == kAddRms) {
    ss = warp_sum(ss);
    if (lane == 0) sh.misc[warp] = ss;
    consumer_sync();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) tot += sh.misc[w];
    inv = rsqrtf(tot / (float)g.K + P.eps);
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint32_t c = tid + q * NCT;
    if (q == 1 && NCT >= nch) break;  // (uniform) no second chunk anywhere
    float v[16], xb[16], w[16];
    chunk_values(cb[q], g.tag_b, xb);
    unpack8(pw[q][0], w);
    unpack8(pw[q][1], w + 8);
    if (g.pro == kHeadNormSilu) {
      // a head's chunks sit on adjacent lanes: reduce its sum of squares there
      float hs = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) hs = fmaf(raw[q][j], raw[q][j], hs);
      for (uint32_t o = 1; o < g.head_dim / 16; o <<= 1) hs += __shfl_xor_sync(FULLMASK, hs, o);
      const float hi = rsqrtf(hs / (float)g.head_dim + P.eps);
      float yn[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) yn[j] = round_bf16(raw[q][j] * hi * w[j]);
      if (g.dump && c < nch) chunk_store_bf16(g.dump + c * 16, yn);
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = silu_fast(xb[j]) * yn[j];
    } else if (g.pro == kPlain) {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = raw[q][j];
    } else if (g.pro == kWhtGate) {
      // a head's D/16 chunks sit on adjacent lanes: the WHT's strides below 16 stay
      // in the chunk, larger ones pair lane with lane ^ (stride / 16)
      float x[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) x[j] = raw[q][j];
#pragma unroll
      for (int h = 1; h < 16; h <<= 1)
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (!(j & h)) {
            const float a0 = x[j], a1 = x[j + h];
            x[j] = a0 + a1;
            x[j + h] = a0 - a1;
          }
      for (uint32_t m = 1; m < g.head_dim / 16; m <<= 1)
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float pv = __shfl_xor_sync(FULLMASK, x[j], m);
          x[j] = (lane & m) ? pv - x[j] : x[j] + pv;
        }
      const float wn = rsqrtf((float)g.head_dim);
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = round_bf16(round_bf16(x[j] * wn) * sigmoidf_(xb[j]));
    } else if (g.pro == kSiluMul) {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = silu_fast(raw[q][j]) * xb[j];
    } else {  // RMSNorm (plain or after the residual add)
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = round_bf16(raw[q][j] * inv * w[j]);
      if (g.dump && c < nch) chunk_store_bf16(g.dump + c * 16, v);
    }
    if (c < nch) {
      XQ x;
      quantize16(v, x);
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) s += v[j];
      qhi[c] = make_uint4(x.hi[0], x.hi[1], x.hi[2], x.hi[3]);
      qlo[c] = make_uint4(x.lo[0], x.lo[1], x.lo[2], x.lo[3]);
      aux[c] = make_float4(__int_as_float(x.qsum128), x.scale, s, 0.f);
    }
  }
  if (tr && tid == 0) tr[9] = global_ns();
  consumer_sync();
}

// An RMSNorm input (kRms, kAddRms) with four consecutive elements per thread:
// thread t of round r holds elements 4 (t + 384 r) .. 4 (t + 384 r) + 3, so the
// loads of a warp are 512 contiguous bytes, every consumer thread takes part, and a
// chunk's four threads are adjacent lanes (its largest magnitude, quantised sum and
// sum are reduced across them). The arithmetic per element is that of the chunk
// form, so the stored chunks are the same bits. R rounds cover K <= 1536 R.
__device__ __forceinline__ uint4 quad_issue(const void* base, uint32_t tag, uint32_t e) {
  if (tag) return ld_tagged4(static_cast<const uint32_t*>(base) + e);
  const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + e);
  return make_uint4(u.x, u.y, 0u, 0u);
}
__device__ __forceinline__ void quad_values(const uint4 w, uint32_t tag, float* x) {
  if (tag) {
    x[0] = tag_value(w.x); x[1] = tag_value(w.y); x[2] = tag_value(w.z); x[3] = tag_value(w.w);
  } else {
    x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
  }
}
// Quantise the four values of this thread as part of chunk c (lanes 4m .. 4m + 3
// of a warp hold one chunk): the same scale, codes and sums as quantize16 over
// the whole chunk. Every lane takes part in the shuffles; `store` selects the
// chunks that exist.
__device__ __forceinline__ void quantize_quad(const float* v, uint32_t c, bool store, uint32_t* qhi, uint32_t* qlo,
                                              float4* aux) {
  const uint32_t j = threadIdx.x & 3;
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  amax = fmaxf(amax, __shfl_xor_sync(FULLMASK, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(FULLMASK, amax, 2));
  const uint32_t E = __float_as_uint(amax) >> 23;
  const bool nz = E >= 15;
  const float up = nz ? __uint_as_float((268u - E) << 23) : 0.f;  // 2^(15-e)
  const float scale = nz ? __uint_as_float((E - 14u) << 23) : 0.f;
  int t[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) t[i] = sat16(v[i] * up);
  int qs = t[0] + t[1] + t[2] + t[3];
  float sx = v[0] + v[1] + v[2] + v[3];
  qs += __shfl_xor_sync(FULLMASK, qs, 1);
  sx += __shfl_xor_sync(FULLMASK, sx, 1);
  qs += __shfl_xor_sync(FULLMASK, qs, 2);
  sx += __shfl_xor_sync(FULLMASK, sx, 2);
  if (store) {
    qlo[4 * c + j] = __byte_perm(__byte_perm(t[0], t[1], 0x0040), __byte_perm(t[2], t[3], 0x0040), 0x5410);
    qhi[4 * c + j] = __byte_perm(__byte_perm(t[0], t[1], 0x0051), __byte_perm(t[2], t[3], 0x0051), 0x5410);
    if (j == 0) aux[c] = make_float4(__int_as_float(128 * qs), scale, sx, 0.f);
  }
}
template <int R>
__device__ __noinline__ void gemv_prologue_quads(unsigned long long* tr) {
  const Program& P = prog();
  const Gemv& g = cur_gemv();
  const Smem sh = smem_map(smem_raw);
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t K = g.K, nch = K / 16;
  uint32_t* qhi = reinterpret_cast<uint32_t*>(sh.uni);
  uint32_t* qlo = qhi + 4 * nch;
  float4* aux = reinterpret_cast<float4*>(qlo + 4 * nch);
  const bool add = g.pro == kAddRms;  // else kRms
  const uint32_t tag_a = g.tag_a, tag_b = add ? g.tag_b : 0u;
  // every global load of the prologue is issued before any is used: one round trip
  uint4 A[R], Bq[R];
  uint2 Wq[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const uint32_t e = 4u * (tid + (uint32_t)NCT * r);
    A[r] = Bq[r] = make_uint4(0u, 0u, 0u, 0u);
    Wq[r] = make_uint2(0u, 0u);
    if (e < K) {
      A[r] = quad_issue(g.a, tag_a, e);
      if (add) Bq[r] = quad_issue(g.b, tag_b, e);
      Wq[r] = *reinterpret_cast<const uint2*>(g.nw + e);
    }
  }
  if (tr && tid == 0) tr[15] = global_ns();  // loads issued
  // the tagged inputs not there yet, polled together until every word has its tag
  uint32_t todo = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const uint32_t e = 4u * (tid + (uint32_t)NCT * r);
    if (e < K && ((tag_a && !tags4_are(A[r], tag_a)) || (tag_b && !tags4_are(Bq[r], tag_b)))) todo |= 1u << r;
  }
  if (todo) {
    const uint64_t t0 = global_ns(), limit = wait_limit();
    for (uint32_t n = 1; todo; ++n) {
      __nanosleep(64);
#pragma unroll
      for (int r = 0; r < R; ++r)
        if ((todo >> r) & 1u) {
          const uint32_t e = 4u * (tid + (uint32_t)NCT * r);
          if (tag_a) A[r] = quad_issue(g.a, tag_a, e);
          if (tag_b) Bq[r] = quad_issue(g.b, tag_b, e);
        }
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (((todo >> r) & 1u) && (!tag_a || tags4_are(A[r], tag_a)) && (!tag_b || tags4_are(Bq[r], tag_b)))
          todo &= ~(1u << r);
      if (todo && (global_ns() - t0 > limit || ((n & 15) == 0 && timed_out(P.status)))) {
        set_status(P.status, kStatusTimeout);
        break;
      }
    }
  }
  // the values before the norm (kept in A as float bits) and their sum of squares
  float ss = 0.f;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const uint32_t e = 4u * (tid + (uint32_t)NCT * r);
    float x[4];
    quad_values(A[r], tag_a, x);
    if (add) {
      float xb[4];
      quad_values(Bq[r], tag_b, xb);
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = round_bf16(x[i] + xb[i]);
      if (blockIdx.x == 0 && e < K)  // one CTA keeps x_resid for the down projection's residual
        st_tagged4(g.resid_out + e, make_uint4(tag_word(x[0], g.out_tag), tag_word(x[1], g.out_tag),
                                                tag_word(x[2], g.out_tag), tag_word(x[3], g.out_tag)));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) ss = fmaf(x[i], x[i], ss);  // zero past the end
    A[r] = make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3]));
  }
  if (tr && tid == 0 && ss != 12345.f) tr[8] = global_ns();  // thread 0's loads have landed
  ss = warp_sum(ss);
  if (lane == 0) sh.misc[warp] = ss;
  consumer_sync();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < NCW; ++w) tot += sh.misc[w];
  const float inv = rsqrtf(tot / (float)K + P.eps);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (4u * (uint32_t)NCT * r >= K) break;  // (uniform) no thread has this round
    const uint32_t e = 4u * (tid + (uint32_t)NCT * r);
    const bool in = e < K;
    const float w[4] = {bf16lo(Wq[r].x), bf16hi(Wq[r].x), bf16lo(Wq[r].y), bf16hi(Wq[r].y)};
    float v[4];
    v[0] = round_bf16(__uint_as_float(A[r].x) * inv * w[0]);
    v[1] = round_bf16(__uint_as_float(A[r].y) * inv * w[1]);
    v[2] = round_bf16(__uint_as_float(A[r].z) * inv * w[2]);
    v[3] = round_bf16(__uint_as_float(A[r].w) * inv * w[3]);
    if (g.dump && in)
      *reinterpret_cast<uint2*>(g.dump + e) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
    if (!in) v[0] = v[1] = v[2] = v[3] = 0.f;
    quantize_quad(v, e / 16, in, qhi, qlo, aux);
  }
  if (tr && tid == 0) tr[9] = global_ns();
  consumer_sync();
}
// The phase's input vector: the RMSNorm inputs in the four-threads-per-chunk form,
// the others in whole chunks per thread.
__device__ __noinline__ void gemv_prologue(unsigned long long* tr) {
  const Gemv& g = cur_gemv();
  if (g.pro == kQuantized) return gemv_prologue_quantized(tr);
  if (g.pro != kRms && g.pro != kAddRms) return gemv_prologue_chunks(tr);
  const uint32_t rounds = (g.K + 4 * NCT - 1) / (4 * NCT);
  if (rounds <= 1) return gemv_prologue_quads<1>(tr);
  if (rounds <= 2) return gemv_prologue_quads<2>(tr);
  if (rounds <= 3) return gemv_prologue_quads<3>(tr);
  if (rounds <= 4) return gemv_prologue_quads<4>(tr);
  if (rounds <= 6) return gemv_prologue_quads<6>(tr);
  return gemv_prologue_quads<8>(tr);
}

// Rows computed whole by one warp with nothing added after the sum (one K-part, no
// residual) are stored by the row loop itself; the others go through the partial
// sums and the epilogue.
__device__ __forceinline__ bool gemv_direct(const Gemv& g) { return g.W == 1 && g.epi == 0; }

// The row loop of a GEMV phase. Warp (rs, kp) computes row rs of every tile over
// the chunks kp, kp + W, ... of each lane, reduces it across the warp and leaves
// the sum in the partials; the producer publishes each tile's first row and row
// count beside its ring offset, so the loop only counts its tiles. Per chunk the
// lane keeps x as hi/lo bytes, 128 * sum(q) and the power-of-two scale: the row's
// part is scale * (s * sum((c - 128) q) + (b / 128 + s) * 128 sum(q)), the first
// sum exact in integers, the bias term on the quantised chunk sum.
// The tile loop for CPL chunks per lane (one instantiation per chunk count, all in
// one out-of-line function so every projection phase enters the same code).
template <int CPL>
__device__ __forceinline__ void gemv_tiles(const Gemv& g, const Smem& sh, uint32_t& it, bool& dead,
                                           unsigned long long* tr) {
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t K = g.K, W = g.W, gstride = g.gstride, soff = g.scale_off, boff = g.bias_off;
  const uint32_t kp = warp % W, rs = warp / W, nch = K / 16;
  const uint4* qhi = reinterpret_cast<const uint4*>(sh.uni);
  const uint4* qlo = qhi + nch;
  const float4* aux = reinterpret_cast<const float4*>(qlo + nch);
  // chunk c of this lane is ch0 + c * cstep; chunks past the row end read chunk 0
  // (valid memory) against x = 0, so the loops are branch-free
  const uint32_t ch0 = lane + 32 * kp, cstep = 32 * W;
  auto chk = [&](int c) { const uint32_t ch = ch0 + c * cstep; return ch < nch ? ch : 0u; };
  XQ xq[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const bool valid = ch0 + c * cstep < nch;
    const uint4 h = qhi[chk(c)], l = qlo[chk(c)];
    const float4 x = aux[chk(c)];
    xq[c].hi[0] = valid ? h.x : 0u; xq[c].hi[1] = valid ? h.y : 0u;
    xq[c].hi[2] = valid ? h.z : 0u; xq[c].hi[3] = valid ? h.w : 0u;
    xq[c].lo[0] = valid ? l.x : 0u; xq[c].lo[1] = valid ? l.y : 0u;
    xq[c].lo[2] = valid ? l.z : 0u; xq[c].lo[3] = valid ? l.w : 0u;
    xq[c].qsum128 = valid ? __float_as_int(x.x) : 0;
    xq[c].scale = valid ? x.y : 0.f;
  }
  const uint32_t rb = g.rb, ntiles = g.ntiles;
  float* part = gemv_partials(sh, nch) + kp * (g.re - rb);  // indexed by row - rb
  const bool direct = gemv_direct(g);
  int* status = prog().status;
  const uint64_t limit = wait_limit();
  if (tr && threadIdx.x == 0) tr[11] = global_ns();
  float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;  // sums of the last tiles' rows
  // their places: in part, or for whole rows in the outputs from obase (~0u: none)
  uint32_t pr0 = ~0u, pr1 = ~0u, pr2 = ~0u, pr3 = ~0u;
  for (uint32_t t = 0; t < ntiles; ++t) {
    const uint32_t st = slot_of(it);
    if (!dead && !mbar_wait(&sh.full[st], parity_of(it), limit)) {
      set_status(status, kStatusTimeout);
      dead = true;
    }
    if (tr && threadIdx.x == 0) {
      if (t == 0) tr[4] = global_ns();
      if (t + 1 == ntiles) tr[5] = global_ns();
    }
    // after a wait ran out nothing of the ring is read, and no slot is released
    // (its copy may still be in flight)
    const uint32_t meta = dead ? 0u : sh.tmeta[st];
    const uint32_t tout = s_tout[st];
    const bool mine = rs < (meta >> 24);
    float sum = 0.f;
    if (mine) {
      const uint8_t* sb = sh.ring + sh.toff[st];
      const uint8_t* crow = sb + rs * K;
      const uint16_t* srow = reinterpret_cast<const uint16_t*>(sb + soff) + rs * gstride;
      const uint16_t* brow = reinterpret_cast<const uint16_t*>(sb + boff) + rs * gstride;
      uint4 w[CPL];
      float sc[CPL], bi[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) {  // all shared-memory loads first
        w[c] = *reinterpret_cast<const uint4*>(crow + chk(c) * 16);
        sc[c] = bf16f(srow[chk(c) >> 2]);
        bi[c] = bf16f(brow[chk(c) >> 2]);
      }
      // the warp's part of the tile is in registers: the slot goes back to the
      // producer before the arithmetic
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[st]);
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const float q128 = (float)xq[c].qsum128;
        sum = fmaf(xq[c].scale, fmaf(sc[c], (float)dot16i(w[c], xq[c]), fmaf(bi[c], 0.0078125f, sc[c]) * q128), sum);
      }
    } else {
      __syncwarp();
      if (lane == 0 && !dead) mbar_arrive(&sh.empty[st]);
    }
    ++it;
    // the lanes' sums of the last four tiles' rows are reduced across the warp
    // together (one transposed reduction instead of four)
    acc3 = acc2; acc2 = acc1; acc1 = acc0; acc0 = sum;
    pr3 = pr2; pr2 = pr1; pr1 = pr0; pr0 = !mine ? ~0u : direct ? tout + rs : (meta & 0xFFFFFFu) + rs - rb;
    if ((t & 3) == 3 || t + 1 == ntiles) {
      float v[4] = {acc0, acc1, acc2, acc3};
      const float tot = reduce_transposed<4>(v, lane);  // lane L: the total of v[L / 8]
      const uint32_t q = lane >> 3;
      const uint32_t pr = q == 0 ? pr0 : q == 1 ? pr1 : q == 2 ? pr2 : pr3;
      if ((lane & 7) == 0 && pr != ~0u) {
        if (direct) gemv_store(g, 0, pr, tot);  // a whole row: its output, straight from the loop
        else part[pr] = tot;
      }
      acc0 = acc1 = acc2 = acc3 = 0.f;
      pr0 = pr1 = pr2 = pr3 = ~0u;
    }
  }
}

__device__ __noinline__ uint32_t gemv_main(uint32_t itd, unsigned long long* tr) {
  const Gemv& g = cur_gemv();
  const Smem sh = smem_map(smem_raw);
  if (tr && threadIdx.x == 0) tr[10] = global_ns();
  uint32_t it = itd & ~kDeadBit;
  bool dead = (itd & kDeadBit) != 0;
  switch (g.cpl) {
    case 1: gemv_tiles<1>(g, sh, it, dead, tr); break;
    case 2: gemv_tiles<2>(g, sh, it, dead, tr); break;
    case 3: gemv_tiles<3>(g, sh, it, dead, tr); break;
    case 4: gemv_tiles<4>(g, sh, it, dead, tr); break;
    default: gemv_tiles<5>(g, sh, it, dead, tr); break;
  }
  if (tr && threadIdx.x == 0) tr[6] = global_ns();
  return it | (dead ? kDeadBit : 0u);
}

// The rows of a GEMV phase, then (unless the row loop stored them) its outputs: the
// K-parts of each row summed in a fixed order, the residual added for the down
// projection, bf16 stores by consecutive threads.
__device__ uint32_t gemv_rows(uint32_t itd, unsigned long long* tr) {
  itd = gemv_main(itd, tr);
  if (gemv_direct(cur_gemv())) return itd;
  consumer_sync();
  if (tr && threadIdx.x == 0) tr[12] = global_ns();
  const Gemv& g = cur_gemv();
  const Smem sh = smem_map(smem_raw);
  const uint32_t rb = g.rb, rows = g.re - g.rb, W = g.W;
  const float* part = gemv_partials(sh, g.K / 16);
  if (g.epi == 3) {
    // a single sequence's gate|up: h = SiLU(gate) * up for the CTA's rows (gate and
    // up rounded to bf16, as their stored outputs would be), quantised per 16-row
    // chunk exactly as the down projection's prologue would (quantize16 on a chunk
    // held by four lanes), stored as codes and chunk exponents
    const uint32_t n = g.pn, lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tag = g.out_tag;
    uint32_t* hq = reinterpret_cast<uint32_t*>(g.out[0]);
    uint32_t* he = reinterpret_cast<uint32_t*>(g.out[1]);
    for (uint32_t base = 64 * warp; base < n; base += 64 * NCW) {  // 64 rows per warp, lanes 0..15
      const uint32_t r0 = base + 4 * lane;
      const bool in = lane < 16 && r0 < n;
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float gs = 0.f, us = 0.f;
        if (in)
          for (uint32_t w = 0; w < W; ++w) {
            gs += part[w * rows + r0 + i];
            us += part[w * rows + n + r0 + i];
          }
        v[i] = in ? silu_fast(round_bf16(gs)) * round_bf16(us) : 0.f;
      }
      float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
      amax = fmaxf(amax, __shfl_xor_sync(FULLMASK, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(FULLMASK, amax, 2));
      const uint32_t E = __float_as_uint(amax) >> 23;
      const float up = E >= 15 ? __uint_as_float((268u - E) << 23) : 0.f;  // 2^(15-e)
      if (in) {
        uint32_t t[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) t[i] = ((uint32_t)(uint16_t)sat16(v[i] * up) << 16) | tag;
        st_tagged4(hq + g.pr0 + r0, make_uint4(t[0], t[1], t[2], t[3]));
        if ((lane & 3) == 0) st_tagged(he + (g.pr0 + r0) / 16, (E << 16) | tag);
      }
    }
    return itd;
  }
  const float* resid = part + W * rows;
  for (uint32_t i = threadIdx.x; i < rows; i += NCT) {
    float y = 0.f;
    for (uint32_t w = 0; w < W; ++w) y += part[w * rows + i];
    if (g.epi == 1) y += resid[i];
    const uint32_t row = rb + i;
    uint32_t sg = 0;
    while (sg + 1 < g.nseg && row >= g.row0[sg + 1]) ++sg;
    gemv_store(g, sg, row - g.row0[sg], y);
  }
  return itd;
}

// ------------------------------------------------------------------ a batch's projections

// The phase buffer of a batched projection pass (bs sequences): the staged inputs
// [bs][K + kXPadH] (f16, or the raw bf16 rows between the two halves of an RMS
// prologue), per sequence and 64-column group {scale, scale * sum of the group's f16
// values} [bs][K/64], and the warps' partial sums [NCW][16 rows][8 sequences].
struct BatchBuf {
  uint16_t* xf;
  float2* xsq;
  float* part;
  uint32_t stride;  // elements
};
__device__ __forceinline__ BatchBuf batch_buf(const Smem& sh, uint32_t K, uint32_t bs) {
  BatchBuf b;
  b.stride = K + kXPadH;
  b.xf = reinterpret_cast<uint16_t*>(sh.uni);
  b.xsq = reinterpret_cast<float2*>(sh.uni + (size_t)bs * b.stride * 2);
  b.part = reinterpret_cast<float*>(b.xsq + (size_t)bs * (K / 64));
  return b;
}

// Two weight codes (the bytes that sel picks) as f16 values code - 128, exactly:
// the f16 with bits 0x64XX is 1024 + XX, and 1024 + XX - 1152 = XX - 128.
__device__ __forceinline__ uint32_t codes_f16x2(uint32_t w, uint32_t sel) {
  const uint32_t h = __byte_perm(w, 0x64646464u, sel);
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
  return r;
}
constexpr uint32_t kLoPair = 0x5140u, kHiPair = 0x5342u;  // bytes 0,1 and 2,3 of a word

// f16 pair {lo, hi} (round to nearest) and back.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ void unpack_words(const uint32_t (&pk)[8], float* x) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    x[2 * k] = bf16lo(pk[k]);
    x[2 * k + 1] = bf16hi(pk[k]);
  }
}

// D += A B for A 16x16 (row-major fragments a0..a3), B 16x8 (b0, b1), f16 in, fp32 sums.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Stage 16 input values (chunk c of sequence s; the four chunks of a 64-column
// group sit on a lane quad, every lane takes part): f16 with the group's factor
// 2^(14-e), 2^e <= group max < 2^(e+1), so the largest stays below 2^15; the group's
// scale 2^(e-14) and the sum of its values for the constant term (bf16 inputs are
// exact in f16 at that factor; others differ from their f16 forms by f16 rounding).
__device__ __forceinline__ void stage16(const BatchBuf& bb, uint32_t ng, const float* v, uint32_t s, uint32_t c,
                                        bool ok) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  amax = fmaxf(amax, __shfl_xor_sync(FULLMASK, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(FULLMASK, amax, 2));
  const uint32_t E = __float_as_uint(amax) >> 23;
  const bool nz = E >= 15;
  const float up = nz ? __uint_as_float((268u - E) << 23) : 0.f;     // 2^(14-e)
  const float scale = nz ? __uint_as_float((E - 14u) << 23) : 0.f;  // 2^(e-14)
  uint32_t h[8];
  float gsum = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    h[k] = pack_f16x2(v[2 * k] * up, v[2 * k + 1] * up);
    gsum += v[2 * k] + v[2 * k + 1];
  }
  gsum += __shfl_xor_sync(FULLMASK, gsum, 1);
  gsum += __shfl_xor_sync(FULLMASK, gsum, 2);
  if (ok) {
    uint4* dst = reinterpret_cast<uint4*>(bb.xf + s * bb.stride + c * 16);
    dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
    dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
    if ((c & 3) == 0) bb.xsq[s * ng + c / 4] = make_float2(scale, gsum);
  }
}

// Form and stage the inputs of sequences [b0, b0 + nb) of a batched projection pass
// (the same forms as gemv_prologue, per sequence). Chunk c of sequence s is item
// s * nch + c; a thread takes items tid + u * NCT, so consecutive items sit on
// consecutive lanes, and nch is a multiple of 4 (of a head's chunks): a group's four
// chunks share a lane quad and a head's chunks an aligned lane group. The loads of a
// round of NI items are issued before any is used (NI sized so that they stay in
// registers). RMS kinds keep the raw rows (bf16) in the staging buffer until the
// sums of squares are in.
// Sequence b's copy of a projection input: tagged words (stride in words) or the
// caller's bf16 vectors (tag 0, stride in elements).
__device__ __forceinline__ const void* seq_vec(const void* base, uint32_t tag, uint32_t stride, uint32_t b) {
  return tag ? static_cast<const void*>(static_cast<const uint32_t*>(base) + (size_t)b * stride)
             : static_cast<const void*>(static_cast<const uint16_t*>(base) + (size_t)b * stride);
}

template <int PRO>
__device__ __noinline__ void prologue_b_kind(uint32_t b0, uint32_t nb, unsigned long long* tr) {
  constexpr bool kTwo = PRO == kAddRms || PRO == kSiluMul || PRO == kHeadNormSilu || PRO == kWhtGate;
  constexpr bool kRmsKind = PRO == kRms || PRO == kAddRms;
  constexpr uint32_t NI = kTwo ? 2 : 4;
  const Program& P = prog();
  const Gemv& g = cur_gemv();
  const Smem sh = smem_map(smem_raw);
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t K = g.K, nch = K / 16, ng = K / 64, items = nb * nch;
  const BatchBuf bb = batch_buf(sh, K, g.bs);
  // chunk c of input b (kWhtGate: head h's gate chunk sits at q_full[h * 2D + D + ...])
  auto bchunk = [&](uint32_t c) {
    return PRO == kWhtGate ? c + ((16 * c) / g.head_dim + 1) * (g.head_dim / 16) : c;
  };
  float ssb[kRmsKind ? kMaxBatch : 1];
#pragma unroll
  for (int b = 0; b < (kRmsKind ? kMaxBatch : 1); ++b) ssb[b] = 0.f;
  bool ok = true;
  for (uint32_t i0 = 0; i0 < items; i0 += NI * NCT) {
    Chunk16 a[NI], x2[kTwo ? NI : 1];
#pragma unroll
    for (uint32_t u = 0; u < NI; ++u) {
      const uint32_t i = i0 + u * NCT + tid;
      const bool ok_i = i < items;  // past the end: no load (its values are unused)
      const uint32_t s = ok_i ? i / nch : 0, c = ok_i ? i % nch : 0;
      a[u].w[0] = a[u].w[1] = a[u].w[2] = a[u].w[3] = make_uint4(0u, 0u, 0u, 0u);
      if constexpr (kTwo) x2[u] = a[u];
      if (ok_i) {
        chunk_issue(seq_vec(g.a, g.tag_a, g.sa, b0 + s), g.tag_a, c, a[u]);
        if constexpr (kTwo) chunk_issue(seq_vec(g.b, g.tag_b, g.sb, b0 + s), g.tag_b, bchunk(c), x2[u]);
      }
    }
    {  // the tagged inputs not there yet, polled together
      constexpr int NP = kTwo ? 8 * NI : 4 * NI;
      const uint32_t* pp[NP];
      uint32_t pt[NP];
      uint4 pw4[NP];
#pragma unroll
      for (uint32_t u = 0; u < NI; ++u) {
        const uint32_t i = i0 + u * NCT + tid;
        const bool in = i < items;
        const uint32_t s = in ? i / nch : 0, c = in ? i % nch : 0;
        chunk_pend(seq_vec(g.a, g.tag_a, g.sa, b0 + s), g.tag_a, c, in, pp, pt, (kTwo ? 8 : 4) * u);
        if constexpr (kTwo) chunk_pend(seq_vec(g.b, g.tag_b, g.sb, b0 + s), g.tag_b, bchunk(c), in, pp, pt, 8 * u + 4);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          pw4[(kTwo ? 8 : 4) * u + k] = a[u].w[k];
          if constexpr (kTwo) pw4[8 * u + 4 + k] = x2[u].w[k];
        }
      }
      ok &= settle4<NP>(pp, pt, pw4);
#pragma unroll
      for (uint32_t u = 0; u < NI; ++u)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          a[u].w[k] = pw4[(kTwo ? 8 : 4) * u + k];
          if constexpr (kTwo) x2[u].w[k] = pw4[8 * u + 4 + k];
        }
    }
    if (tr && tid == 0 && i0 == 0 && a[0].w[0].x != 0x12345678u) tr[8] = global_ns();  // loads landed
#pragma unroll
    for (uint32_t u = 0; u < NI; ++u) {
      const uint32_t i = i0 + u * NCT + tid;
      const bool ok_i = i < items;
      const uint32_t s = ok_i ? i / nch : 0, c = ok_i ? i % nch : 0;
      float raw[16], v[16];
      chunk_values(a[u], g.tag_a, raw);
      if constexpr (kRmsKind) {
        if constexpr (PRO == kAddRms) {
          float xb[16];
          chunk_values(x2[u], g.tag_b, xb);
#pragma unroll
          for (int k = 0; k < 16; ++k) raw[k] = round_bf16(raw[k] + xb[k]);
          if (ok_i && blockIdx.x == 0)  // one CTA stores x_resid
            chunk_store_tagged(g.resid_out + (size_t)(b0 + s) * g.sres_out + c * 16, raw, g.out_tag);
        }
        uint32_t pk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) pk[k] = pack_bf16x2(raw[2 * k], raw[2 * k + 1]);  // exact: bf16 values
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) ss = fmaf(raw[j], raw[j], ss);
        if (ok_i) {
#pragma unroll
          for (int b = 0; b < kMaxBatch; ++b) ssb[b] += s == (uint32_t)b ? ss : 0.f;
          uint4* dst = reinterpret_cast<uint4*>(bb.xf + s * bb.stride + c * 16);
          dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      } else {
        if constexpr (PRO == kSiluMul) {
          float xb[16];
          chunk_values(x2[u], g.tag_b, xb);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = silu_fast(raw[j]) * xb[j];
        } else if constexpr (PRO == kHeadNormSilu) {
          float hs = 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j) hs = fmaf(raw[j], raw[j], hs);
          for (uint32_t o = 1; o < g.head_dim / 16; o <<= 1) hs += __shfl_xor_sync(FULLMASK, hs, o);
          const float hi = rsqrtf(hs / (float)g.head_dim + P.eps);
          float xb[16], w[16];
          chunk_values(x2[u], g.tag_b, xb);
          const uint4* wp = reinterpret_cast<const uint4*>(g.nw + (c * 16) % g.head_dim);
          unpack8(wp[0], w);
          unpack8(wp[1], w + 8);
          uint32_t pk[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            pk[k] = pack_bf16x2(raw[2 * k] * hi * w[2 * k], raw[2 * k + 1] * hi * w[2 * k + 1]);
          unpack_words(pk, v);
          if (g.dump && ok_i) chunk_store_bf16(g.dump + (size_t)(b0 + s) * (P.seq_stride / 2) + c * 16, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] *= silu_fast(xb[j]);
        } else if constexpr (PRO == kWhtGate) {
          // a head's chunks sit on an aligned group of adjacent lanes (nch is a
          // multiple of the head's D / 16 chunks): strides below 16 in the chunk,
          // larger ones across lanes
          float xb[16];
          chunk_values(x2[u], g.tag_b, xb);
#pragma unroll
          for (int h = 1; h < 16; h <<= 1)
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (!(j & h)) {
                const float a0 = raw[j], a1 = raw[j + h];
                raw[j] = a0 + a1;
                raw[j + h] = a0 - a1;
              }
          for (uint32_t m = 1; m < g.head_dim / 16; m <<= 1)
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float pv = __shfl_xor_sync(FULLMASK, raw[j], m);
              raw[j] = (lane & m) ? pv - raw[j] : raw[j] + pv;
            }
          const float wn = rsqrtf((float)g.head_dim);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = round_bf16(round_bf16(raw[j] * wn) * sigmoidf_(xb[j]));
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = raw[j];
        }
        stage16(bb, ng, v, s, c, ok_i);
      }
    }
  }
  if (!ok) set_status(P.status, kStatusTimeout);
  if (tr && tid == 0) tr[9] = global_ns();
  if constexpr (kRmsKind) {
    // each sequence's sum of squares: per thread, per warp, then over the warps in a
    // fixed order; then the staged raw rows normalised and converted in place
    float* part = sh.misc;  // [kMaxBatch][NCW]
#pragma unroll
    for (int b = 0; b < kMaxBatch; ++b) {
      const float w = warp_sum(ssb[b]);
      if (lane == 0) part[b * NCW + warp] = w;
    }
    consumer_sync();
    float inv_all[kMaxBatch];
#pragma unroll
    for (int b = 0; b < kMaxBatch; ++b) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < NCW; ++w) tot += part[b * NCW + w];
      inv_all[b] = rsqrtf(tot / (float)K + P.eps);
    }
    if (tr && tid == 0) tr[10] = global_ns();
    for (uint32_t i0 = 0; i0 < items; i0 += 4 * NCT) {
      uint4 r[4][2], wv[4][2];
#pragma unroll
      for (uint32_t u = 0; u < 4; ++u) {
        const uint32_t i = i0 + u * NCT + tid;
        const bool ok = i < items;
        const uint32_t s = ok ? i / nch : 0, c = ok ? i % nch : 0;
        const uint4* src = reinterpret_cast<const uint4*>(bb.xf + s * bb.stride + c * 16);
        r[u][0] = src[0];
        r[u][1] = src[1];
        const uint4* wp = reinterpret_cast<const uint4*>(g.nw + c * 16);
        wv[u][0] = wp[0];
        wv[u][1] = wp[1];
      }
#pragma unroll
      for (uint32_t u = 0; u < 4; ++u) {
        const uint32_t i = i0 + u * NCT + tid;
        const bool ok = i < items;
        const uint32_t s = ok ? i / nch : 0, c = ok ? i % nch : 0;
        float raw[16], w[16], v[16];
        unpack8(r[u][0], raw);
        unpack8(r[u][1], raw + 8);
        unpack8(wv[u][0], w);
        unpack8(wv[u][1], w + 8);
        float inv = inv_all[0];
#pragma unroll
        for (int q = 1; q < kMaxBatch; ++q) inv = s == (uint32_t)q ? inv_all[q] : inv;
        uint32_t pk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) pk[k] = pack_bf16x2(raw[2 * k] * inv * w[2 * k], raw[2 * k + 1] * inv * w[2 * k + 1]);
        unpack_words(pk, v);
        if (g.dump && ok) chunk_store_bf16(g.dump + (size_t)(b0 + s) * (P.seq_stride / 2) + c * 16, v);
        stage16(bb, ng, v, s, c, ok);
      }
    }
  }
  if (tr && tid == 0) tr[11] = global_ns();
  consumer_sync();
}

__device__ __forceinline__ void gemv_prologue_b(uint32_t b0, uint32_t nb, unsigned long long* tr) {
  switch (cur_gemv().pro) {
    case kRms: prologue_b_kind<kRms>(b0, nb, tr); break;
    case kAddRms: prologue_b_kind<kAddRms>(b0, nb, tr); break;
    case kSiluMul: prologue_b_kind<kSiluMul>(b0, nb, tr); break;
    case kHeadNormSilu: prologue_b_kind<kHeadNormSilu>(b0, nb, tr); break;
    case kWhtGate: prologue_b_kind<kWhtGate>(b0, nb, tr); break;
    default: prologue_b_kind<kPlain>(b0, nb, tr); break;
  }
}

template <bool TWO>
struct GroupOps {
  const uint8_t *wa, *wb;
  const uint16_t *sc, *bi, *xrow;
  const float2 *sqa, *sqb;
  uint32_t ra, rb, gstride;
  // the group's four products as two chains (columns 0-31, 32-63 of the slice
  // pattern), summed at the end: rows g, g + 8 x sequences 2t, 2t + 1
  __device__ __forceinline__ void sums(uint32_t gr, float (&acc)[4]) const {
    const uint4 xa = *reinterpret_cast<const uint4*>(xrow + gr * 64);
    const uint4 xb = *reinterpret_cast<const uint4*>(xrow + gr * 64 + 8);
    const uint4 u = *reinterpret_cast<const uint4*>(wa + gr * 64);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (TWO) v = *reinterpret_cast<const uint4*>(wb + gr * 64);
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    mma_f16(c0, codes_f16x2(u.x, kLoPair), TWO ? codes_f16x2(v.x, kLoPair) : 0u, codes_f16x2(u.x, kHiPair),
            TWO ? codes_f16x2(v.x, kHiPair) : 0u, xa.x, xa.y);
    mma_f16(c1, codes_f16x2(u.z, kLoPair), TWO ? codes_f16x2(v.z, kLoPair) : 0u, codes_f16x2(u.z, kHiPair),
            TWO ? codes_f16x2(v.z, kHiPair) : 0u, xb.x, xb.y);
    mma_f16(c0, codes_f16x2(u.y, kLoPair), TWO ? codes_f16x2(v.y, kLoPair) : 0u, codes_f16x2(u.y, kHiPair),
            TWO ? codes_f16x2(v.y, kHiPair) : 0u, xa.z, xa.w);
    mma_f16(c1, codes_f16x2(u.w, kLoPair), TWO ? codes_f16x2(v.w, kLoPair) : 0u, codes_f16x2(u.w, kHiPair),
            TWO ? codes_f16x2(v.w, kHiPair) : 0u, xb.z, xb.w);
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = c0[k] + c1[k];
  }
  // y += scale_row * scale_seq * sums + (bias_row + 128 scale_row) * sum_seq
  __device__ __forceinline__ void add(uint32_t gr, const float (&acc)[4], float (&y)[2][2]) const {
    const float2 qa = sqa[gr], qb = sqb[gr];
    const float sA = bf16f(sc[ra * gstride + gr]), tA = fmaf(sA, 128.f, bf16f(bi[ra * gstride + gr]));
    y[0][0] = fmaf(sA * qa.x, acc[0], fmaf(tA, qa.y, y[0][0]));
    y[0][1] = fmaf(sA * qb.x, acc[1], fmaf(tA, qb.y, y[0][1]));
    if (TWO) {
      const float sB = bf16f(sc[rb * gstride + gr]), tB = fmaf(sB, 128.f, bf16f(bi[rb * gstride + gr]));
      y[1][0] = fmaf(sB * qa.x, acc[2], fmaf(tB, qa.y, y[1][0]));
      y[1][1] = fmaf(sB * qb.x, acc[3], fmaf(tB, qb.y, y[1][1]));
    }
  }
};

// One warp's share of a batched tile: the column groups j, j + W, ... of tile rows
// g and g + 8 (TWO) against the pass's sequences, two groups at a time (added in
// column order). Per 64-column group, four m16n8k16 products: thread (g = lane/4,
// t = lane%4) supplies the codes of rows g (and g + 8) and sequence g's input for
// the 16 columns at 16t of the group, the same permutation of k in both operands
// (columns 4m..4m+3 of that slice in product m), and receives rows g, g + 8 of
// sequences 2t, 2t + 1. Each group's sums are scaled by the row's and the
// sequence's group scales, the affine constant term taken against the group's
// input sum.
template <bool TWO>
__device__ __forceinline__ void batch_tile_groups(const uint8_t* tile, uint32_t nr, uint32_t K, uint32_t gstride,
                                                  uint32_t scale_off, uint32_t bias_off, uint32_t j, uint32_t W,
                                                  const uint16_t* xrow, const float2* sqa, const float2* sqb,
                                                  float (&y)[2][2]) {
  const uint32_t lane = threadIdx.x & 31, gq = lane >> 2, t = lane & 3, ng = K / 64;
  GroupOps<TWO> op;
  op.ra = min(gq, nr - 1);
  op.rb = min(gq + 8, nr - 1);
  op.wa = tile + op.ra * K + t * 16;
  op.wb = tile + op.rb * K + t * 16;
  op.sc = reinterpret_cast<const uint16_t*>(tile + scale_off);
  op.bi = reinterpret_cast<const uint16_t*>(tile + bias_off);
  op.xrow = xrow;
  op.sqa = sqa;
  op.sqb = sqb;
  op.gstride = gstride;
  uint32_t gr = j;
  for (; gr + W < ng; gr += 2 * W) {
    float a0[4], a1[4];
    op.sums(gr, a0);
    op.sums(gr + W, a1);
    op.add(gr, a0, y);
    op.add(gr + W, a1, y);
  }
  if (gr < ng) {
    float a0[4];
    op.sums(gr, a0);
    op.add(gr, a0, y);
  }
}

// The tiles of a batched projection pass. Team `team` (warps team*W .. team*W+W-1)
// takes the CTA's tiles team, team + T, ...; its warps release a tile with T
// arrivals each (T teams x W warps = every consumer warp's count), write their
// partial sums, and the team adds them in warp order and writes the rows of each
// sequence (+ residual) as bf16. Tiles of other teams are skipped unread.
__device__ __noinline__ uint32_t gemv_tiles_b(uint32_t itd, uint32_t b0, uint32_t nb, unsigned long long* tr) {
  const Gemv& g = cur_gemv();
  const Smem sh = smem_map(smem_raw);
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, t = lane & 3;
  const uint32_t K = g.K, ng = K / 64, T = g.T, W = NCW / T;
  const uint32_t team = warp / W, j = warp - team * W;
  const BatchBuf bb = batch_buf(sh, K, g.bs);
  int* status = prog().status;
  uint32_t it = itd & ~kDeadBit;
  bool dead = (itd & kDeadBit) != 0;
  // inputs of sequence g (B operand) and group scales of sequences 2t, 2t + 1 (the
  // outputs); sequences past the pass read sequence 0's (their results are unused)
  const uint16_t* xrow = bb.xf + (gq < nb ? gq : 0) * bb.stride + t * 16;
  const float2* sqa = bb.xsq + (2 * t < nb ? 2 * t : 0) * ng;
  const float2* sqb = bb.xsq + (2 * t + 1 < nb ? 2 * t + 1 : 0) * ng;
  float* mine = bb.part + warp * 128;         // [16 rows][8 sequences]
  const float* tp = bb.part + team * W * 128;  // the team's partials
  const uint64_t limit = wait_limit();
  // the down projection's residual rows of the pass's sequences, polled together
  // once (one L2 round trip) instead of per output inside the tile loop
  float* resid = bb.part + NCW * 128;  // [row - rb][nb]
  if (g.epi == 1) {
    const uint32_t rows = g.re - g.rb;
    for (uint32_t e = threadIdx.x; e < rows * nb; e += NCT) {
      const uint32_t rho = e / nb, sq = e - rho * nb;
      resid[e] = tagged_value(static_cast<const uint32_t*>(g.resid_in) + (size_t)(b0 + sq) * g.sres_in + g.rb + rho,
                              g.tag_r);
    }
    consumer_sync();
  }
  for (uint32_t tl = 0; tl < g.ntiles; ++tl, ++it) {
    const uint32_t st = slot_of(it);
    // every warp waits for every tile, its team's or not: a warp that skipped a
    // slot's phase could take a later phase of the slot for complete too early
    if (!dead && !mbar_wait(&sh.full[st], parity_of(it), limit)) {
      set_status(status, kStatusTimeout);
      dead = true;
    }
    if (tl % T != team) continue;
    if (tr && threadIdx.x == 0) {
      if (tl == 0) tr[4] = global_ns();
      if (tl + T >= g.ntiles) tr[5] = global_ns();
    }
    const uint32_t meta = dead ? 0u : sh.tmeta[st];
    const uint32_t r0 = meta & 0xFFFFFFu, nr = meta >> 24;
    float y[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    if (nr > 8) {
      batch_tile_groups<true>(sh.ring + sh.toff[st], nr, K, g.gstride, g.scale_off, g.bias_off, j, W, xrow, sqa,
                              sqb, y);
    } else if (nr) {
      batch_tile_groups<false>(sh.ring + sh.toff[st], nr, K, g.gstride, g.scale_off, g.bias_off, j, W, xrow, sqa,
                               sqb, y);
    }
    __syncwarp();
    if (lane == 0 && !dead) mbar_arrive_n(&sh.empty[st], T);
    mine[gq * 8 + 2 * t] = y[0][0];
    mine[gq * 8 + 2 * t + 1] = y[0][1];
    mine[(gq + 8) * 8 + 2 * t] = y[1][0];
    mine[(gq + 8) * 8 + 2 * t + 1] = y[1][1];
    named_barrier(2 + team, W * 32);
    for (uint32_t e = j * 32 + lane; e < nr * nb; e += W * 32) {
      const uint32_t rho = e / nb, s = e - rho * nb, row = r0 + rho;
      float acc = 0.f;
      for (uint32_t jj = 0; jj < W; ++jj) acc += tp[jj * 128 + rho * 8 + s];
      if (g.epi == 1) acc += resid[(row - g.rb) * nb + s];
      uint32_t sg = 0;
      while (sg + 1 < g.nseg && row >= g.row0[sg + 1]) ++sg;
      gemv_store(g, sg, (size_t)(b0 + s) * g.sout[sg] + row - g.row0[sg], acc);
    }
    named_barrier(2 + team, W * 32);  // the partials are read before the next tile's
  }
  if (tr && threadIdx.x == 0) tr[6] = global_ns();
  return it | (dead ? kDeadBit : 0u);
}

// ------------------------------------------------------------------ attention phases

struct Span {
  uint32_t pos, S, t0, t1, tc_end, ntiles;
  bool ok, has_fresh;
};

// The device position as this CTA read it at kernel start (shared memory).

// A paged cache's splits start at multiples of 8 tokens, so that no 8-token tile
// straddles two pool blocks.
__device__ __forceinline__ Span attn_span(const Program& P, uint32_t capacity, uint32_t b, bool paged) {
  Span sp;
  if (P.d_pos) {
    const int32_t p = launch_pos(b);
    const uint32_t lim = min(capacity, P.max_seq);
    sp.ok = p >= 0 && (uint32_t)p < lim;
    sp.pos = sp.ok ? (uint32_t)p : 0;
    sp.S = sp.pos + 1;
  } else {
    sp.ok = P.pos < capacity;
    sp.pos = P.pos;
    sp.S = P.S;
  }
  const uint32_t s = blockIdx.x;
  const bool mine = s < P.P && sp.ok;
  auto cut = [&](uint32_t k) {
    const uint32_t t = (uint32_t)(((uint64_t)sp.S * k) / P.P);
    return paged && k < P.P ? t & ~7u : t;
  };
  sp.t0 = mine ? cut(s) : 0;
  sp.t1 = mine ? cut(s + 1) : 0;
  sp.has_fresh = mine && sp.S == sp.pos + 1 && sp.pos >= sp.t0 && sp.pos < sp.t1;
  sp.tc_end = sp.has_fresh ? sp.pos : sp.t1;
  sp.ntiles = (mine && sp.tc_end > sp.t0) ? (sp.tc_end - sp.t0 + kTS - 1) / kTS : 0;
  return sp;
}

// RMSNorm over one head (this lane's EPL elements at d = lane*EPL, weights wv),
// rounded to bf16, then RoPE on dims [0, R) with rotate-half pairing, rounded to
// bf16; cs[i] = (cos, sin) of the position's angle for frequency i < R/2.
template <int EPL>
__device__ __forceinline__ void norm_rope(float* x, const float* wv, const Program& P, const float2* cs, float* buf,
                                          uint32_t lane) {
  const uint32_t D = EPL * 32, R = P.R, half = R / 2;
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) ss = fmaf(x[e], x[e], ss);
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)D + P.eps);
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    x[e] = round_bf16(x[e] * inv * wv[e]);
    buf[lane * EPL + e] = x[e];
  }
  __syncwarp();
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const uint32_t d = lane * EPL + e;
    if (d < R) {
      const float2 c = cs[d < half ? d : d - half];
      x[e] = d < half ? round_bf16(buf[d] * c.x - buf[d + half] * c.y) : round_bf16(buf[d] * c.x + buf[d - half] * c.y);
    }
  }
  __syncwarp();
}


// ------------------------------------------------------------------ Turbo8 helpers

// Orthonormal Walsh-Hadamard transform (Sylvester order) of one head's row, held
// EPL consecutive elements per lane: butterflies of stride h pair elements i and
// i + h (bit h of i clear) into (x_i + x_{i+h}, x_i - x_{i+h}); strides below EPL
// stay in the lane, larger ones pair lane with lane ^ (h / EPL). Then x 1/sqrt(D).
template <int EPL>
__device__ __forceinline__ void wht_row(float* x, uint32_t lane, float norm) {
#pragma unroll
  for (int h = 1; h < EPL; h <<= 1)
#pragma unroll
    for (int e = 0; e < EPL; ++e)
      if (!(e & h)) {
        const float a = x[e], b = x[e + h];
        x[e] = a + b;
        x[e + h] = a - b;
      }
#pragma unroll
  for (uint32_t m = 1; m < 32; m <<= 1)
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float p = __shfl_xor_sync(FULLMASK, x[e], m);
      x[e] = (lane & m) ? p - x[e] : x[e] + p;
    }
#pragma unroll
  for (int e = 0; e < EPL; ++e) x[e] *= norm;
}

// Two fp32 values as FP8 E4M3 (round to nearest even, saturating), x0 in the low
// byte; and two E4M3 codes (low byte first) back to fp32 (exact through f16).
__device__ __forceinline__ uint32_t e4m3x2_of(float x0, float x1) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x1), "f"(x0));
  return r;
}
__device__ __forceinline__ float2 e4m3x2_value(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}
// EPL codes (little-endian bytes) of a lane, as a word pair
template <int EPL>
__device__ __forceinline__ uint2 load_codes(const uint8_t* p) {
  if constexpr (EPL == 8) return *reinterpret_cast<const uint2*>(p);
  else if constexpr (EPL == 4) return make_uint2(*reinterpret_cast<const uint32_t*>(p), 0u);
  else return make_uint2(*reinterpret_cast<const uint16_t*>(p), 0u);
}
template <int EPL>
__device__ __forceinline__ void store_codes(uint8_t* p, uint2 c) {
  if constexpr (EPL == 8) *reinterpret_cast<uint2*>(p) = c;
  else if constexpr (EPL == 4) *reinterpret_cast<uint32_t*>(p) = c.x;
  else *reinterpret_cast<uint16_t*>(p) = (uint16_t)c.x;
}
template <int EPL>
__device__ __forceinline__ void dequant_codes(uint2 c, float s, float* x) {
#pragma unroll
  for (int e = 0; e < EPL; e += 2) {
    const uint32_t w = e < 4 ? c.x : c.y;
    const float2 v = e4m3x2_value(w >> (8 * (e % 4)));
    x[e] = v.x * s;
    x[e + 1] = v.y * s;
  }
}
// Turbo8 quantisation of a row held EPL per lane (groups of 16 on 16 / EPL lanes):
// scale = bf16(amax / 448), codes = E4M3(x / scale); returns the codes and the
// group's scale, and leaves the dequantised values (code * scale, exact) in x.
template <int EPL>
__device__ __forceinline__ uint2 turbo8_quant(float* x, float& scale) {
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int o = 1; o < 16 / EPL; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(FULLMASK, amax, o));
  const float s = round_bf16(amax / 448.f);
  uint2 c = make_uint2(0u, 0u);
#pragma unroll
  for (int e = 0; e < EPL; e += 2) {
    const uint32_t two = s > 0.f ? e4m3x2_of(x[e] / s, x[e + 1] / s) : 0u;
    if (e < 4) c.x |= two << (8 * e);
    else c.y |= two << (8 * (e - 4));
  }
  dequant_codes<EPL>(c, s, x);
  scale = s;
  return c;
}

// Split-KV attention of one split (CTA). Warp w serves the HPW consecutive q-heads
// of head group w % NG (one kv-head) and every TI-th tile, TI = 12 / NG; the TI
// partial softmax states of a head group are merged in shared memory at the end.
template <int D, int HPW, bool T8>
__device__ __noinline__ uint32_t attn_consume(uint32_t itd, uint32_t ph, unsigned long long* tr) {
  uint32_t it = itd & ~kDeadBit;
  bool dead = (itd & kDeadBit) != 0;
  const Program& P = prog();
  const LayerDesc& L = cur_layer();
  const Smem sh = smem_map(smem_raw);
  constexpr int EPL = D / 32;
  constexpr int NV = HPW * kTS;
  constexpr int SH = NV == 8 ? 2 : NV == 16 ? 1 : 0;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t s = blockIdx.x;
  const Span sp = attn_span(P, L.capacity, s_seq.b, L.btab != nullptr);
  constexpr bool t8 = T8;  // the cache's format: Turbo8 (rotated basis) or bf16
  const uint32_t H = P.H, Hkv = P.Hkv, rowh = Hkv * D, rowbytes = rowh * (t8 ? 1 : 2);
  const uint32_t sstride = turbo8_sstride(Hkv, D), srow = t8 ? sstride * 2 : 0u;
  const uint32_t part = kTS * (rowbytes + srow);  // a tile's K part (rows, then Turbo8 scales); V follows
  const uint32_t NG = H / HPW, TI = NCW / NG;  // warps beyond NG * TI only keep the ring moving
  if (!sp.ok) {
    if (s == 0 && threadIdx.x == 0) set_status(P.status, kStatusRange);
    return itd;
  }
  if (s >= P.P) return itd;
  float2* cs = reinterpret_cast<float2*>(sh.uni);        // RoPE (cos, sin), [R/2]
  float* fresh = reinterpret_cast<float*>(sh.uni) + 256;  // k then v, [Hkv][D] each
  float* buf = fresh + 2 * rowh;                          // per-warp [D] for RoPE, then merge space
  // the position's rotation angles, once per CTA: fp32 angle, accurate sin/cos
  if (threadIdx.x < P.R / 2) {
    float sn, cn;
    sincosf((float)sp.pos * P.inv_freq[threadIdx.x], &sn, &cn);
    cs[threadIdx.x] = make_float2(cn, sn);
  }
  // every load of the phase's inputs in one batch: this warp's q-heads and their
  // norm weights; for the appending CTA, the new token's k and v rows
  const bool appender = sp.has_fresh || (sp.S != sp.pos + 1 && s == 0);
  const uint32_t hg = warp % NG, ti = warp / NG;
  const bool active = ti < TI;
  const uint32_t h0 = hg * HPW, g = h0 / (H / Hkv);
  float q[HPW][EPL], m[HPW], l[HPW], acc[HPW][EPL], qw[EPL];
  const uint32_t tin = phase_tag(ph - 1);  // q, k, v: the projection phase before
  const uint32_t* qf = reinterpret_cast<const uint32_t*>(s_seq.scratch + P.sm.q_full);
  load_row<EPL>(L.q_norm + lane * EPL, qw);
  const bool kv_warp = appender && warp < Hkv;
  float kx[EPL], vx[EPL], kw[EPL];
  if (kv_warp) load_row<EPL>(L.k_norm + lane * EPL, kw);
  {  // this warp's q-heads and, for the appending CTA, the new k and v: polled together
    constexpr int NR = HPW + 2;  // rows of EPL tagged words per lane
    const uint32_t* rows[NR];
#pragma unroll
    for (int j = 0; j < HPW; ++j) rows[j] = qf + (size_t)(h0 + j) * 2 * D + lane * EPL;
    rows[HPW] = reinterpret_cast<const uint32_t*>(s_seq.scratch + P.sm.k) + warp * D + lane * EPL;
    rows[HPW + 1] = reinterpret_cast<const uint32_t*>(s_seq.scratch + P.sm.v) + warp * D + lane * EPL;
    bool ok;
    if constexpr (EPL % 4 == 0) {
      constexpr int G = EPL / 4, N = NR * G;
      const uint32_t* pp[N];
      uint32_t pt[N];
      uint4 w[N];
#pragma unroll
      for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int k = 0; k < G; ++k) {
          pp[r * G + k] = rows[r] + 4 * k;
          pt[r * G + k] = (r < HPW || kv_warp) ? tin : 0u;
          w[r * G + k] = pt[r * G + k] ? ld_tagged4(pp[r * G + k]) : make_uint4(0u, 0u, 0u, 0u);
        }
      ok = settle4<N>(pp, pt, w);
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        float* dst = r < HPW ? q[r < HPW ? r : 0] : (r == HPW ? kx : vx);
#pragma unroll
        for (int k = 0; k < G; ++k) {
          dst[4 * k] = tag_value(w[r * G + k].x);
          dst[4 * k + 1] = tag_value(w[r * G + k].y);
          dst[4 * k + 2] = tag_value(w[r * G + k].z);
          dst[4 * k + 3] = tag_value(w[r * G + k].w);
        }
      }
    } else {
      constexpr int N = NR * EPL;
      const uint32_t* pp[N];
      uint32_t pt[N];
      uint32_t w[N];
#pragma unroll
      for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int k = 0; k < EPL; ++k) {
          pp[r * EPL + k] = rows[r] + k;
          pt[r * EPL + k] = (r < HPW || kv_warp) ? tin : 0u;
          w[r * EPL + k] = pt[r * EPL + k] ? ld_tagged(pp[r * EPL + k]) : 0u;
        }
      ok = settle1<N>(pp, pt, w);
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        float* dst = r < HPW ? q[r < HPW ? r : 0] : (r == HPW ? kx : vx);
#pragma unroll
        for (int k = 0; k < EPL; ++k) dst[k] = tag_value(w[r * EPL + k]);
      }
    }
    if (!ok) set_status(P.status, kStatusTimeout);
  }
  consumer_sync();  // the angle table
  const float wnorm = rsqrtf((float)D);  // the WHT's 1/sqrt(D)
  if (kv_warp) {  // the new token's k (normed, rotated) and v: appended by exactly one CTA
    norm_rope<EPL>(kx, kw, P, cs, buf + warp * D, lane);
    if (t8) {
      // Turbo8: k and v rotated (bf16), quantised per 16, appended as codes and
      // scales; the fresh row keeps the dequantised values every split reads
      wht_row<EPL>(kx, lane, wnorm);
      wht_row<EPL>(vx, lane, wnorm);
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        kx[e] = round_bf16(kx[e]);
        vx[e] = round_bf16(vx[e]);
      }
      if (P.dump) {
        uint16_t* kr = reinterpret_cast<uint16_t*>(s_seq.scratch + P.sm.k_rot) + warp * D + lane * EPL;
        uint16_t* vr = reinterpret_cast<uint16_t*>(s_seq.scratch + P.sm.v_rot) + warp * D + lane * EPL;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          kr[e] = to_bf16(kx[e]);
          vr[e] = to_bf16(vx[e]);
        }
      }
      float sk, sv;
      const uint2 ck = turbo8_quant<EPL>(kx, sk), cv = turbo8_quant<EPL>(vx, sv);
      const size_t row = (size_t)sp.pos * rowh + warp * D + lane * EPL;
      store_codes<EPL>(L.kc + row, ck);
      store_codes<EPL>(L.vc + row, cv);
      if ((lane * EPL) % 16 == 0) {
        const size_t si = (size_t)sp.pos * sstride + (warp * D + lane * EPL) / 16;
        L.ks[si] = to_bf16(sk);
        L.vs[si] = to_bf16(sv);
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        fresh[warp * D + lane * EPL + e] = kx[e];
        fresh[rowh + warp * D + lane * EPL + e] = vx[e];
      }
    } else {
      const size_t prow = kv_row(L, sp.pos);  // paged: the row in the pool
      uint16_t* kd = reinterpret_cast<uint16_t*>(L.kc) + prow * rowh + warp * D + lane * EPL;
      uint16_t* vd = reinterpret_cast<uint16_t*>(L.vc) + prow * rowh + warp * D + lane * EPL;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        fresh[warp * D + lane * EPL + e] = kx[e];
        fresh[rowh + warp * D + lane * EPL + e] = vx[e];
        kd[e] = to_bf16(kx[e]);
        vd[e] = to_bf16(vx[e]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < HPW; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[j][e] = 0.f;
    if (active) {
      norm_rope<EPL>(q[j], qw, P, cs, buf + warp * D, lane);
      if (t8) {  // q rotated into the cache's basis (bf16)
        wht_row<EPL>(q[j], lane, wnorm);
#pragma unroll
        for (int e = 0; e < EPL; ++e) q[j][e] = round_bf16(q[j][e]);
      }
    }
  }
  consumer_sync();  // the fresh row is visible to every warp; the RoPE buffers are free
  if (tr && threadIdx.x == 0) tr[3] = global_ns();

  const uint32_t midx = lane >> SH, mj = midx / kTS, mt = midx % kTS;
  const uint64_t limit = wait_limit();
  for (uint32_t i = 0; i < sp.ntiles; ++i) {
    const uint32_t st = slot_of(it);
    const bool mine = active && (i % TI) == ti;
    // every warp waits for every tile before releasing it, so no warp can run a
    // ring round ahead and complete a slot's release early
    if (!dead && !mbar_wait(&sh.full[st], parity_of(it), limit)) {
      set_status(P.status, kStatusTimeout);
      dead = true;
    }
    if (tr && threadIdx.x == 0) {
      if (i == 0) tr[4] = global_ns();
      if (i + 1 == sp.ntiles) tr[5] = global_ns();
    }
    if (mine && !dead) {
      const uint8_t* base = sh.ring + sh.toff[st];
      const uint32_t n = min((uint32_t)kTS, sp.tc_end - (sp.t0 + i * kTS));
      float d[NV];
      // Turbo8: a lane's EPL elements lie in one group of 16, so its K scale multiplies
      // the lane's partial score once and its V scale folds into the token's weight
      const uint32_t sidx = (g * D + lane * EPL) / 16;  // this lane's group in a token's scale row
      float vsc[kTS];
#pragma unroll
      for (int t = 0; t < kTS; ++t) {  // rows t >= n hold stale data: their scores are masked
        float kf[EPL];
        float ksc = 1.f;
        if constexpr (T8) {
          dequant_codes<EPL>(load_codes<EPL>(base + t * rowbytes + g * D + lane * EPL), 1.f, kf);
          ksc = bf16f(reinterpret_cast<const uint16_t*>(base + kTS * rowbytes + t * srow)[sidx]);
          vsc[t] = bf16f(reinterpret_cast<const uint16_t*>(base + part + kTS * rowbytes + t * srow)[sidx]);
        } else {
          load_row<EPL>(reinterpret_cast<const uint16_t*>(base + t * rowbytes) + g * D + lane * EPL, kf);
        }
#pragma unroll
        for (int j = 0; j < HPW; ++j) {
          float x = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) x = fmaf(q[j][e], kf[e], x);
          d[j * kTS + t] = T8 ? x * ksc : x;
        }
      }
      float sc = reduce_transposed<NV>(d, lane) * P.scale_log2;
      sc = mt < n ? sc : -INFINITY;
      float mx = sc;
#pragma unroll
      for (int o = 1 << SH; o < (kTS << SH); o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(FULLMASK, mx, o));
      float mold = m[0];
#pragma unroll
      for (int j = 1; j < HPW; ++j) mold = mj == (uint32_t)j ? m[j] : mold;
      const float mnew = fmaxf(mold, mx);
      const float p = exp2f(sc - mnew);
      float ps = p;
#pragma unroll
      for (int o = 1 << SH; o < (kTS << SH); o <<= 1) ps += __shfl_xor_sync(FULLMASK, ps, o);
#pragma unroll
      for (int j = 0; j < HPW; ++j) {
        const float mn = __shfl_sync(FULLMASK, mnew, (j * kTS) << SH);
        const float sum = __shfl_sync(FULLMASK, ps, (j * kTS) << SH);
        const float corr = exp2f(m[j] - mn);
        l[j] = fmaf(l[j], corr, sum);
        m[j] = mn;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[j][e] *= corr;
      }
      // unrolled over the tile's rows (independent loads); rows t >= n hold stale
      // bytes that may not even be finite, so they are selected out, not weighted by 0
#pragma unroll
      for (uint32_t t = 0; t < (uint32_t)kTS; ++t) {
        float vf[EPL];
        if constexpr (T8)
          dequant_codes<EPL>(load_codes<EPL>(base + part + t * rowbytes + g * D + lane * EPL), 1.f, vf);
        else
          load_row<EPL>(reinterpret_cast<const uint16_t*>(base + part + t * rowbytes) + g * D + lane * EPL, vf);
        const bool live = t < n;
#pragma unroll
        for (int j = 0; j < HPW; ++j) {
          float pj = __shfl_sync(FULLMASK, p, (j * kTS + t) << SH);
          if constexpr (T8) pj *= vsc[t];
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[j][e] = live ? fmaf(pj, vf[e], acc[j][e]) : acc[j][e];
        }
      }
    }
    __syncwarp();
    if (lane == 0 && !dead) mbar_arrive(&sh.empty[st]);  // every warp releases every tile
    ++it;
  }
  if (sp.has_fresh && ti == 0) {
    float kf[EPL], vf[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      kf[e] = fresh[g * D + lane * EPL + e];
      vf[e] = fresh[rowh + g * D + lane * EPL + e];
    }
#pragma unroll
    for (int j = 0; j < HPW; ++j) {
      float x = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) x = fmaf(q[j][e], kf[e], x);
      const float sc = warp_sum(x) * P.scale_log2;
      const float mn = fmaxf(m[j], sc);
      const float corr = exp2f(m[j] - mn), pp = exp2f(sc - mn);
      l[j] = fmaf(l[j], corr, pp);
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[j][e] = fmaf(acc[j][e], corr, pp * vf[e]);
      m[j] = mn;
    }
  }
  if (tr && threadIdx.x == 0) tr[6] = global_ns();
  // merge the TI partial states of each head group: the warps of token split u
  // hand theirs over one split at a time ([NG][HPW][D + 2] floats)
  float* mb = buf;
  for (uint32_t u = 1; u < TI; ++u) {
    if (active && ti == u) {
      float* dst = mb + hg * HPW * (D + 2);
#pragma unroll
      for (int j = 0; j < HPW; ++j) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) dst[j * (D + 2) + lane * EPL + e] = acc[j][e];
        if (lane == 0) {
          dst[j * (D + 2) + D] = m[j];
          dst[j * (D + 2) + D + 1] = l[j];
        }
      }
    }
    consumer_sync();
    if (ti == 0) {
      const float* src = mb + hg * HPW * (D + 2);
#pragma unroll
      for (int j = 0; j < HPW; ++j) {
        const float mu = src[j * (D + 2) + D], lu = src[j * (D + 2) + D + 1];
        if (mu == -INFINITY) continue;
        const float mn = fmaxf(m[j], mu);
        const float c0 = exp2f(m[j] - mn), c1 = exp2f(mu - mn);
        l[j] = l[j] * c0 + lu * c1;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[j][e] = acc[j][e] * c0 + src[j * (D + 2) + lane * EPL + e] * c1;
        m[j] = mn;
      }
    }
    consumer_sync();
  }
  if (ti == 0) {
    float* part_o = reinterpret_cast<float*>(s_seq.scratch + P.sm.part_o);
    float* part_ml = reinterpret_cast<float*>(s_seq.scratch + P.sm.part_ml);
#pragma unroll
    for (int j = 0; j < HPW; ++j) {
      const uint32_t h = h0 + j;
      float* po = part_o + ((size_t)s * H + h) * D + lane * EPL;
#pragma unroll
      for (int e = 0; e < EPL; ++e) po[e] = acc[j][e];
      if (lane == 0) {
        part_ml[((size_t)s * H + h) * 2] = m[j];
        part_ml[((size_t)s * H + h) * 2 + 1] = l[j];
      }
    }
  }
  consumer_sync();  // the merge space is free again; every partial of the split is stored
  if (threadIdx.x == 0) {  // publish them: the split's flag, released at GPU scope
    uint32_t* flags = reinterpret_cast<uint32_t*>(s_seq.scratch + P.sm.flags);
    st_release(flags + s, phase_tag(ph));
  }
  return it | (dead ? kDeadBit : 0u);
}

// Merge of the P partials of (head h, 32 dims) per CTA, then the output gate:
// ga = bf16(bf16(attn) * sigmoid(gate)). A split's partials are read once its flag
// carries the attention phase's tag (acquire), through L2.
__device__ __forceinline__ float ld_f32_l2(const float* p) {
  float r;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(r) : "l"(p) : "memory");
  return r;
}
__device__ __noinline__ void combine_consume(uint32_t ph) {
  const Program& P = prog();
  const LayerDesc& L = cur_layer();
  const Smem sh = smem_map(smem_raw);
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t nd = P.D / 32, item = blockIdx.x;
  const Span sp = attn_span(P, L.capacity, s_seq.b, L.btab != nullptr);
  if (item >= P.H * nd) return;
  const uint32_t h = item / nd, d = (item % nd) * 32 + lane;
  uint32_t* ga = reinterpret_cast<uint32_t*>(s_seq.scratch + P.sm.ga);
  const uint32_t tag = phase_tag(ph);
  if (!sp.ok) {
    if (warp == 0) st_tagged(ga + (size_t)h * P.D + d, tag_word(0.f, tag));
    return;
  }
  const float* part_o = reinterpret_cast<const float*>(s_seq.scratch + P.sm.part_o);
  const float* part_ml = reinterpret_cast<const float*>(s_seq.scratch + P.sm.part_ml);
  const uint32_t* flags = reinterpret_cast<const uint32_t*>(s_seq.scratch + P.sm.flags);
  const uint32_t tflag = phase_tag(ph - 1);
  const uint64_t limit = wait_limit();
  bool ok = true;
  float M = -INFINITY, Ls = 0.f, O = 0.f;
  for (uint32_t base = 0; base < P.P; base += NCW * 4) {
    float ms[4], ls[4], os[4];
    {  // the splits' flags first (polled together), then their partials
      uint32_t todo = 0, f[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t sp_ = base + warp + NCW * k;
        f[k] = sp_ < P.P ? ld_acquire(flags + sp_) : tflag;
        if (f[k] != tflag) todo |= 1u << k;
      }
      if (todo) {
        const uint64_t t0 = global_ns();
        for (uint32_t n = 1; todo; ++n) {
          __nanosleep(64);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if ((todo >> k) & 1u) f[k] = ld_acquire(flags + base + warp + NCW * k);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (((todo >> k) & 1u) && f[k] == tflag) todo &= ~(1u << k);
          if (todo && (global_ns() - t0 > limit || ((n & 15) == 0 && timed_out(P.status)))) {
            ok = false;
            break;
          }
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t sp_ = base + warp + NCW * k;
      const bool in = sp_ < P.P;
      ms[k] = in ? ld_f32_l2(part_ml + ((size_t)sp_ * P.H + h) * 2) : -INFINITY;
      ls[k] = in ? ld_f32_l2(part_ml + ((size_t)sp_ * P.H + h) * 2 + 1) : 0.f;
      os[k] = in ? ld_f32_l2(part_o + ((size_t)sp_ * P.H + h) * P.D + d) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (ms[k] == -INFINITY) continue;  // a split with no tokens
      const float mn = fmaxf(M, ms[k]);
      const float c0 = exp2f(M - mn), c1 = exp2f(ms[k] - mn);
      Ls = Ls * c0 + ls[k] * c1;
      O = O * c0 + os[k] * c1;
      M = mn;
    }
  }
  float gate = 0.f;
  if (warp == 0) {
    uint32_t w;
    ok &= ld_tagged_wait(reinterpret_cast<const uint32_t*>(s_seq.scratch + P.sm.q_full) + (size_t)h * 2 * P.D + P.D + d,
                         phase_tag(ph - 2), w, limit, P.status);
    gate = tag_value(w);
  }
  if (!ok) set_status(P.status, kStatusTimeout);
  float* part = reinterpret_cast<float*>(sh.uni);  // [3][16][32]
  part[(0 * NCW + warp) * 32 + lane] = M;
  part[(1 * NCW + warp) * 32 + lane] = Ls;
  part[(2 * NCW + warp) * 32 + lane] = O;
  consumer_sync();
  if (warp == 0) {
    M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NCW; ++w) M = fmaxf(M, part[w * 32 + lane]);
    Ls = 0.f;
    O = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) {
      const float mw = part[w * 32 + lane];
      if (mw == -INFINITY) continue;
      const float c = exp2f(mw - M);
      Ls = fmaf(part[(NCW + w) * 32 + lane], c, Ls);
      O = fmaf(part[(2 * NCW + w) * 32 + lane], c, O);
    }
    const float attn = round_bf16(O / Ls);
    // a Turbo8 layer's output is still in the rotated basis: the o_proj prologue
    // rotates each head back and applies the gate there
    st_tagged(ga + (size_t)h * P.D + d, tag_word(L.kv_dtype == kKvTurbo8 ? attn : attn * sigmoidf_(gate), tag));
  }
  consumer_sync();
}

// ------------------------------------------------------------------ Gated DeltaNet phase

// Work item (v-head h, 32 state columns j) per CTA. Given the head's q, k, gate and
// beta, state columns are independent:
//   u_v = sum_i (g S[i][v]) k_i,  S[i][v] <- g S[i][v] + k_i beta (v_v - u_v),
//   y_v = sum_i S[i][v] q_i / sqrt(Dk),
// so the [Dk][32] fp32 slice is read into registers once (it arrives through the
// ring while the layer's input projection streams: nothing before it in the step
// writes the state), updated, and written once.
constexpr int kGdnWarps = 8;  // warps holding state rows (Dk / 8 rows each)
// The linear-attention phase's inputs that do not depend on the step's earlier
// phases (the CTA's state block [Dk][32] fp32, its channels' convolution state
// [2 Dk + 32][Kc] fp32 and weights [2 Dk + 32][Kc] bf16) come as one ring tile per
// sequence, right after the layer's input projection tiles.
__host__ __device__ inline uint32_t gdn_tile_bytes(uint32_t Dk, uint32_t Kc) { return Dk * 128 + (2 * Dk + 32) * Kc * 6; }

// The CTA's linear-attention work item: v-head h, columns [v0, v0 + 32) of its state.
struct GdnItem {
  bool ok;
  uint32_t h, j, hk, v0;
};
__device__ __forceinline__ GdnItem gdn_item(const Program& P) {
  GdnItem it;
  const uint32_t nsl = P.Dv / 32;
  it.ok = blockIdx.x < P.Hv * nsl;
  it.h = it.ok ? blockIdx.x / nsl : 0;
  it.j = it.ok ? blockIdx.x % nsl : 0;
  it.hk = it.h / (P.Hv / P.Hk);
  it.v0 = it.j * 32;
  return it;
}

// The convolution state of the q/k channels, shifted by one token (newest last):
// the linear-attention phase reads it in every CTA of the channel's v-heads, so it
// is written in the output projection phase, after that phase's input (the readout
// of every linear-attention CTA, hence after all their reads of it) is in, each CTA
// taking a share of the channels (one warp). tag: that of qkv.
__device__ __noinline__ void conv_shift_qk(float* conv_state, const uint8_t* scratch, uint32_t tag) {
  const Program& P = prog();
  const uint32_t lane = threadIdx.x & 31, Kc = P.Kc;
  const uint32_t nqk = 2 * P.Hk * P.Dk, per = (nqk + gridDim.x - 1) / gridDim.x;
  const uint32_t c0 = blockIdx.x * per, c1 = min(nqk, c0 + per);
  const uint32_t* qkv = reinterpret_cast<const uint32_t*>(scratch + P.sm.qkv);
  for (uint32_t ch = c0 + lane; ch < c1; ch += 32) {
    float* cs = conv_state + (size_t)ch * Kc;
    const float x = tagged_value(qkv + ch, tag);
    float v[kMaxKc];
#pragma unroll
    for (int t = 0; t < kMaxKc; ++t) v[t] = t + 1 < (int)Kc ? cs[t + 1] : x;
#pragma unroll
    for (int t = 0; t < kMaxKc; ++t)
      if (t < (int)Kc) cs[t] = v[t];
  }
}

template <int DK>
__device__ __noinline__ uint32_t gdn_consume(uint32_t itd, uint32_t ph) {
  const Program& P = prog();
  const LayerDesc& L = cur_layer();
  const Smem sh = smem_map(smem_raw);
  constexpr int RPT = DK / kGdnWarps;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const GdnItem w = gdn_item(P);
  if (!w.ok) return itd;  // (uniform over the CTA)
  const uint32_t h = w.h, v0 = w.v0, Kc = P.Kc;
  float* act = reinterpret_cast<float*>(sh.uni);  // [2 Dk + 32]
  float* red = act + 2 * DK + 32;                 // [2][NCW][32]
  const uint32_t tin = phase_tag(ph - 1);  // qkv, dt_raw, b_raw: the projection phase before
  // this channel (thread < 2 Dk + 32): q, k of the k-head, v of the slice
  const bool chan = tid < 2 * DK + 32;
  const uint32_t ch = tid < DK ? w.hk * DK + tid
                    : tid < 2 * DK ? P.Hk * DK + w.hk * DK + (tid - DK)
                                   : 2 * P.Hk * DK + h * P.Dv + v0 + (tid - 2 * DK);
  const uint32_t* qkv = reinterpret_cast<const uint32_t*>(s_seq.scratch + P.sm.qkv);
  float x = 0.f;
  {
    const uint32_t* pp[1] = {qkv + (chan ? ch : 0u)};
    const uint32_t pt[1] = {chan ? tin : 0u};
    uint32_t w[1] = {chan ? ld_tagged(pp[0]) : 0u};
    if (!settle1<1>(pp, pt, w)) set_status(P.status, kStatusTimeout);
    x = tag_value(w[0]);
  }
  float alog = 0.f, dtb = 0.f, dtr = 0.f, brw = 0.f;
  if (tid == 0) {
    alog = L.a_log[h];
    dtb = bf16f(L.dt_bias[h]);
    const uint32_t* pp[2] = {reinterpret_cast<const uint32_t*>(s_seq.scratch + P.sm.dt_raw) + h,
                             reinterpret_cast<const uint32_t*>(s_seq.scratch + P.sm.b_raw) + h};
    const uint32_t pt[2] = {tin, tin};
    uint32_t w[2] = {ld_tagged(pp[0]), ld_tagged(pp[1])};
    if (!settle1<2>(pp, pt, w)) set_status(P.status, kStatusTimeout);
    dtr = tag_value(w[0]);
    brw = tag_value(w[1]);
  }
  const uint32_t slot = slot_of(itd & ~kDeadBit);
  if (!(itd & kDeadBit) && !mbar_wait(&sh.full[slot], parity_of(itd & ~kDeadBit), wait_limit())) {
    set_status(P.status, kStatusTimeout);
    itd |= kDeadBit;
  }
  const bool dead = (itd & kDeadBit) != 0;
  // after a wait ran out the tile is not read (it may still be arriving)
  const float* st_s = reinterpret_cast<const float*>(sh.ring + (dead ? 0u : sh.toff[slot]));
  const float* cs_s = st_s + DK * 32;
  const uint16_t* cw_s = reinterpret_cast<const uint16_t*>(cs_s + (2 * DK + 32) * Kc);
  // causal conv update + SiLU
  if (chan) {
    // v channels belong to this CTA alone and are written here; the q/k channels of
    // a k-head are read by every CTA of its v-heads during this phase, so
    // conv_shift_qk shifts them in the next one
    float* cnew = tid >= 2 * DK && !dead ? L.conv_state + (size_t)ch * Kc : nullptr;
    float o = 0.f;
    for (uint32_t t = 0; t < Kc; ++t) {
      const float sv = t + 1 < Kc ? cs_s[tid * Kc + t + 1] : x;  // shift left, newest last
      o = fmaf(bf16f(cw_s[tid * Kc + t]), sv, o);
      if (cnew) cnew[t] = sv;
    }
    act[tid] = siluf_(o);
  }
  if (tid == 0) {
    // gate = exp(softplus(dt + dt_bias) * -exp(A_log)); beta = sigmoid(b)
    const float xd = dtr + dtb;
    const float spl = xd > 20.f ? xd : log1pf(expf(xd));
    sh.misc[0] = expf(spl * -expf(alog));
    sh.misc[1] = sigmoidf_(brw);
  }
  consumer_sync();
  // per-head L2 norm of q and k (eps 1e-6), then bf16 as qkv_smooth is
  {
    float sq = 0.f, sk = 0.f;
    for (uint32_t i = tid; i < DK; i += NCT) {
      sq = fmaf(act[i], act[i], sq);
      sk = fmaf(act[DK + i], act[DK + i], sk);
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    if (lane == 0) {
      red[warp] = sq;
      red[32 + warp] = sk;
    }
    consumer_sync();
    float tq = 0.f, tk = 0.f;
#pragma unroll
    for (int i = 0; i < NCW; ++i) {
      tq += red[i];
      tk += red[32 + i];
    }
    const float iq = rsqrtf(tq + P.l2_eps), ik = rsqrtf(tk + P.l2_eps);
    consumer_sync();
    for (uint32_t i = tid; i < 2 * DK + 32; i += NCT) {
      const float v = act[i];
      act[i] = round_bf16(i < DK ? v * iq : (i < 2 * DK ? v * ik : v));
    }
    if (P.dump && chan) {  // debug: qkv_smooth (q/k channels by the k-head's first CTA)
      const bool first = w.j == 0 && w.h % (P.Hv / P.Hk) == 0;
      if (tid >= 2 * DK || first)
        reinterpret_cast<uint16_t*>(s_seq.scratch + P.sm.qkv_smooth)[ch] = to_bf16(act[tid]);
    }
    consumer_sync();
  }
  // delta rule on the slice: thread (warp, lane) of the first 8 warps holds rows
  // warp*RPT + r of column lane
  const float g = sh.misc[0], beta = sh.misc[1];
  const float* qv = act;
  const float* kv = act + DK;
  const bool holder = warp < kGdnWarps;
  float st[RPT];
  float u = 0.f;
  if (holder) {
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      st[r] = st_s[(warp * RPT + r) * 32 + lane] * g;
      u = fmaf(st[r], kv[warp * RPT + r], u);
    }
    red[warp * 32 + lane] = u;
  }
  consumer_sync();
  if (lane == 0 && !dead) mbar_arrive(&sh.empty[slot]);  // the tile is read (every warp releases it)
  ++itd;
  u = 0.f;
#pragma unroll
  for (int w = 0; w < kGdnWarps; ++w) u += red[w * 32 + lane];
  const float delta = beta * (act[2 * DK + lane] - u);
  float y = 0.f;
  if (holder) {
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      st[r] = fmaf(kv[warp * RPT + r], delta, st[r]);
      y = fmaf(st[r], qv[warp * RPT + r], y);
    }
    float* sp = L.ssm + ((size_t)blockIdx.x * DK + warp * RPT) * 32 + lane;  // block (h, v0 / 32)
    if (!dead) {
#pragma unroll
      for (int r = 0; r < RPT; ++r) sp[r * 32] = st[r];
    }
    red[kGdnWarps * 32 + warp * 32 + lane] = y;
  }
  consumer_sync();
  if (warp == 0) {
    y = 0.f;
#pragma unroll
    for (int w = 0; w < kGdnWarps; ++w) y += red[kGdnWarps * 32 + w * 32 + lane];
    uint32_t* yo = reinterpret_cast<uint32_t*>(s_seq.scratch + P.sm.y);
    st_tagged(yo + (size_t)h * P.Dv + v0 + lane, tag_word(y * P.gdn_out_scale, phase_tag(ph)));
  }
  consumer_sync();
  return itd;
}

// ------------------------------------------------------------------ producer schedule

// The producer walks the CTA's tiles of the whole launch, phase after phase and,
// within a phase, sequence after sequence (a batch's projections: pass after
// pass), in the order the consumers take them. Everything that changes per tile
// lives in registers; the current layer and GEMV descriptions and the ring
// placement of the tiles in flight sit in shared memory and are read once per
// phase or segment (a walk that keeps its cursor in memory costs a chain of
// dependent loads per tile, and the producer's issue rate bounds the stream).
struct ProdShared {
  LayerDesc L;
  Gemv g;
  uint32_t vstart[kDecSlots];  // ring placement of the tiles in flight
};
__shared__ ProdShared s_prod;

// Tile i takes slot i % kDecSlots and the ring bytes [v_i, v_i + span_i) of a
// virtual byte stream, placed at v_i mod the ring's size; a tile that would cross
// the ring's end starts at the next multiple of the size. It may be written once
// every tile that started more than size - span_i bytes before its end is consumed,
// and once the slot's previous tile (i - kDecSlots) is. Consumption is in order, so
// `vcons` (the start of the oldest unconsumed tile) and `tail` (its index) describe
// all of it.
struct Ring {
  uint32_t i, tail, vnext, vcons, size;  // size: the ring's bytes
  bool dead;
};

// Room for tile rg.i (span bytes in the ring, `total` bytes arriving): waits
// (bounded) until the tiles it overwrites are consumed, publishes its ring offset
// and GEMV rows, and arms its slot's full barrier. Null once a wait has run out.
__device__ __forceinline__ uint8_t* ring_claim(Ring& rg, const Smem& sh, uint32_t span, uint32_t total,
                                               uint32_t meta, uint32_t tout, int* status) {
  span = (span + 127) & ~127u;
  uint32_t v = rg.vnext, ph = v % rg.size;
  if (ph + span > rg.size) {
    v += rg.size - ph;
    ph = 0;
  }
  while (rg.tail < rg.i && (rg.i - rg.tail >= (uint32_t)kDecSlots || v + span - rg.vcons > rg.size)) {
    if (!mbar_wait(&sh.empty[slot_of(rg.tail)], parity_of(rg.tail), wait_limit())) {
      set_status(status, kStatusTimeout);
      rg.dead = true;
      return nullptr;
    }
    ++rg.tail;
    rg.vcons = rg.tail < rg.i ? s_prod.vstart[slot_of(rg.tail)] : v;
  }
  const uint32_t st = slot_of(rg.i);
  s_prod.vstart[st] = v;
  sh.toff[st] = ph;
  sh.tmeta[st] = meta;
  s_tout[st] = tout;
  mbar_arrive_expect_tx(&sh.full[st], total);
  rg.vnext = v + span;
  return sh.ring + ph;
}

// The producer (one thread). Weights are read from HBM by a batch's first pass
// over a phase and kept in L2 for the others (evict-last), the last pass marking
// them evict-first. Before it returns it waits (bounded) for every copy it issued
// that the consumers have not released, so that none is in flight when the CTA
// exits (consumers stop taking tiles after one of their waits has run out).
__device__ __noinline__ void produce_all(const LayerDesc* layers) {
  const Program& P = prog();
  const Smem sh = smem_map(smem_raw);
  const uint64_t stream = policy_evict_first(), keep = policy_evict_last();
  int* const status = P.status;
  unsigned long long* const trace = P.trace;
  const uint32_t trace_phases = P.trace_phases, n_layers = P.n_layers, batch = P.batch;
  Ring rg = {0u, 0u, 0u, 0u, P.ring_bytes, false};
  uint32_t phc = 0;  // phases opened (the timeline's phase index + 1)
  bool fresh = false;
  // timeline: when the phase's first tile is issued
  auto issued = [&]() {
    if (fresh) {
      fresh = false;
      if (trace && phc - 1 < trace_phases) trace[((size_t)blockIdx.x * trace_phases + phc - 1) * kTraceSlots + 7] = global_ns();
    }
    ++rg.i;
  };
  for (uint32_t l = 0; l < n_layers; ++l) {
    s_prod.L = layers[l];
    const LayerDesc& L = s_prod.L;
    const int np = n_phases(L.kind);
    for (int p = 0; p < np; ++p) {
      ++phc;
      fresh = true;
      const int ty = phase_type(L.kind, p);
      if (ty == kPhGemv) {
        gemv_of(P, L, l, p, 0, 0, s_prod.g);
        const Gemv& g = s_prod.g;
        const uint32_t K = g.K, gs = g.gstride, R = g.R, soff = g.scale_off, boff = g.bias_off;
        const uint32_t span = boff + R * gs * 2, rb = g.rb, re = g.re, nseg = g.nseg;
        const uint32_t npass = batch > 1 ? g.npass : 1u;
        if (g.epi == 3) {  // a single sequence's gate|up: the CTA's gate rows, then the same up rows
          const uint32_t lo = g.pr0, n = g.pn;
          for (uint32_t sg = 0; sg < 2; ++sg)
            for (uint32_t r = lo; r < lo + n; r += R) {
              const uint32_t nr = min(R, lo + n - r), cb = nr * K, sb = nr * gs * 2;
              // the tile's first row as its place in the partial sums: gate 0 .. n-1, up n .. 2n-1
              uint8_t* dst = ring_claim(rg, sh, span, cb + 2 * sb, (sg * n + r - lo) | (nr << 24), 0u, status);
              if (!dst) goto drain;
              uint64_t* fb = &sh.full[slot_of(rg.i)];
              bulk_g2s_stream(dst, g.seg[sg].codes + (size_t)r * K, cb, fb, stream);
              bulk_g2s_stream(dst + soff, g.seg[sg].scales + (size_t)r * gs, sb, fb, stream);
              bulk_g2s_stream(dst + boff, g.seg[sg].biases + (size_t)r * gs, sb, fb, stream);
              issued();
            }
          continue;
        }
        for (uint32_t pass = 0; pass < npass; ++pass) {
          const uint64_t pol = pass + 1 < npass ? keep : stream;
          for (uint32_t sg = 0; sg < nseg; ++sg) {
            const uint32_t base = g.row0[sg], lo = max(rb, base), hi = min(re, g.row0[sg + 1]);
            if (lo >= hi) continue;
            const uint32_t obase = (uint32_t)((g.out[sg] - g.out[0]) / out_esz(g));
            const uint8_t* codes = g.seg[sg].codes;
            const uint16_t* scales = g.seg[sg].scales;
            const uint16_t* biases = g.seg[sg].biases;
            for (uint32_t r = lo; r < hi; r += R) {
              const uint32_t nr = min(R, hi - r), local = r - base, cb = nr * K, sb = nr * gs * 2;
              uint8_t* dst = ring_claim(rg, sh, span, cb + 2 * sb, r | (nr << 24), obase + local, status);
              if (!dst) goto drain;
              uint64_t* fb = &sh.full[slot_of(rg.i)];
              bulk_g2s_stream(dst, codes + (size_t)local * K, cb, fb, pol);
              bulk_g2s_stream(dst + soff, scales + (size_t)local * gs, sb, fb, pol);
              bulk_g2s_stream(dst + boff, biases + (size_t)local * gs, sb, fb, pol);
              issued();
            }
          }
        }
      } else if (ty == kPhAttn) {
        const bool t8 = L.kv_dtype == kKvTurbo8;
        const uint32_t rowh = P.Hkv * P.D, rowbytes = rowh * (t8 ? 1 : 2);
        const uint32_t ss = turbo8_sstride(P.Hkv, P.D), srow = ss * 2;  // Turbo8 scales per token
        for (uint32_t b = 0; b < batch; ++b) {
          // paged: one pool, sequence b's table; the entry of the next block is loaded
          // while the current block's tiles are issued
          const bool paged = L.btab != nullptr;
          const int32_t* btab = paged ? L.btab + (size_t)(L.capacity >> L.bt_shift) * b : nullptr;
          const uint32_t bsh = L.bt_shift, bmask = (1u << bsh) - 1u;
          uint32_t lb_cur = ~0u, lb_nxt = ~0u;
          int32_t pb_cur = 0, pb_nxt = 0;
          const size_t seq_off = paged ? 0 : (size_t)L.capacity * rowbytes * b;
          const uint8_t* kc = L.kc + seq_off;
          const uint8_t* vc = L.vc + seq_off;
          const uint16_t* ks = t8 ? L.ks + (size_t)L.capacity * ss * b : nullptr;
          const uint16_t* vs = t8 ? L.vs + (size_t)L.capacity * ss * b : nullptr;
          const Span sp = attn_span(P, L.capacity, b, L.btab != nullptr);
          for (uint32_t t = 0; t < sp.ntiles; ++t) {
            const uint32_t tt = sp.t0 + t * kTS, n = min((uint32_t)kTS, sp.tc_end - tt);
            // rows past n are read (masked) by the consumers. A tile: K rows, then
            // (Turbo8) K scales, V rows, V scales, each part kTS tokens long.
            const uint32_t part = kTS * (rowbytes + (t8 ? srow : 0u));
            size_t row = tt;
            if (paged) {  // the tile lies in one block (splits and tiles start at multiples of 8)
              const uint32_t lb = tt >> bsh;
              if (lb != lb_cur) {
                pb_cur = lb == lb_nxt ? pb_nxt : __ldg(btab + lb);
                lb_cur = lb;
                lb_nxt = lb + 1;
                if ((lb_nxt << bsh) < sp.tc_end) pb_nxt = __ldg(btab + lb_nxt);
                else lb_nxt = ~0u;
              }
              row = ((size_t)(uint32_t)pb_cur << bsh) | (tt & bmask);
            }
            uint8_t* dst = ring_claim(rg, sh, 2 * part, 2 * n * (rowbytes + (t8 ? srow : 0u)), 0u, 0u, status);
            if (!dst) goto drain;
            uint64_t* fb = &sh.full[slot_of(rg.i)];
            bulk_g2s(dst, kc + row * rowbytes, n * rowbytes, fb);
            bulk_g2s(dst + part, vc + row * rowbytes, n * rowbytes, fb);
            if (t8) {
              bulk_g2s(dst + kTS * rowbytes, ks + (size_t)tt * ss, n * srow, fb);
              bulk_g2s(dst + part + kTS * rowbytes, vs + (size_t)tt * ss, n * srow, fb);
            }
            issued();
          }
        }
      } else if (ty == kPhGdn) {
        // the work item's state block, conv state and conv weights, one tile per sequence
        const GdnItem w = gdn_item(P);
        if (!w.ok) continue;
        const uint32_t Dk = P.Dk, Kc = P.Kc, nch = 2 * Dk + 32;
        const uint32_t ch[3] = {w.hk * Dk, P.Hk * Dk + w.hk * Dk, 2 * P.Hk * Dk + w.h * P.Dv + w.v0};
        const uint32_t nc[3] = {Dk, Dk, 32};
        const uint32_t bytes = gdn_tile_bytes(Dk, Kc);
        for (uint32_t b = 0; b < batch; ++b) {
          const float* ssm = L.ssm + (size_t)P.Hv * P.Dk * P.Dv * b;
          const float* conv = L.conv_state + (size_t)P.C * Kc * b;
          uint8_t* dst = ring_claim(rg, sh, bytes, bytes, 0u, 0u, status);
          if (!dst) goto drain;
          uint64_t* fb = &sh.full[slot_of(rg.i)];
          bulk_g2s(dst, ssm + (size_t)blockIdx.x * Dk * 32, Dk * 128, fb);
          uint32_t done = 0;
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            bulk_g2s(dst + Dk * 128 + done * Kc * 4, conv + (size_t)ch[j] * Kc, nc[j] * Kc * 4, fb);
            bulk_g2s(dst + Dk * 128 + nch * Kc * 4 + done * Kc * 2, L.conv_w + (size_t)ch[j] * Kc, nc[j] * Kc * 2, fb);
            done += nc[j];
          }
          issued();
        }
      }
    }
  }
drain:  // let the copies still in flight land before the CTA can exit
  for (uint32_t j = rg.tail; j < rg.i; ++j) mbar_wait(&sh.full[slot_of(j)], parity_of(j), drain_limit());
}

// ------------------------------------------------------------------ the helper warp

// The work between phases that no consumer should wait for, one phase ahead of the
// consumers: while they run phase ph, the descriptions of phase ph + 1 (the layer's
// and the GEMV's, formed on one thread, ~1 us), and in a linear-attention layer's
// gate|up phase the shift of the q/k channels' conv state (every linear-attention
// CTA has read it by then: the phase before waited for all their readouts). Its
// waits use at least the default limit, so that the consumers never run on
// descriptions it has not formed.
__device__ __noinline__ void helper_loop() {
  const Program& P = prog();
  const uint32_t lane = threadIdx.x & 31;
  const uint64_t limit = drain_limit();
  // until the consumers are in phase ph (so phase ph - 1's buffers are free and
  // phase ph's descriptions are in place); false when the wait runs out
  auto wait_entered = [&](uint32_t ph) {
    if (ld_volatile_shared(&s_ph.entered) > ph) return true;
    const uint64_t t0 = global_ns();
    while (ld_volatile_shared(&s_ph.entered) <= ph) {
      if (global_ns() - t0 > limit) {
        set_status(P.status, kStatusTimeout);
        return false;
      }
      __nanosleep(128);
    }
    return true;
  };
  uint32_t ph = 0;
  for (uint32_t l = 0; l < P.n_layers; ++l) {
    const uint32_t ph0 = ph;
    if (!wait_entered(ph0)) return;
    const int kind = s_lay0[l & 1].kind;  // formed before the consumers entered phase ph0
    const int np = n_phases(kind);
    for (int p = 0; p < np; ++p, ++ph) {
      if (p > 0 && !wait_entered(ph)) return;
      if (p + 1 < np) form_phase(l, p + 1, ph + 1, ph0);
      else if (l + 1 < P.n_layers) form_phase(l + 1, 0, ph + 1, ph + 1);
      if (kind == kLayerGDN && p == 3) {  // gate|up of a linear-attention layer
        const LayerDesc& L = s_lay0[l & 1];
        for (uint32_t b = 0; b < P.batch; ++b)
          conv_shift_qk(L.conv_state + (size_t)P.C * P.Kc * b, seq_scratch(P, b), phase_tag(ph0));
      }
      __syncwarp();
      if (lane == 0) st_volatile_shared(&s_ph.prepped, ph + 2);  // phases 0 .. ph + 1 formed
      __syncwarp();
    }
  }
}

// ------------------------------------------------------------------ the kernel

template <int D, int HPW, int DK, bool BATCHED>
__global__ void __launch_bounds__(kDecThreads, 1) decode_kernel(const __grid_constant__ Program Pk) {
  const Smem sh = smem_map(smem_raw, Pk.ring_bytes);
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the program's header into shared memory: 4-byte words (the parameter block is
  // 8-byte aligned); the phase loops then never read the large parameter block
  for (uint32_t i = threadIdx.x; i < kHeadBytes / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(s_head)[i] = reinterpret_cast<const uint32_t*>(&Pk)[i];
  const Program& P = prog();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kDecSlots; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], NCW);
    }
    mbar_fence_init();
    // the consumers/helper handshake starts before any phase: nothing entered, phase 0
    // to be formed by consumer warp 0
    s_ph.entered = 0u;
    s_ph.prepped = 1u;
    s_ph.layers = Pk.layers;
    s_dead_cta = 0u;
  }
  if (threadIdx.x < Pk.batch) s_pos[threadIdx.x] = Pk.d_pos ? Pk.d_pos[threadIdx.x] : 0;
  __syncthreads();

  if (warp == NCW) {
    // ------------------------------------------------ producer: the whole schedule
    if (lane == 0) produce_all(Pk.layers);
    return;
  }
  if (warp == NCW + 1) {
    // ------------------------------------------------ helper: descriptions, conv shift
    // (phase 0's descriptions are formed by consumer warp 0 before the first phase)
    if (P.n_layers > 0) helper_loop();
    return;
  }

  // -------------------------------------------------- consumers: the phases in order
  // Each phase runs for the batch's sequences back to back (they are independent).
  // No grid barrier: each phase waits inside for the tagged inputs it reads. Between
  // phases warp 0 fetches the coming phase's descriptions (the layer's, rebased to
  // the first sequence, and the GEMV's) once every warp is done with the last.
  uint32_t itd = 0, ph = 0;  // ring position | kDeadBit; the launch's phase index
  auto mark = [&](uint32_t k) {
    if (P.trace && threadIdx.x == 0 && ph < P.trace_phases)
      P.trace[((size_t)blockIdx.x * P.trace_phases + ph) * kTraceSlots + k] = global_ns();
  };
  auto slots = [&]() -> unsigned long long* {
    return P.trace && ph < P.trace_phases ? P.trace + ((size_t)blockIdx.x * P.trace_phases + ph) * kTraceSlots
                                          : nullptr;
  };
  // warp 0: the consumers' view of sequence b (a batch's phases other than the
  // projections run once per sequence): its scratch block and vectors, the layer's
  // caches rebased to it
  auto set_seq = [&](uint32_t b) {
    if (BATCHED) {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(&cur_layer0());
      uint32_t* dst = reinterpret_cast<uint32_t*>(&cur_layer());
      for (uint32_t i = lane; i < sizeof(LayerDesc) / 4; i += 32) dst[i] = src[i];
      __syncwarp();
      if (lane == 0 && b) seq_caches(P, cur_layer(), b);
    }
    if (lane == 0) {
      s_seq.scratch = seq_scratch(P, b);
      s_seq.x_in = P.x_in + (size_t)b * P.E;
      s_seq.x_out = P.x_out + (size_t)b * P.E;
      s_seq.b = b;
    }
    __syncwarp();
  };
  // warp 0 at a phase's entry: wait (bounded) until the helper has formed the
  // phase's descriptions, select their buffers, tell the helper. A wait that runs
  // out leaves the descriptions unusable: the CTA's consumers then touch no ring
  // tile for the rest of the launch (dead).
  auto enter = [&](uint32_t l, uint32_t ph_) {
    if (lane == 0) {
      bool ok = ld_volatile_shared(&s_ph.prepped) > ph_;
      if (!ok) {
        const uint64_t t0 = global_ns();
        while (!(ok = ld_volatile_shared(&s_ph.prepped) > ph_) && global_ns() - t0 <= drain_limit()) __nanosleep(64);
      }
      if (!ok) {
        set_status(P.status, kStatusTimeout);
        s_dead_cta = 1u;
      }
      s_sel = (ph_ & 1u) | ((l & 1u) << 1);
      st_volatile_shared(&s_ph.entered, ph_ + 1);
    }
    __syncwarp();
    set_seq(0);
  };
  if (warp == 0 && P.n_layers > 0) {
    form_phase(0, 0, 0, 0);
    enter(0, 0);
  }
  for (uint32_t l = 0; l < P.n_layers; ++l) {
    for (int p = 0;; ++p, ++ph) {
      if (l > 0 || p > 0) {
        mark(0);
        consumer_sync();  // every warp is done with the last phase
        mark(13);
        if (warp == 0) enter(l, ph);
        mark(14);
      }
      consumer_sync();
      if (s_dead_cta) itd |= kDeadBit;
      mark(1);
      const int kind = cur_layer0().kind;
      const int ty = phase_type(kind, p);
      if (BATCHED && ty == kPhGemv) {  // every sequence in passes over the weights, on tensor cores
        const uint32_t bs = cur_gemv().bs, npass = cur_gemv().npass;
        for (uint32_t pass = 0; pass < npass; ++pass) {
          const uint32_t b0 = pass * bs, nb = min(bs, P.batch - b0);
          if (pass > 0) consumer_sync();  // every team is done with the last pass's inputs
          gemv_prologue_b(b0, nb, pass == 0 ? slots() : nullptr);
          if (pass == 0) mark(3);
          itd = gemv_tiles_b(itd, b0, nb, pass == 0 ? slots() : nullptr);
          if (pass == 0) mark(12);
        }
      } else {
        const uint32_t nb = BATCHED ? P.batch : 1u;
        for (uint32_t b = 0; b < nb; ++b) {
          if (b > 0) {  // the next sequence: its descriptions, once every warp is done with the last
            consumer_sync();
            if (warp == 0) set_seq(b);
            consumer_sync();
          }
          if (ty == kPhGemv) {
            gemv_prologue(slots());
            mark(3);
            itd = gemv_rows(itd, slots());
          } else if (ty == kPhAttn) {
            itd = cur_layer().kv_dtype == kKvTurbo8 ? attn_consume<D, HPW, true>(itd, ph, slots())
                                                    : attn_consume<D, HPW, false>(itd, ph, slots());
          } else if (ty == kPhGdn) {
            itd = gdn_consume<DK>(itd, ph);
          } else {
            combine_consume(ph);
          }
        }
      }
      mark(2);
      if (p + 1 >= n_phases(kind)) {
        ++ph;
        break;
      }
    }
  }
  consumer_sync();
  if (P.advance && blockIdx.x == 0 && threadIdx.x < P.batch) P.advance[threadIdx.x] += 1;
  if (P.wait_probe && threadIdx.x == 0) {  // debug: a bounded wait on a word nothing may set,
    const uint64_t t0 = global_ns();      // after the forward's work (nothing waits on it)
    while (ld_acquire(P.wait_probe) == 0u) {
      if (global_ns() - t0 > P.wait_ns) {
        set_status(P.status, kStatusTimeout);
        break;
      }
      __nanosleep(256);
    }
  }
}


template <int D, int HPW, bool BT>
DecodeKernel pick_dk(uint32_t Dk) {
  switch (Dk) {
    case 32: return decode_kernel<D, HPW, 32, BT>;
    case 64: return decode_kernel<D, HPW, 64, BT>;
    case 128: return decode_kernel<D, HPW, 128, BT>;
  }
  return nullptr;
}
template <int D>
DecodeKernel pick_h(uint32_t hpw, uint32_t Dk, bool batched) {
  switch (hpw) {
    case 1: return batched ? pick_dk<D, 1, true>(Dk) : pick_dk<D, 1, false>(Dk);
    case 2: return batched ? pick_dk<D, 2, true>(Dk) : pick_dk<D, 2, false>(Dk);
  }
  return nullptr;
}

// q-heads per attention warp: 2 when they pair up within a kv-head's group, else
// 1, with no more head groups (H / HPW) than consumer warps; the remaining warps
// split the tokens (TI = 12 / (H / HPW) warps per head group). (Four heads per
// warp measured slower at head dim 256: register pressure.)
uint32_t attn_hpw(uint32_t H, uint32_t Hkv) {
  if (Hkv == 0 || H % Hkv) return 0;
  const uint32_t grp = H / Hkv;
  for (uint32_t hpw : {2u, 1u})
    if (grp % hpw == 0 && H / hpw <= (uint32_t)NCW) return hpw;
  return 0;
}

}  // namespace

// The kernel for head dim D, by q-heads per warp, GDN key head dim and batching
// (each D is instantiated in a translation unit of its own).
template <int D>
DecodeKernel decode_kernel_for(uint32_t hpw, uint32_t Dk, bool batched) {
  return pick_h<D>(hpw, Dk, batched);
}

}  // namespace q35
