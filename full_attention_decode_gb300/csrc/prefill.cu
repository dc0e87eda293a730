// Multi-token prefill kernels (prefill.h). The prompt's tokens are the columns of
// every projection, so the projections are dense contractions and run on the
// fifth-generation tensor cores: tcgen05.mma with bf16 operands in shared memory
// and fp32 accumulators in tensor memory. The int8 group-64 weights are
// dequantised by the CTA's threads on their way into shared memory (as bf16, or
// as the sum of two bf16 values, exact to 2^-16). The attention and the Gated
// DeltaNet recurrence keep the single-token forward's arithmetic, token after
// token where the method is sequential.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "prefill.h"

#include <algorithm>
#include <type_traits>

#include <cuda_fp16.h>

namespace q35pf {
using namespace q35;
namespace {

// ------------------------------------------------------------------ tcgen05

// A GEMM tile: 128 weight rows (the MMA's M) x 256 tokens (its N), K in blocks of
// one quantisation group (64). Each operand tile of a K-block (128 weight rows or
// 256 token rows of 64 bf16) is in the K-major layout with the 128-byte swizzle:
// row r at r * 128, its 16-byte chunk j at chunk position j ^ (r % 8) (the tile
// 1024-byte aligned), so eight consecutive rows' copies of one chunk fall in
// different banks; 8-row groups are 1024 bytes apart (the descriptor's stride
// offset). In the exact form the weights enter the MMA as the bf16 sum hi + lo
// (hi = bf16(w), lo = bf16(w - hi), so hi + lo is w to 2^-16 relative): both
// weight tiles multiply the same token tile into one accumulator. The plain form
// takes hi alone.
// Shared memory: a ring of kRaw K-blocks as loaded by the tensor-memory-access
// engine (the token tile and the raw codes, 128 rows of 64 bytes, both swizzled by
// the copy itself), filled kAhead blocks ahead, and the stages of dequantised
// weight tiles written by the CTA's threads.
constexpr uint32_t kBM = 128, kBN = 256, kDqThreads = 256, kGemmThreads = kDqThreads + 64;
constexpr uint32_t kRaw = 4, kAhead = kRaw - 2;
constexpr uint32_t kTileBytes = kBM * 64 * 2;  // a weight tile (hi or lo)
constexpr uint32_t kXBytes = kBN * 64 * 2;     // a token tile
constexpr uint32_t kCodeBytes = kBM * 64;
constexpr uint32_t kRawBytes = kXBytes + kCodeBytes;
// weight stages: two of hi + lo (exact form) or four of hi (plain form), 64 KiB
template <bool EXACT>
struct WStages {
  static constexpr uint32_t n = EXACT ? 2 : 4, bytes = EXACT ? 2 * kTileBytes : kTileBytes;
};
constexpr uint32_t kGemmSmem = kRaw * kRawBytes + 4 * kTileBytes + 1024;  // + alignment slack

__device__ __forceinline__ uint32_t sw_off(uint32_t r, uint32_t j) { return r * 128 + ((j ^ (r & 7)) << 4); }

// Shared-memory matrix descriptor (K-major, 128-byte swizzle): start address / 16
// (bits 0-13), leading offset field 1 (unused by this layout), stride offset
// 1024 / 16 (bits 32-45), the fixed version 1 (46-47), base offset 0 (the
// tiles are 1024-byte aligned), layout 2 = 128-byte swizzle (bits 61-63). The
// K = 16 slices of a tile start 32 bytes apart: the swizzle is applied to the
// address bits, so a slice's start needs no other change.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024u >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A and B
// (7-9 = 1, 10-12 = 1), both K-major (15, 16 = 0), N / 8 at bits 17-22, M / 16 at
// bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((kBN >> 3) << 17) | ((kBM >> 4) << 24);

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy stores to shared memory made visible to the tensor core's reads.
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate)
      : "memory");
}
// Arrive once on bar when every MMA this thread issued before is complete.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}
// 16 consecutive fp32 columns of the warp's 32 lanes (lane i of the warp: TMEM lane
// base + i), waited for before they are returned.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])::"memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit) return false;
  return true;
}

// Eight codes (bytes of c0, c1) dequantised as w = fmaf(s, code, b) (exact for the
// format's bias -128 s) and split into bf16 pairs hi = bf16(w), lo = bf16(w - hi)
// (lo only when EXACT).
template <bool EXACT>
__device__ __forceinline__ void dequant8(uint32_t c0, uint32_t c1, float s, float b, uint4& hi, uint4& lo) {
  float f[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // byte i of the word as the low byte of 2^23: its value exactly, then minus 2^23
    f[i] = __uint_as_float(__byte_perm(c0, 0x4B000000u, 0x7440u + i)) - 8388608.0f;
    f[4 + i] = __uint_as_float(__byte_perm(c1, 0x4B000000u, 0x7440u + i)) - 8388608.0f;
  }
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float w0 = fmaf(s, f[2 * i], b), w1 = fmaf(s, f[2 * i + 1], b);
    const __nv_bfloat162 ph = __floats2bfloat162_rn(w0, w1);
    h[i] = *reinterpret_cast<const uint32_t*>(&ph);
    if (EXACT) {
      const float2 hf = __bfloat1622float2(ph);
      const __nv_bfloat162 pl = __floats2bfloat162_rn(w0 - hf.x, w1 - hf.y);
      l[i] = *reinterpret_cast<const uint32_t*>(&pl);
    } else {
      l[i] = 0u;
    }
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// The GEMM's operands as tensor maps (tokens: bf16 [T][ldx], boxes of 64 x 256
// with the 128-byte swizzle; codes: u8 [N][K], boxes of 64 x 128 with the 64-byte
// swizzle), zero-filled outside the matrices.
struct GemmArgs {
  CUtensorMap tx;
  CUtensorMap tc;
  Gemm g;
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// One CTA: rows [n0, n0 + 128) x tokens [t0, t0 + 256), ten warps. Warps 0-7
// dequantise: thread (r, half) turns half of weight row n0 + r's codes of each
// K-block into the block's weight stage and arrives on the stage's barrier. Lane 0
// of warp 8 copies each K-block's token tile and codes kAhead blocks ahead (one
// barrier per raw slot, completed by the copies' byte count); lane 0 of warp 9,
// once a block's copies have landed and its weight stage is complete, issues its
// K=16 MMAs (hi, and lo in the exact form) and commits them to the raw slot's
// second barrier, whose arrival frees the raw slot (refilled kAhead blocks later)
// and the weight stage (rewritten WStages::n blocks later). No barrier of the whole
// CTA inside the loop: the dequantising warps run ahead of the MMAs as far as the
// stages allow.
template <bool EXACT>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmArgs A) {
  using WS = WStages<EXACT>;
  const Gemm& g = A.g;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ uint64_t full[kRaw], done[kRaw], wready[4];
  __shared__ uint32_t s_tmem;
  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t n0 = blockIdx.x * kBM, t0 = blockIdx.y * kBN;
  if (tid == 0) {
    for (uint32_t s = 0; s < kRaw; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&done[s], 1);
    }
    for (uint32_t s = 0; s < 4; ++s) mbar_init(&wready[s], kDqThreads);
    mbar_fence_init();
  }
  if (warp == 9) {
    tmem_alloc(&s_tmem, kBN);
    tmem_relinquish();
  }
  tc_before_sync();
  __syncthreads();
  tc_after_sync();
  const uint32_t tmem = s_tmem;
  // this CTA's K-blocks (split K: the z-th of gridDim.z equal ranges); kb below counts
  // from the range's start
  const uint32_t nkt = g.K / 64, kb0 = blockIdx.z * nkt / gridDim.z;
  const uint32_t nk = (blockIdx.z + 1) * nkt / gridDim.z - kb0;
  // the tiles from the first 1024-byte boundary of the dynamic shared memory
  const uint32_t sraw = smem_addr(smem), sbase = (sraw + 1023u) & ~1023u;
  uint8_t* raw = smem + (sbase - sraw);
  uint8_t* wst = raw + kRaw * kRawBytes;
  bool ok = true;
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (ok && !mbar_wait_bounded(bar, parity, g.wait_ns)) {
      set_status(g.status, kStatusTimeout);
      ok = false;
    }
  };
  if (warp == 8) {
    if (lane == 0) {  // the copies
      auto issue = [&](uint32_t kb) {  // K-block kb into its raw slot
        uint8_t* X = raw + (kb % kRaw) * kRawBytes;
        uint64_t* bar = &full[kb % kRaw];
        mbar_arrive_expect_tx(bar, kXBytes + kCodeBytes);
        tma_load_2d(X, &A.tx, (int32_t)((kb0 + kb) * 64), (int32_t)t0, bar);
        tma_load_2d(X + kXBytes, &A.tc, (int32_t)((kb0 + kb) * 64), (int32_t)n0, bar);
      };
      for (uint32_t kb = 0; kb < kAhead && kb < nk; ++kb) issue(kb);
      for (uint32_t kb = 0; kb + kAhead < nk; ++kb) {  // the slot's last reader was MMA(kb + kAhead - kRaw)
        if (kb + kAhead >= kRaw) wait(&done[(kb + kAhead) % kRaw], ((kb + kAhead - kRaw) / kRaw) & 1);
        issue(kb + kAhead);
      }
    }
  } else if (warp == 9) {
    if (lane == 0) {  // the MMAs
      for (uint32_t kb = 0; kb < nk; ++kb) {
        wait(&full[kb % kRaw], (kb / kRaw) & 1);
        wait(&wready[kb % WS::n], (kb / WS::n) & 1);
        tc_after_sync();
        const uint32_t sx = sbase + (kb % kRaw) * kRawBytes;
        const uint32_t sh = sbase + kRaw * kRawBytes + (kb % WS::n) * WS::bytes, sl = sh + kTileBytes;
#pragma unroll
        for (uint32_t kk = 0; kk < 4; ++kk) {  // K = 16 per MMA: 32 bytes of each row
          mma_bf16(tmem, smem_desc(sh + kk * 32), smem_desc(sx + kk * 32), (kb | kk) != 0);
          if (EXACT) mma_bf16(tmem, smem_desc(sl + kk * 32), smem_desc(sx + kk * 32), 1u);
        }
        mma_commit(&done[kb % kRaw]);
      }
    }
  } else {
    const uint32_t r = tid & 127, half = tid >> 7;
    const uint32_t n = n0 + r;
    const bool nin = n < g.N;
    const uint16_t* srow = g.scales + (size_t)(nin ? n : 0) * g.gstride + kb0;
    const uint16_t* brow = g.biases + (size_t)(nin ? n : 0) * g.gstride + kb0;
    const uint32_t j0 = 4 * half;
    // scale and bias of the row, two blocks ahead in registers
    uint16_t sc0 = 0, bi0 = 0, sc1 = 0, bi1 = 0;
    if (nin) {
      sc0 = __ldg(srow);
      bi0 = __ldg(brow);
      if (nk > 1) {
        sc1 = __ldg(srow + 1);
        bi1 = __ldg(brow + 1);
      }
    }
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    for (uint32_t kb = 0; kb < nk; ++kb) {
      const float fs = bf16f(sc0), fb = bf16f(bi0);
      sc0 = sc1;
      bi0 = bi1;
      if (nin && kb + 2 < nk) {
        sc1 = __ldg(srow + kb + 2);
        bi1 = __ldg(brow + kb + 2);
      }
      // the weight stage's last reader was MMA(kb - WS::n)
      if (kb >= WS::n) wait(&done[(kb - WS::n) % kRaw], ((kb - WS::n) / kRaw) & 1);
      wait(&full[kb % kRaw], (kb / kRaw) & 1);
      // the codes tile arrives with the 64-byte swizzle: 16-byte chunk c of row r at
      // chunk position c ^ ((r / 2) % 4), so a warp's 32 rows read one chunk each
      // without bank conflicts
      const uint8_t* Cs = raw + (kb % kRaw) * kRawBytes + kXBytes + r * 64;
      const uint32_t sw = (r >> 1) & 3;
      uint8_t* Wh = wst + (kb % WS::n) * WS::bytes;
      uint8_t* Wl = Wh + kTileBytes;
      {
        const uint4 a0 = *reinterpret_cast<const uint4*>(Cs + (((2 * half) ^ sw) << 4));
        const uint4 a1 = *reinterpret_cast<const uint4*>(Cs + (((2 * half + 1) ^ sw) << 4));
        uint4 h[4], l[4];
        dequant8<EXACT>(a0.x, a0.y, fs, fb, h[0], l[0]);
        dequant8<EXACT>(a0.z, a0.w, fs, fb, h[1], l[1]);
        dequant8<EXACT>(a1.x, a1.y, fs, fb, h[2], l[2]);
        dequant8<EXACT>(a1.z, a1.w, fs, fb, h[3], l[3]);
#pragma unroll
        for (uint32_t i = 0; i < 4; ++i) {
          *reinterpret_cast<uint4*>(Wh + sw_off(r, j0 + i)) = nin ? h[i] : zero;
          if (EXACT) *reinterpret_cast<uint4*>(Wl + sw_off(r, j0 + i)) = nin ? l[i] : zero;
        }
      }
      fence_async_shared();  // the weight stores, for the tensor core
      mbar_arrive(&wready[kb % WS::n]);
    }
  }
  // every MMA is done when the last commit has arrived; warps 0-7 read TMEM lanes
  // 32 (w % 4) .. (their weight rows) over tokens [128 (w / 4), +128)
  const uint32_t last = nk - 1;
  if (warp < 8) {
    wait(&done[last % kRaw], (last / kRaw) & 1);
    tc_after_sync();
  }
  const uint32_t q = warp & 3, ch = warp >> 2;
  const uint32_t row = n0 + 32 * q + lane;
#pragma unroll 1
  for (uint32_t c = 0; warp < 8 && c < kBN / 2; c += 16) {
    float v[16];
    tmem_ld16(tmem + ((32 * q) << 16) + (kBN / 2) * ch + c, v);
    if (ok && row < g.N) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t tt = t0 + (kBN / 2) * ch + c + i;
        if (tt < g.T) {
          if (gridDim.z > 1) {  // a split's partial sum, added up by the finishing kernel
            g.ws[((size_t)blockIdx.z * g.T + tt) * g.N + row] = v[i];
          } else {
            float y = v[i];
            if (g.R) y += bf16f(g.R[(size_t)tt * g.ldy + row]);
            g.Y[(size_t)tt * g.ldy + row] = to_bf16(y);
          }
        }
      }
    }
  }
  tc_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc_after_sync();
    tmem_dealloc(tmem, kBN);
  }
}

// The split-K sum: Y[t][n] = bf16(sum_z ws[z][t][n] (+ R[t][n])), splits added in
// order.
__global__ void gemm_finish_kernel(const Gemm g, uint32_t splits) {
  const size_t total = (size_t)g.T * g.N;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const size_t t = i / g.N, n = i % g.N;
    float y = 0.f;
    for (uint32_t z = 0; z < splits; ++z) y += g.ws[z * total + i];
    if (g.R) y += bf16f(g.R[t * g.ldy + n]);
    g.Y[t * g.ldy + n] = to_bf16(y);
  }
}

// ------------------------------------------------------------------ norms

// Eight bf16 values of a 16-byte word as floats, and back (round to nearest even).
__device__ __forceinline__ void unpack8(const uint4 u, float* x) {
  x[0] = bf16lo(u.x); x[1] = bf16hi(u.x); x[2] = bf16lo(u.y); x[3] = bf16hi(u.y);
  x[4] = bf16lo(u.z); x[5] = bf16hi(u.z); x[6] = bf16lo(u.w); x[7] = bf16hi(u.w);
}
__device__ __forceinline__ uint4 pack8(const float* x) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = (uint32_t)to_bf16(x[2 * i]) | ((uint32_t)to_bf16(x[2 * i + 1]) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const uint32_t warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();  // red is free (an earlier reduction has been read)
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (uint32_t w = 0; w < nw; ++w) t += red[w];
  return t;
}

// One block per token; 8 values per thread and pass.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t* a, const uint16_t* b, uint16_t* resid,
                                                      const uint16_t* w, uint16_t* out, uint32_t E, float eps) {
  __shared__ float red[8];
  const size_t base = (size_t)blockIdx.x * E;
  float ss = 0.f;
  for (uint32_t i = 8 * threadIdx.x; i < E; i += 8 * blockDim.x) {
    const uint4 ua = *reinterpret_cast<const uint4*>(a + base + i);
    float x[8];
    unpack8(ua, x);
    if (b) {
      float y[8];
      unpack8(*reinterpret_cast<const uint4*>(b + base + i), y);
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = round_bf16(x[j] + y[j]);
      if (resid) *reinterpret_cast<uint4*>(resid + base + i) = pack8(x);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = fmaf(x[j], x[j], ss);
  }
  const float inv = rsqrtf(block_sum(ss, red) / (float)E + eps);
  for (uint32_t i = 8 * threadIdx.x; i < E; i += 8 * blockDim.x) {
    float x[8], wv[8];
    if (b && resid) {
      unpack8(*reinterpret_cast<const uint4*>(resid + base + i), x);
    } else {
      unpack8(*reinterpret_cast<const uint4*>(a + base + i), x);
      if (b) {
        float y[8];
        unpack8(*reinterpret_cast<const uint4*>(b + base + i), y);
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = round_bf16(x[j] + y[j]);
      }
    }
    unpack8(*reinterpret_cast<const uint4*>(w + i), wv);
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = x[j] * inv * wv[j];
    *reinterpret_cast<uint4*>(out + base + i) = pack8(x);
  }
}

__global__ void silu_mul_kernel(const uint16_t* g, const uint16_t* u, uint16_t* h, size_t n8) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    float x[8], y[8];
    unpack8(reinterpret_cast<const uint4*>(g)[i], x);
    unpack8(reinterpret_cast<const uint4*>(u)[i], y);
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = siluf_(x[j]) * y[j];
    reinterpret_cast<uint4*>(h)[i] = pack8(x);
  }
}

// ------------------------------------------------------------------ full attention

// Turbo8 (WHT-rotated FP8 E4M3 codes, a bf16 scale per 16 elements). A warp holds
// a head's D-vector with lane L holding elements [L EPL, L EPL + EPL), EPL = D / 32.
// The orthonormal Walsh-Hadamard transform in Sylvester order: butterflies over the
// element index's low bits inside the lane, then over the lane bits by shuffles,
// scaled by 1 / sqrt(D).
template <int EPL>
__device__ __forceinline__ void wht_lanes(float* x, uint32_t lane, float norm) {
#pragma unroll
  for (int hb = 1; hb < EPL; hb <<= 1)
#pragma unroll
    for (int e = 0; e < EPL; ++e)
      if (!(e & hb)) {
        const float u = x[e], w = x[e + hb];
        x[e] = u + w;
        x[e + hb] = u - w;
      }
#pragma unroll
  for (uint32_t m = 1; m < 32; m <<= 1)
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, x[e], m);
      x[e] = (lane & m) ? o - x[e] : x[e] + o;
    }
#pragma unroll
  for (int e = 0; e < EPL; ++e) x[e] *= norm;
}
__device__ __forceinline__ uint32_t e4m3_pair(float x0, float x1) {  // x0 in the low byte
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x1), "f"(x0));
  return r;
}
__device__ __forceinline__ float2 e4m3_pair_value(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}
// Quantise the warp's row (bf16 values in x): per group of 16 elements (16 / EPL
// lanes) scale = bf16(amax / 448), code = E4M3(x / scale) rounded to nearest even
// and saturated; a zero group keeps scale 0 and codes 0. Stores the lane's EPL
// codes at codes[L EPL ..] and each group's scale at scales[group].
template <int EPL>
__device__ __forceinline__ void turbo8_store(const float* x, uint32_t lane, uint8_t* codes, uint16_t* scales) {
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int o = 1; o < 16 / EPL; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = round_bf16(amax / 448.f);
#pragma unroll
  for (int e = 0; e < EPL; e += 2)
    *reinterpret_cast<uint16_t*>(codes + lane * EPL + e) =
        (uint16_t)(sc > 0.f ? e4m3_pair(x[e] / sc, x[e + 1] / sc) : 0u);
  if ((lane * EPL) % 16 == 0) scales[lane * EPL / 16] = to_bf16(sc);
}

// The cache row (in units of token rows) of logical token t: itself, or its row in
// the pool block the table names.
__device__ __forceinline__ size_t cache_row(const Attn& a, uint32_t t) {
  if (!a.btab) return t;
  const uint32_t m = (1u << a.bt_shift) - 1u;
  return ((size_t)(uint32_t)a.btab[t >> a.bt_shift] << a.bt_shift) | (t & m);
}

// Per (token, head slot) one warp: slots [0, H) are the q-heads (RMSNorm with
// q_norm, RoPE, into qr), [H, H + Hkv) the k-heads (RMSNorm with k_norm, RoPE,
// appended to the K cache), [H + Hkv, H + 2 Hkv) the v-heads (appended to the V
// cache). Each value is rounded to bf16 after the norm and after the rotation. For
// a Turbo8 cache the rows are then rotated by the WHT and rounded to bf16 again:
// q kept so in qr, k and v quantised into the cache's codes and scales.
template <int EPL>
__global__ void __launch_bounds__(128) qk_rope_kernel(const Attn a) {
  constexpr int D = 32 * EPL;
  __shared__ float buf[4][2][D];
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t slots = a.H + 2 * a.Hkv;
  const uint32_t item = blockIdx.x * 4 + warp;
  if (item >= a.T * slots) return;
  const uint32_t t = item / slots, sl = item % slots, pos = a.p0 + t;
  const size_t crow = cache_row(a, pos);
  const size_t kvrow = crow * a.Hkv * D;
  float* x = buf[warp][0];
  float* y = buf[warp][1];
  const bool isv = sl >= a.H + a.Hkv, isq = sl < a.H;
  const uint32_t hd = isq ? sl : isv ? sl - a.H - a.Hkv : sl - a.H;
  if (isv) {  // v: as projected
    const uint16_t* src = a.v + ((size_t)t * a.Hkv + hd) * D;
    for (uint32_t d = lane; d < D; d += 32) y[d] = bf16f(src[d]);
  } else {
    const uint16_t* src = isq ? a.qf + ((size_t)t * a.H + hd) * 2 * D : a.k + ((size_t)t * a.Hkv + hd) * D;
    const uint16_t* nw = isq ? a.q_norm : a.k_norm;
    float ss = 0.f;
    for (uint32_t d = lane; d < D; d += 32) {
      const float v = bf16f(src[d]);
      x[d] = v;
      ss = fmaf(v, v, ss);
    }
    const float inv = rsqrtf(warp_sum(ss) / (float)D + a.eps);
    for (uint32_t d = lane; d < D; d += 32) x[d] = round_bf16(x[d] * inv * bf16f(nw[d]));
    __syncwarp();
    const uint32_t half = a.R / 2;
    for (uint32_t d = lane; d < D; d += 32) {
      float v = x[d];
      if (d < a.R) {
        const uint32_t i = d < half ? d : d - half;
        float sn, cs;
        sincosf((float)pos * a.inv_freq[i], &sn, &cs);
        v = d < half ? x[d] * cs - x[d + half] * sn : x[d] * cs + x[d - half] * sn;
      }
      y[d] = round_bf16(v);
    }
  }
  __syncwarp();
  if (!a.turbo8) {
    uint16_t* dst = isq ? a.qr + ((size_t)t * a.H + hd) * D : (isv ? a.vc : a.kc) + kvrow + hd * D;
    for (uint32_t d = lane; d < D; d += 32) dst[d] = to_bf16(y[d]);
    return;
  }
  float r[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) r[e] = y[lane * EPL + e];
  wht_lanes<EPL>(r, lane, rsqrtf((float)D));
#pragma unroll
  for (int e = 0; e < EPL; ++e) r[e] = round_bf16(r[e]);
  if (isq) {
    uint16_t* dst = a.qr + ((size_t)t * a.H + hd) * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) dst[e] = to_bf16(r[e]);
    return;
  }
  uint8_t* codes = reinterpret_cast<uint8_t*>(isv ? a.vc : a.kc) + kvrow + hd * D;
  uint16_t* scales = (isv ? a.vs : a.ks) + crow * a.sstride + hd * (D / 16);
  turbo8_store<EPL>(r, lane, codes, scales);
}

// Causal attention: one CTA per (kv-head g, 8 consecutive tokens), warp w for token
// t = 8 * blockIdx.x + w and the HPG q-heads of group g. Key tiles of 32 rows of K
// and V (rows [0, p0 + t] for token t) are staged in shared memory, K rows padded
// by 16 bytes. Scores: lane j takes key j of the tile over all D dims; the online
// softmax runs in the log2 domain; P V: lane L holds dims [DPL L, DPL L + DPL).
// A Turbo8 cache: the tiles are decoded (E4M3 code times its group's scale, exact
// in fp32) into fp32 tiles (K rows padded by 4 elements), q is the rotated q, and the
// output is rotated back by the WHT before the gate (each step rounded to bf16).
template <int D, int HPG, bool T8>
__global__ void __launch_bounds__(256) attn_kernel(const Attn a) {
  constexpr int KT = 32, KS = T8 ? D + 4 : D + 8, DPL = D / 32;
  using TE = typename std::conditional<T8, float, uint16_t>::type;  // tile element
  extern __shared__ __align__(16) uint8_t dsm[];
  TE* Ks = reinterpret_cast<TE*>(dsm);  // [KT][KS]
  TE* Vs = Ks + KT * KS;                // [KT][D]
  uint16_t (*Qs)[HPG][D] = reinterpret_cast<uint16_t (*)[HPG][D]>(Vs + KT * D);  // [8][HPG][D]
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t g = blockIdx.y, tb = blockIdx.x * 8;
  const uint32_t t = tb + warp;
  const bool live = t < a.T;
  const uint32_t tmax = min(a.T - 1, tb + 7);
  const uint32_t nkeys = a.p0 + tmax + 1;  // keys the CTA's last token sees
  const uint32_t mykeys = live ? a.p0 + t + 1 : 0;
  const uint32_t kvw = a.Hkv * D;          // elements per cache row
  // this warp's q rows into shared memory
  if (live)
    for (uint32_t i = lane; i < HPG * D / 8; i += 32) {
      const uint32_t h = i / (D / 8), d8 = i % (D / 8);
      *reinterpret_cast<uint4*>(&Qs[warp][h][8 * d8]) =
          *reinterpret_cast<const uint4*>(a.qr + ((size_t)t * a.H + g * HPG + h) * D + 8 * d8);
    }
  const float sl2 = 1.4426950408889634f / sqrtf((float)D);  // log2(e) / sqrt(D)
  float m[HPG], l[HPG], o[HPG][DPL];
#pragma unroll
  for (int h = 0; h < HPG; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[h][i] = 0.f;
  }
  for (uint32_t k0 = 0; k0 < nkeys; k0 += KT) {
    __syncthreads();  // the last tile is consumed
    for (uint32_t i = threadIdx.x; i < KT * D / 8; i += blockDim.x) {
      const uint32_t j = i / (D / 8), d8 = i % (D / 8);
      if constexpr (T8) {
        float kx[8], vx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) kx[e] = vx[e] = 0.f;
        if (k0 + j < nkeys) {
          const size_t row = cache_row(a, k0 + j);
          const size_t off = row * kvw + g * D + 8 * d8;
          const uint2 kc = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(a.kc) + off);
          const uint2 vc = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(a.vc) + off);
          const size_t sidx = row * a.sstride + g * (D / 16) + d8 / 2;
          const float ksc = bf16f(a.ks[sidx]), vsc = bf16f(a.vs[sidx]);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const uint32_t kw = e < 4 ? kc.x : kc.y, vw = e < 4 ? vc.x : vc.y;
            const float2 kf = e4m3_pair_value(kw >> (8 * (e % 4))), vf = e4m3_pair_value(vw >> (8 * (e % 4)));
            kx[e] = kf.x * ksc;
            kx[e + 1] = kf.y * ksc;
            vx[e] = vf.x * vsc;
            vx[e + 1] = vf.y * vsc;
          }
        }
        *reinterpret_cast<float4*>(&Ks[j * KS + 8 * d8]) = make_float4(kx[0], kx[1], kx[2], kx[3]);
        *reinterpret_cast<float4*>(&Ks[j * KS + 8 * d8 + 4]) = make_float4(kx[4], kx[5], kx[6], kx[7]);
        *reinterpret_cast<float4*>(&Vs[j * D + 8 * d8]) = make_float4(vx[0], vx[1], vx[2], vx[3]);
        *reinterpret_cast<float4*>(&Vs[j * D + 8 * d8 + 4]) = make_float4(vx[4], vx[5], vx[6], vx[7]);
      } else {
        uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
        if (k0 + j < nkeys) {
          const size_t off = cache_row(a, k0 + j) * kvw + g * D + 8 * d8;
          kv = *reinterpret_cast<const uint4*>(a.kc + off);
          vv = *reinterpret_cast<const uint4*>(a.vc + off);
        }
        *reinterpret_cast<uint4*>(&Ks[j * KS + 8 * d8]) = kv;
        *reinterpret_cast<uint4*>(&Vs[j * D + 8 * d8]) = vv;
      }
    }
    __syncthreads();
    if (k0 >= mykeys) continue;  // (warp-uniform) past this token's keys
    // scores of key k0 + lane for the HPG heads
    float s[HPG];
#pragma unroll
    for (int h = 0; h < HPG; ++h) s[h] = 0.f;
#pragma unroll 4
    for (uint32_t d8 = 0; d8 < D / 8; ++d8) {
      float kx[8];
      if constexpr (T8) {
        const float4 k0v = *reinterpret_cast<const float4*>(&Ks[lane * KS + 8 * d8]);
        const float4 k1v = *reinterpret_cast<const float4*>(&Ks[lane * KS + 8 * d8 + 4]);
        kx[0] = k0v.x; kx[1] = k0v.y; kx[2] = k0v.z; kx[3] = k0v.w;
        kx[4] = k1v.x; kx[5] = k1v.y; kx[6] = k1v.z; kx[7] = k1v.w;
      } else {
        unpack8(*reinterpret_cast<const uint4*>(&Ks[lane * KS + 8 * d8]), kx);
      }
#pragma unroll
      for (int h = 0; h < HPG; ++h) {
        float qx[8];
        unpack8(*reinterpret_cast<const uint4*>(&Qs[warp][h][8 * d8]), qx);
#pragma unroll
        for (int e = 0; e < 8; ++e) s[h] = fmaf(qx[e], kx[e], s[h]);
      }
    }
    const bool kin = k0 + lane < mykeys;
    float p[HPG];
#pragma unroll
    for (int h = 0; h < HPG; ++h) {
      const float x = kin ? s[h] * sl2 : -INFINITY;
      const float mn = fmaxf(m[h], warp_max(x));
      const float corr = exp2f(m[h] - mn);  // 0 on the first tile (m = -inf)
      p[h] = kin ? exp2f(x - mn) : 0.f;
      l[h] = l[h] * corr + warp_sum(p[h]);
      m[h] = mn;
#pragma unroll
      for (int i = 0; i < DPL; ++i) o[h][i] *= corr;
    }
    const uint32_t jn = min((uint32_t)KT, mykeys - k0);
    for (uint32_t j = 0; j < jn; ++j) {
      float vx[DPL];
      if constexpr (T8) {
#pragma unroll
        for (int i = 0; i < DPL; ++i) vx[i] = Vs[j * D + DPL * lane + i];
      } else if constexpr (DPL == 8) {
        unpack8(*reinterpret_cast<const uint4*>(&Vs[j * D + 8 * lane]), vx);
      } else if constexpr (DPL == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(&Vs[j * D + 4 * lane]);
        vx[0] = bf16lo(u.x); vx[1] = bf16hi(u.x); vx[2] = bf16lo(u.y); vx[3] = bf16hi(u.y);
      } else {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(&Vs[j * D + 2 * lane]);
        vx[0] = bf16lo(u); vx[1] = bf16hi(u);
      }
#pragma unroll
      for (int h = 0; h < HPG; ++h) {
        const float pj = __shfl_sync(0xffffffffu, p[h], j);
#pragma unroll
        for (int i = 0; i < DPL; ++i) o[h][i] = fmaf(pj, vx[i], o[h][i]);
      }
    }
  }
  if (!live) return;
  // attn = bf16(o / l) (Turbo8: rotated back, bf16 again); gated = bf16(attn * sigmoid(gate))
#pragma unroll
  for (int h = 0; h < HPG; ++h) {
    const uint32_t hh = g * HPG + h;
    const float inv = 1.0f / l[h];
    const uint16_t* gate = a.qf + ((size_t)t * a.H + hh) * 2 * D + D;
    uint16_t* out = a.ga + ((size_t)t * a.H + hh) * D;
    float at[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) at[i] = round_bf16(o[h][i] * inv);
    if constexpr (T8) {
      wht_lanes<DPL>(at, lane, rsqrtf((float)D));
#pragma unroll
      for (int i = 0; i < DPL; ++i) at[i] = round_bf16(at[i]);
    }
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
      const uint32_t d = DPL * lane + i;
      out[d] = to_bf16(at[i] * sigmoidf_(bf16f(gate[d])));
    }
  }
}

// ------------------------------------------------------------------ Gated DeltaNet

// Per (token, channel): the causal conv's output for token t reads the inputs of
// tokens t - Kc + 1 .. t, those before the prompt from the state (slot Kc - 1 is the
// newest), then SiLU into act (fp32). No output depends on another, so every
// (token, channel) is its own thread; the state is advanced afterwards.
__global__ void conv_kernel(const Gdn g, float* act) {
  const size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (idx >= (size_t)g.T * g.C) return;
  const uint32_t c = (uint32_t)(idx % g.C), t = (uint32_t)(idx / g.C), Kc = g.Kc;
  float s = 0.f;
  for (uint32_t j = 0; j < Kc; ++j) {
    const int src = (int)t - (int)(Kc - 1) + (int)j;
    const float x = src >= 0 ? bf16f(g.qkv[(size_t)src * g.C + c]) : g.conv_state[(size_t)c * Kc + Kc + src];
    s = fmaf(bf16f(g.conv_w[(size_t)c * Kc + j]), x, s);
  }
  act[idx] = siluf_(s);
}

// The conv state after the prompt: slot j holds the input of token T - Kc + j (the
// old state's slot T + j for the ones before the prompt; read before written).
__global__ void conv_state_kernel(const Gdn g) {
  const uint32_t c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= g.C) return;
  const uint32_t Kc = g.Kc;
  float* st = g.conv_state + (size_t)c * Kc;
  for (uint32_t j = 0; j < Kc; ++j) {
    const int src = (int)g.T - (int)Kc + (int)j;
    st[j] = src >= 0 ? bf16f(g.qkv[(size_t)src * g.C + c]) : st[g.T + j];
  }
}

// Per token: the Q and K heads L2-normalised (eps 1e-6) and every channel rounded
// to bf16 (qkv_smooth); the decay gate and beta of every v-head (fp32).
__global__ void __launch_bounds__(256) gdn_prep_kernel(const Gdn g, const float* act) {
  const uint32_t t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* a = act + (size_t)t * g.C;
  uint16_t* q = g.qs + (size_t)t * g.C;
  const uint32_t nqk = 2 * g.Hk;
  for (uint32_t hd = warp; hd < nqk; hd += blockDim.x >> 5) {
    float ss = 0.f;
    for (uint32_t i = lane; i < g.Dk; i += 32) ss = fmaf(a[hd * g.Dk + i], a[hd * g.Dk + i], ss);
    const float inv = rsqrtf(warp_sum(ss) + 1e-6f);
    for (uint32_t i = lane; i < g.Dk; i += 32) q[hd * g.Dk + i] = to_bf16(a[hd * g.Dk + i] * inv);
  }
  for (uint32_t c = nqk * g.Dk + threadIdx.x; c < g.C; c += blockDim.x) q[c] = to_bf16(a[c]);
  for (uint32_t h = threadIdx.x; h < g.Hv; h += blockDim.x) {
    const float x = bf16f(g.dt_raw[(size_t)t * g.Hv + h]) + bf16f(g.dt_bias[h]);
    const float sp = x > 20.f ? x : log1pf(expf(x));
    g.gb[((size_t)t * g.Hv + h) * 2] = expf(sp * -expf(g.a_log[h]));
    g.gb[((size_t)t * g.Hv + h) * 2 + 1] = sigmoidf_(bf16f(g.b_raw[(size_t)t * g.Hv + h]));
  }
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// The delta rule over the T tokens for one state block (v-head h, columns
// [32 cb, 32 cb + 32)): with RG row groups, lane (c = lane % CW, group = lane / CW)
// of warp w holds rows [group Dk/RG, +Dk/RG) of column CW w + c in registers for the
// whole prompt (CW = 32 / RG columns per warp, 32 / CW warps). Per token: S = g S;
// u = S^T k; S += k (beta (v - u)); y = S^T q / sqrt(Dk), the column sums over the
// row groups by log2(RG) shuffles. The tokens' k, q, v, gate and beta come through
// shared memory in chunks of 32 tokens, copied asynchronously one chunk ahead.
template <int DK>
struct alignas(16) RecTok {
  uint16_t k[DK];
  uint16_t q[DK];
  uint16_t v[32];
  float gb[4];  // gate, beta (two words of padding)
};
template <int DK, int RG>
__global__ void __launch_bounds__(32 * RG) gdn_rec_kernel(const Gdn g) {
  constexpr int RPT = DK / RG, CW = 32 / RG, CH = 32, PK = DK / 8, PER = 2 * PK + 4 + 1;
  static_assert(RPT % 8 == 0, "rows per lane in whole 16-byte pieces");
  __shared__ RecTok<DK> buf[2][CH];
  const uint32_t h = blockIdx.x, cb = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t c = CW * warp + (lane % CW), grp = lane / CW, r0 = grp * RPT;
  const uint32_t nb = g.Dv / 32, j = h / (g.Hv / g.Hk);
  const uint32_t kbase = g.Hk * DK + j * DK, qbase = j * DK, vbase = 2 * g.Hk * DK + h * g.Dv + 32 * cb;
  auto stage = [&](uint32_t c0, int b) {  // tokens [c0, c0 + CH) into buffer b
    for (uint32_t i = threadIdx.x; i < (uint32_t)(CH * PER); i += blockDim.x) {
      const uint32_t tt = i / PER, p = i % PER, t = c0 + tt;
      if (t >= g.T) continue;
      const uint16_t* qs = g.qs + (size_t)t * g.C;
      RecTok<DK>& d = buf[b][tt];
      if (p < (uint32_t)PK) cp_async16(&d.k[8 * p], qs + kbase + 8 * p);
      else if (p < (uint32_t)(2 * PK)) cp_async16(&d.q[8 * (p - PK)], qs + qbase + 8 * (p - PK));
      else if (p < (uint32_t)(2 * PK + 4)) cp_async16(&d.v[8 * (p - 2 * PK)], qs + vbase + 8 * (p - 2 * PK));
      else cp_async8(&d.gb[0], g.gb + ((size_t)t * g.Hv + h) * 2);
    }
    cp_async_commit();
  };
  auto colsum = [](float x) {
#pragma unroll
    for (int o = CW; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
  };
  float* S = g.ssm + ((size_t)(h * nb + cb) * DK) * 32;
  float st[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) st[i] = S[(r0 + i) * 32 + c];
  const float rs = rsqrtf((float)DK);
  const uint32_t nch = (g.T + CH - 1) / CH;
  stage(0, 0);
  for (uint32_t ci = 0; ci < nch; ++ci) {
    if (ci + 1 < nch) {
      stage((ci + 1) * CH, (ci + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // chunk ci is in shared memory for every thread
    const uint32_t n = min((uint32_t)CH, g.T - ci * CH);
    for (uint32_t tt = 0; tt < n; ++tt) {
      const RecTok<DK>& d = buf[ci & 1][tt];
      const float gh = d.gb[0], bh = d.gb[1];
      const float v = bf16f(d.v[c]);
      float kx[RPT], qx[RPT];
#pragma unroll
      for (int i = 0; i < RPT; i += 8) {
        unpack8(*reinterpret_cast<const uint4*>(&d.k[r0 + i]), kx + i);
        unpack8(*reinterpret_cast<const uint4*>(&d.q[r0 + i]), qx + i);
      }
      float ua[4] = {0.f, 0.f, 0.f, 0.f};  // four chains, summed in a fixed order
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        st[i] *= gh;
        ua[i & 3] = fmaf(st[i], kx[i], ua[i & 3]);
      }
      const float u = colsum((ua[0] + ua[1]) + (ua[2] + ua[3]));
      const float dlt = bh * (v - u);
      float ya[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        st[i] = fmaf(kx[i], dlt, st[i]);
        ya[i & 3] = fmaf(st[i], qx[i], ya[i & 3]);
      }
      const float y = colsum((ya[0] + ya[1]) + (ya[2] + ya[3]));
      const uint32_t t = ci * CH + tt;
      if (grp == 0) g.y[(size_t)t * g.Hv * g.Dv + h * g.Dv + 32 * cb + c] = to_bf16(y * rs);
    }
    __syncthreads();  // buffer ci & 1 is free for chunk ci + 2
  }
#pragma unroll
  for (int i = 0; i < RPT; ++i) S[(r0 + i) * 32 + c] = st[i];
}

// Per (token, v-head) one warp: y_norm = bf16(RMSNorm(y_h) * norm_w), then the
// out_proj input bf16(SiLU(z) * y_norm).
__global__ void __launch_bounds__(128) gdn_out_kernel(const Gdn g) {
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t item = blockIdx.x * 4 + warp;
  if (item >= g.T * g.Hv) return;
  const size_t base = (size_t)item * g.Dv;  // [t][h] rows of Dv
  float ss = 0.f;
  for (uint32_t d = lane; d < g.Dv; d += 32) {
    const float v = bf16f(g.y[base + d]);
    ss = fmaf(v, v, ss);
  }
  const float inv = rsqrtf(warp_sum(ss) / (float)g.Dv + g.eps);
  for (uint32_t d = lane; d < g.Dv; d += 32) {
    const float yn = round_bf16(bf16f(g.y[base + d]) * inv * bf16f(g.norm_w[d]));
    g.yin[base + d] = to_bf16(siluf_(bf16f(g.z[base + d])) * yn);
  }
}

}  // namespace

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}
// A 2D tensor map over a row-major [rows][cols] matrix (row stride in bytes), boxes
// of 64 columns x box_rows rows, zero fill outside.
bool tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
             uint64_t stride_bytes, uint32_t box_rows, CUtensorMapSwizzle sw) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {stride_bytes};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

cudaError_t gemm(const Gemm& g, cudaStream_t st) {
  if (g.T == 0) return cudaSuccess;
  GemmArgs a;
  a.g = g;
  if (!tmap_2d(&a.tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.X, g.K, g.T, (uint64_t)g.ldx * 2, kBN,
               CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tmap_2d(&a.tc, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.codes, g.K, g.N, g.K, kBM, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  const auto k = g.exact ? gemm_kernel<true> : gemm_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e != cudaSuccess) return e;
  const uint32_t tiles = ((g.N + kBM - 1) / kBM) * ((g.T + kBN - 1) / kBN), nk = g.K / 64;
  // split K while the tiles would leave more than half of the 152 SMs idle
  uint32_t splits = 1;
  if (g.ws && tiles * 2 <= 152) splits = std::min(std::min(152u / tiles, 8u), nk);
  if (splits < 2) a.g.ws = nullptr, splits = 1;
  const dim3 grid((g.N + kBM - 1) / kBM, (g.T + kBN - 1) / kBN, splits);
  k<<<grid, kGemmThreads, kGemmSmem, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || splits == 1) return e;
  const size_t total = (size_t)g.T * g.N;
  const uint32_t blocks = (uint32_t)std::min<size_t>((total + 255) / 256, 152 * 8);
  gemm_finish_kernel<<<blocks, 256, 0, st>>>(a.g, splits);
  return cudaGetLastError();
}

cudaError_t rmsnorm(const uint16_t* a, const uint16_t* b, uint16_t* resid, const uint16_t* w, uint16_t* out,
                    uint32_t T, uint32_t E, float eps, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  rmsnorm_kernel<<<T, 256, 0, st>>>(a, b, resid, w, out, E, eps);
  return cudaGetLastError();
}

cudaError_t silu_mul(const uint16_t* g, const uint16_t* u, uint16_t* h, size_t n, cudaStream_t st) {
  const size_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  const uint32_t blocks = (uint32_t)std::min<size_t>((n8 + 255) / 256, 152 * 8);
  silu_mul_kernel<<<blocks, 256, 0, st>>>(g, u, h, n8);
  return cudaGetLastError();
}

namespace {
template <int D, int HPG>
cudaError_t attn_launch(const Attn& a, dim3 grid, cudaStream_t st) {
  // key and value tiles (32 rows; bf16, K rows padded by 8, or fp32 decoded Turbo8
  // rows, K rows padded by 4) and 8 tokens' q rows
  if (a.turbo8) {
    const uint32_t bytes = (32 * (D + 4) + 32 * D) * 4 + 8 * HPG * D * 2;
    cudaError_t e =
        cudaFuncSetAttribute(attn_kernel<D, HPG, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    attn_kernel<D, HPG, true><<<grid, 256, bytes, st>>>(a);
  } else {
    const uint32_t bytes = (32 * (D + 8) + 32 * D + 8 * HPG * D) * 2;
    cudaError_t e =
        cudaFuncSetAttribute(attn_kernel<D, HPG, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    attn_kernel<D, HPG, false><<<grid, 256, bytes, st>>>(a);
  }
  return cudaGetLastError();
}
template <int D>
cudaError_t attn_for(const Attn& a, dim3 grid, cudaStream_t st) {
  switch (a.H / a.Hkv) {
    case 1: return attn_launch<D, 1>(a, grid, st);
    case 2: return attn_launch<D, 2>(a, grid, st);
    case 4: return attn_launch<D, 4>(a, grid, st);
    case 8: return attn_launch<D, 8>(a, grid, st);
  }
  return cudaErrorInvalidValue;
}
}  // namespace

cudaError_t attention(const Attn& a, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  const uint32_t items = a.T * (a.H + 2 * a.Hkv), blocks = (items + 3) / 4;
  switch (a.D) {
    case 64: qk_rope_kernel<2><<<blocks, 128, 0, st>>>(a); break;
    case 128: qk_rope_kernel<4><<<blocks, 128, 0, st>>>(a); break;
    case 256: qk_rope_kernel<8><<<blocks, 128, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid((a.T + 7) / 8, a.Hkv);
  switch (a.D) {
    case 64: return attn_for<64>(a, grid, st);
    case 128: return attn_for<128>(a, grid, st);
    case 256: return attn_for<256>(a, grid, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t gdn(const Gdn& g, cudaStream_t st) {
  if (g.T == 0) return cudaSuccess;
  const size_t n = (size_t)g.T * g.C;
  conv_kernel<<<(uint32_t)((n + 255) / 256), 256, 0, st>>>(g, g.act);
  conv_state_kernel<<<(g.C + 255) / 256, 256, 0, st>>>(g);
  gdn_prep_kernel<<<g.T, 256, 0, st>>>(g, g.act);
  const dim3 grid(g.Hv, g.Dv / 32);
  switch (g.Dk) {  // rows per lane: 8 (Dk 32), 8 (Dk 64), 16 (Dk 128)
    case 32: gdn_rec_kernel<32, 4><<<grid, 128, 0, st>>>(g); break;
    case 64: gdn_rec_kernel<64, 8><<<grid, 256, 0, st>>>(g); break;
    case 128: gdn_rec_kernel<128, 8><<<grid, 256, 0, st>>>(g); break;
    default: return cudaErrorInvalidValue;
  }
  gdn_out_kernel<<<(g.T * g.Hv + 3) / 4, 128, 0, st>>>(g);
  return cudaGetLastError();
}

}  // namespace q35pf
