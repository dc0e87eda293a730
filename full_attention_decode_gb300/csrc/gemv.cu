// Quantised GEMV y = W x for int8 group-64 affine weights (the QuantWeights::gemv
// family of the pages "full_attention.rs" and "linear_attention.rs": gemv,
// gemv_gate_up_with, gemv_silu_gate, gemv_silu_gate_resid), on sm_103a.
//
// One launch covers up to four matrices that read the same input vector (their
// rows are concatenated), so q/k/v, a/b/qkv/z and gate/up each take one launch.
// Each CTA owns a contiguous, balanced range of rows. A producer warp streams the
// rows' codes, scales and biases through a ring of shared-memory stages with bulk
// (TMA-engine) copies and mbarriers; the first stages are issued before the
// kernel waits on its predecessor, since weights never depend on it.
//
// Eight consumer warps keep their slice of x in registers for the whole kernel,
// as 16-bit fixed point per 16-element chunk (x ~= q * 2^(e-15), q = 256 hi + lo,
// a power-of-two scale per chunk; exact for every element within 2^8 of its
// chunk's largest, since bf16 carries 8 significant bits). A 16-code chunk then
// costs eight dp4a, which give sum (c - 128) q exactly in int32, and the group
// identity
//     sum_k (s_g c_k + b_g) x_k = s_g * sum_k (c_k - 128) x_k + (b_g + 128 s_g) * sum_k x_k
// applies the scale and bias once per chunk. The -128 offset keeps the two terms
// from cancelling when b is close to -128 s (the usual affine 8-bit format).
// Each warp accumulates four tiles' rows in registers and reduces them together
// with one transposed warp reduction (6 shuffles per 4 rows).
//
// The prologue forms x from the preceding kernel's outputs (RMSNorm, residual
// add + RMSNorm, SiLU gating, per-head RMSNorm with SiLU(z) gating) and the
// epilogue optionally adds a residual, so the pages' separate rms_norm,
// add_rms_norm and sigmoid/SiLU launches disappear into the GEMVs.
#include "common.cuh"
#include "kernels.h"

namespace q35 {

namespace {

struct Tile {
  uint32_t r, nr, seg;
};

// The CTA's rows [r, re) cut into tiles of at most R rows that never straddle a
// segment end. Producer and consumers walk the same sequence.
struct TileIter {
  uint32_t r, re, R, seg;
  __device__ __forceinline__ bool next(const GemvArgs& a, Tile& t) {
    if (r >= re) return false;
    while (r >= a.seg[seg].row0 + a.seg[seg].rows) ++seg;
    const uint32_t end = min(re, a.seg[seg].row0 + a.seg[seg].rows);
    t.r = r;
    t.nr = min(R, end - r);
    t.seg = seg;
    r += t.nr;
    return true;
  }
};

__device__ __forceinline__ void unpack8(const uint4 u, float* x) {
  x[0] = bf16lo(u.x); x[1] = bf16hi(u.x);
  x[2] = bf16lo(u.y); x[3] = bf16hi(u.y);
  x[4] = bf16lo(u.z); x[5] = bf16hi(u.z);
  x[6] = bf16lo(u.w); x[7] = bf16hi(u.w);
}
__device__ __forceinline__ void load16(const uint16_t* p, float* x) {
  unpack8(*reinterpret_cast<const uint4*>(p), x);
  unpack8(*reinterpret_cast<const uint4*>(p + 8), x + 8);
}

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

__device__ __forceinline__ void quantize16(const float* v, XQ& q) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  // amax = m * 2^e with 0.5 <= m < 1, e = E - 126 for the biased exponent E; the
  // scale is 2^(e-15). Chunks whose largest element is below 2^-112 count as zero.
  const uint32_t E = __float_as_uint(amax) >> 23;
  const bool nz = E >= 15;
  const float up = __uint_as_float((268u - (nz ? E : 15u)) << 23);  // 2^(15-e)
  q.scale = nz ? __uint_as_float((E - 14u) << 23) : 0.f;             // 2^(e-15)
  int qs = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t hi = 0, lo = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int t = nz ? __float2int_rn(v[4 * w + j] * up) : 0;
      t = max(-32768, min(32767, t));
      qs += t;
      hi |= (uint32_t)((t >> 8) & 0xFF) << (8 * j);
      lo |= (uint32_t)(t & 0xFF) << (8 * j);
    }
    q.hi[w] = hi;
    q.lo[w] = lo;
  }
  q.qsum128 = 128 * qs;
}

// sum over the 16 codes of one chunk of (c - 128) * x, from dp4a on 16-bit x.
__device__ __forceinline__ float dot16(const uint4 w, const XQ& q) {
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
  return (float)(ah * 256 + (int)al) * q.scale;
}

// Sum over the 32 lanes of v[0..3]; lane L ends with the total of v[2*b4 + b3]
// (b4, b3 = bits 4 and 3 of L).
__device__ __forceinline__ float reduce4(const float* v, uint32_t lane) {
  const bool b4 = lane & 16, b3 = lane & 8;
  const float w0 = (b4 ? v[2] : v[0]) + __shfl_xor_sync(0xffffffffu, b4 ? v[0] : v[2], 16);
  const float w1 = (b4 ? v[3] : v[1]) + __shfl_xor_sync(0xffffffffu, b4 ? v[1] : v[3], 16);
  float z = (b3 ? w1 : w0) + __shfl_xor_sync(0xffffffffu, b3 ? w0 : w1, 8);
  z += __shfl_xor_sync(0xffffffffu, z, 4);
  z += __shfl_xor_sync(0xffffffffu, z, 2);
  z += __shfl_xor_sync(0xffffffffu, z, 1);
  return z;
}

template <typename T>
__device__ __forceinline__ T sel4(const T* v, uint32_t j) {
  return j == 0 ? v[0] : j == 1 ? v[1] : j == 2 ? v[2] : v[3];
}

template <int PRO, int EPI, int CPL>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_q8g64_kernel(const __grid_constant__ GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.bar_off);
  uint64_t* empty = full + a.nstage;
  float* red = reinterpret_cast<float*>(empty + a.nstage);  // [2][4 tiles][8 warps]
  float* pro = red + 64;                                    // [8] prologue partial sums

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t G = gridDim.x, bid = blockIdx.x;
  const uint32_t rb = (uint32_t)(((uint64_t)a.total_rows * bid) / G);
  const uint32_t re = (uint32_t)(((uint64_t)a.total_rows * (bid + 1)) / G);
  const uint32_t W = a.W, R = kGemvConsumerWarps / W;

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < a.nstage; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGemvConsumerWarps);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == kGemvConsumerWarps) {
    // ------------------------------------------------ producer
    if (lane == 0) {
      // Pull this CTA's whole weight range toward L2 first: under programmatic
      // dependent launch this overlaps the predecessor, so HBM stays busy across
      // the kernel boundary and the ring below refills from L2.
      for (uint32_t sg = 0; sg < a.nseg; ++sg) {
        const GemvSeg& s = a.seg[sg];
        const uint32_t lo = max(rb, s.row0), hi = min(re, s.row0 + s.rows);
        if (lo >= hi) continue;
        const uint32_t l0 = lo - s.row0, n = hi - lo;
        prefetch_l2(s.codes + (size_t)l0 * a.K, (uint64_t)n * a.K);
        prefetch_l2(s.scales + (size_t)l0 * a.gstride, (uint64_t)n * a.gstride * 2);
        prefetch_l2(s.biases + (size_t)l0 * a.gstride, (uint64_t)n * a.gstride * 2);
      }
      const uint64_t pol = policy_evict_first();
      TileIter it{rb, re, R, 0};
      Tile t;
      uint32_t i = 0;
      bool waited = false, ok = true;
      while (it.next(a, t)) {
        const uint32_t st = i % a.nstage;
        if (i >= a.nstage) {
          if (!waited) {  // the ring is primed: now depend on the predecessor
            pdl_wait();
            pdl_launch();
            waited = true;
          }
          if (!mbar_wait(&empty[st], ((i / a.nstage) - 1) & 1)) {
            set_status(a.status, kStatusTimeout);
            ok = false;
            break;
          }
        }
        const GemvSeg& s = a.seg[t.seg];
        const uint32_t local = t.r - s.row0;
        uint8_t* dst = smem + st * a.stage_stride;
        const uint32_t cb = t.nr * a.K, sb = t.nr * a.gstride * 2;
        mbar_arrive_expect_tx(&full[st], cb + 2 * sb);
        bulk_g2s_stream(dst, s.codes + (size_t)local * a.K, cb, &full[st], pol);
        bulk_g2s_stream(dst + a.stage_scale_off, s.scales + (size_t)local * a.gstride, sb, &full[st], pol);
        bulk_g2s_stream(dst + a.stage_bias_off, s.biases + (size_t)local * a.gstride, sb, &full[st], pol);
        ++i;
      }
      if (!waited) {
        pdl_wait();
        pdl_launch();
      }
      if (!ok) {  // let the copies already issued land before the CTA can exit
        const uint32_t first = i > a.nstage ? i - a.nstage : 0;
        for (uint32_t j = first; j < i; ++j) mbar_wait(&full[j % a.nstage], (j / a.nstage) & 1);
      }
    }
    return;
  }

  // -------------------------------------------------- consumers
  pdl_wait();
  pdl_launch();

  const uint32_t kp = warp % W, rs = warp / W, nchunks = a.K / 16;
  // chunk c of this lane: index lane + 32 (kp + W c); chunks past the row end are
  // read at index 0 (valid memory) against x = 0, so every loop is branch-free.
  uint32_t chk[CPL];
  bool valid[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const uint32_t ch = lane + 32 * (kp + W * c);
    valid[c] = ch < nchunks;
    chk[c] = valid[c] ? ch : 0;
  }

  // ---- per-CTA statistics of the prologue
  float inv = 0.f;
  if constexpr (PRO == kProRmsNorm || PRO == kProAddRmsNorm) {
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      if (valid[c]) {
        float xa[16];
        load16(a.a + chk[c] * 16, xa);
        if constexpr (PRO == kProAddRmsNorm) {
          float xb[16];
          load16(a.b + chk[c] * 16, xb);
#pragma unroll
          for (int j = 0; j < 16; ++j) xa[j] = round_bf16(xa[j] + xb[j]);
          if (bid == 0 && rs == 0) {  // the rows-0 warps of CTA 0 cover x once: store x_resid
            uint32_t pk[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              pk[j] = (uint32_t)to_bf16(xa[2 * j]) | ((uint32_t)to_bf16(xa[2 * j + 1]) << 16);
            uint4* dst = reinterpret_cast<uint4*>(a.resid_out + chk[c] * 16);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) ss = fmaf(xa[j], xa[j], ss);
      }
    }
    ss = warp_sum(ss);
    if (W > 1) {  // the W warps of a row group hold disjoint parts of x
      if (lane == 0) pro[warp] = ss;
      named_barrier(1, kGemvConsumerWarps * 32);
      ss = 0.f;
      for (uint32_t w = 0; w < W; ++w) ss += pro[rs * W + w];
    }
    inv = rsqrtf(ss / (float)a.K + a.eps);
  }

  // ---- this lane's x chunks, quantised
  XQ xq[CPL];
  float xs[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    float v[16];
    const uint32_t k0 = chk[c] * 16;
    float xa[16];
    load16(a.a + k0, xa);
    if constexpr (PRO == kProPlain) {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = xa[j];
    } else if constexpr (PRO == kProRmsNorm) {
      float w[16];
      load16(a.nw + k0, w);
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = round_bf16(xa[j] * inv * w[j]);
    } else if constexpr (PRO == kProAddRmsNorm) {
      float xb[16], w[16];
      load16(a.b + k0, xb);
      load16(a.nw + k0, w);
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = round_bf16(round_bf16(xa[j] + xb[j]) * inv * w[j]);
    } else if constexpr (PRO == kProSiluMul) {
      float xb[16];
      load16(a.b + k0, xb);
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = silu_fast(xa[j]) * xb[j];
    } else {  // kProHeadNormSilu: a = y, b = z; the head's chunks sit on adjacent lanes
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) ss = fmaf(xa[j], xa[j], ss);
      for (uint32_t o = 1; o < a.head_dim / 16; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float hi = rsqrtf(ss / (float)a.head_dim + a.eps);
      float xb[16], w[16];
      load16(a.b + k0, xb);
      load16(a.nw + k0 % a.head_dim, w);
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = silu_fast(xb[j]) * round_bf16(xa[j] * hi * w[j]);
    }
    if (!valid[c]) {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = 0.f;
    }
    xs[c] = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) xs[c] += v[j];
    quantize16(v, xq[c]);
  }

  // ---- main loop: batches of four tiles, one row per warp per tile
  TileIter it{rb, re, R, 0};
  uint32_t i = 0, batch = 0;
  bool dead = false;  // a wait gave up: keep joining the barriers, compute nothing
  const uint32_t jl = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);  // tile whose total this lane ends with
  while (true) {
    float acc[4];
    uint32_t trow[4], tcnt[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[j] = 0.f;
      trow[j] = 0;
      tcnt[j] = 0;
      Tile t;
      if (it.next(a, t)) {
        trow[j] = t.r;
        tcnt[j] = t.nr;
        const uint32_t st = i % a.nstage;
        if (!dead && !mbar_wait(&full[st], (i / a.nstage) & 1)) {
          set_status(a.status, kStatusTimeout);
          dead = true;
        }
        if (!dead && rs < t.nr) {
          const uint8_t* sbase = smem + st * a.stage_stride;
          const uint8_t* crow = sbase + rs * a.K;
          const uint16_t* srow = reinterpret_cast<const uint16_t*>(sbase + a.stage_scale_off) + rs * a.gstride;
          const uint16_t* brow = reinterpret_cast<const uint16_t*>(sbase + a.stage_bias_off) + rs * a.gstride;
          float part[CPL];
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const uint4 w = *reinterpret_cast<const uint4*>(crow + chk[c] * 16);
            const float s = bf16f(srow[chk[c] >> 2]);
            const float b = fmaf(128.0f, s, bf16f(brow[chk[c] >> 2]));
            part[c] = fmaf(s, dot16(w, xq[c]), b * xs[c]);
          }
#pragma unroll
          for (int c = 1; c < CPL; ++c) part[0] += part[c];
          acc[j] = part[0];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done reading the stage
        ++i;
      }
    }
    if (tcnt[0] == 0) break;
    const float tot = reduce4(acc, lane);
    const uint32_t r0 = sel4(trow, jl), n0 = sel4(tcnt, jl);
    bool store = false;
    float y = tot;
    if (W == 1) {
      store = (lane & 7) == 0 && rs < n0;
    } else {
      float* buf = red + (batch & 1) * 32;
      if ((lane & 7) == 0) buf[jl * 8 + warp] = tot;
      named_barrier(1, kGemvConsumerWarps * 32);
      if (kp == 0 && (lane & 7) == 0 && rs < n0) {
        y = 0.f;
        for (uint32_t w = 0; w < W; ++w) y += buf[jl * 8 + rs * W + w];
        store = true;
      }
    }
    if (store && !dead) {
      const uint32_t row = r0 + rs;
      uint32_t sg = 0;
      while (row >= a.seg[sg].row0 + a.seg[sg].rows) ++sg;
      const uint32_t local = row - a.seg[sg].row0;
      if constexpr (EPI == kEpiResid) y += bf16f(a.resid_in[local]);
      a.seg[sg].out[local] = to_bf16(y);
    }
    ++batch;
    if (tcnt[3] == 0) break;
  }
}

__global__ void dequant_kernel(const uint8_t* codes, const uint16_t* scales, const uint16_t* biases,
                               uint32_t n, uint32_t k, uint32_t gstride, float* out) {
  const uint64_t total = (uint64_t)n * k;
  for (uint64_t e = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; e < total;
       e += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t r = (uint32_t)(e / k), c = (uint32_t)(e % k);
    const float s = bf16f(scales[(size_t)r * gstride + c / 64]);
    const float b = bf16f(biases[(size_t)r * gstride + c / 64]);
    out[e] = fmaf(s, (float)codes[e], b);
  }
}

using GemvKernel = void (*)(GemvArgs);

template <int CPL>
GemvKernel pick_cpl(int pro, int epi) {
  if (epi == kEpiResid) return pro == kProSiluMul ? gemv_q8g64_kernel<kProSiluMul, kEpiResid, CPL> : nullptr;
  switch (pro) {
    case kProPlain: return gemv_q8g64_kernel<kProPlain, kEpiStore, CPL>;
    case kProRmsNorm: return gemv_q8g64_kernel<kProRmsNorm, kEpiStore, CPL>;
    case kProAddRmsNorm: return gemv_q8g64_kernel<kProAddRmsNorm, kEpiStore, CPL>;
    case kProSiluMul: return gemv_q8g64_kernel<kProSiluMul, kEpiStore, CPL>;
    case kProHeadNormSilu: return gemv_q8g64_kernel<kProHeadNormSilu, kEpiStore, CPL>;
  }
  return nullptr;
}

GemvKernel pick_kernel(int pro, int epi, uint32_t cpl) {
  switch (cpl) {
    case 1: return pick_cpl<1>(pro, epi);
    case 2: return pick_cpl<2>(pro, epi);
    case 3: return pick_cpl<3>(pro, epi);
    case 4: return pick_cpl<4>(pro, epi);
    case 5: return pick_cpl<5>(pro, epi);
  }
  return nullptr;
}

}  // namespace

bool gemv_plan(GemvPlan& p, int num_sms) {
  GemvArgs& a = p.args;
  if (a.K == 0 || a.K % 64 != 0 || a.K > (uint32_t)kGemvMaxK || a.nseg == 0 || a.nseg > kGemvMaxSegs) return false;
  const uint32_t nchunks = a.K / 16;
  a.W = 0;
  for (uint32_t W = 1; W <= 8; W *= 2) {
    const uint32_t cpl = (nchunks + 32 * W - 1) / (32 * W);
    if (cpl <= (uint32_t)kGemvCplMax) {
      a.W = W;
      a.cpl = cpl;
      break;
    }
  }
  if (a.W == 0) return false;
  const uint32_t R = kGemvConsumerWarps / a.W;
  a.gstride = ((a.K / 64 + 7) / 8) * 8;
  const uint32_t cb = R * a.K, sb = R * a.gstride * 2;
  a.stage_scale_off = (cb + 15) / 16 * 16;
  a.stage_bias_off = a.stage_scale_off + sb;
  a.stage_stride = (a.stage_bias_off + sb + 127) / 128 * 128;
  a.nstage = kGemvSmemBudget / a.stage_stride;
  if (a.nstage > 8) a.nstage = 8;
  if (a.nstage < 2) return false;
  a.bar_off = a.nstage * a.stage_stride;
  p.smem = a.bar_off + 2 * a.nstage * 8 + 64 * 4 + 8 * 4;
  uint32_t total = 0;
  for (uint32_t s = 0; s < a.nseg; ++s) {
    a.seg[s].row0 = total;
    total += a.seg[s].rows;
  }
  a.total_rows = total;
  if (total == 0) return false;
  if (p.prologue == kProHeadNormSilu) {
    // a head's chunks must sit on adjacent lanes of one warp
    const uint32_t m = a.head_dim / 16;
    if (a.head_dim % 16 || m == 0 || m > 32 || (m & (m - 1)) || a.K % a.head_dim) return false;
  }
  p.grid = total < (uint32_t)num_sms ? total : (uint32_t)num_sms;
  return pick_kernel(p.prologue, p.epilogue, a.cpl) != nullptr;
}

cudaError_t gemv_launch(const GemvPlan& p, cudaStream_t stream, bool pdl) {
  GemvKernel k = pick_kernel(p.prologue, p.epilogue, p.args.cpl);
  if (!k) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, p.args);
}

cudaError_t gemv_set_attributes() {
  const int pros[5] = {kProPlain, kProRmsNorm, kProAddRmsNorm, kProSiluMul, kProHeadNormSilu};
  for (uint32_t cpl = 1; cpl <= (uint32_t)kGemvCplMax; ++cpl)
    for (int epi = 0; epi < 2; ++epi)
      for (int pi = 0; pi < 5; ++pi) {
        GemvKernel k = pick_kernel(pros[pi], epi, cpl);
        if (!k) continue;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kGemvSmemBudget + 4096);
        if (e != cudaSuccess) return e;
      }
  return cudaSuccess;
}

cudaError_t dequant_launch(const uint8_t* codes, const uint16_t* scales, const uint16_t* biases, uint32_t n,
                           uint32_t k, uint32_t gstride, float* out, cudaStream_t stream) {
  const uint64_t total = (uint64_t)n * k;
  uint64_t blocks = (total + 255) / 256;
  if (blocks > 65535) blocks = 65535;
  dequant_kernel<<<(unsigned)blocks, 256, 0, stream>>>(codes, scales, biases, n, k, gstride, out);
  return cudaGetLastError();
}

}  // namespace q35
