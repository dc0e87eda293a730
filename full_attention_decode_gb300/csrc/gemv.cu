// Quantised GEMV y = W x for int8 group-64 affine weights (the QuantWeights::gemv
// family of the pages "full_attention.rs" and "linear_attention.rs": gemv,
// gemv_gate_up_with, gemv_silu_gate, gemv_silu_gate_resid), on sm_103a.
//
// One launch covers up to four matrices that read the same input vector (their
// rows are concatenated), so q/k/v, a/b/qkv/z and gate/up each take one launch.
// Each CTA owns a contiguous, balanced range of rows. A producer warp streams the
// rows' codes, scales and biases through a ring of shared-memory stages with bulk
// (TMA-engine) copies and mbarriers; the first stages are issued before the
// kernel waits on its predecessor, since weights never depend on it. Eight
// consumer warps each keep their slice of x in registers for the whole kernel and
// reduce rows with the group identity
//     sum_k (s_g c_k + b_g) x_k = s_g * sum_k c_k x_k + b_g * sum_k x_k,
// so each weight costs one byte-to-float conversion and one FMA (or, in the
// integer mode, a quarter of a dp4a on 16-bit fixed-point x).
// The prologue forms x from the preceding kernel's outputs (RMSNorm, residual
// add + RMSNorm, SiLU gating, per-head RMSNorm with SiLU(z) gating) and the
// epilogue optionally adds a residual, so the pages' separate rms_norm,
// add_rms_norm and sigmoid/SiLU launches disappear into the GEMVs.
#include "common.cuh"
#include "kernels.h"

namespace q35 {

int g_gemv_mode = 1;

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

// x values of the 16 inputs k0 .. k0+15 as the prologue defines them.
template <int PRO>
__device__ __forceinline__ void x_chunk(const GemvArgs& a, uint32_t k0, float inv, const float* hinv,
                                        float* v) {
  float xa[16];
  unpack8(*reinterpret_cast<const uint4*>(a.a + k0), xa);
  unpack8(*reinterpret_cast<const uint4*>(a.a + k0 + 8), xa + 8);
  if constexpr (PRO == kProPlain) {
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = xa[j];
  } else if constexpr (PRO == kProRmsNorm) {
    float w[16];
    unpack8(*reinterpret_cast<const uint4*>(a.nw + k0), w);
    unpack8(*reinterpret_cast<const uint4*>(a.nw + k0 + 8), w + 8);
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = round_bf16(xa[j] * inv * w[j]);
  } else if constexpr (PRO == kProAddRmsNorm) {
    float xb[16], w[16];
    unpack8(*reinterpret_cast<const uint4*>(a.b + k0), xb);
    unpack8(*reinterpret_cast<const uint4*>(a.b + k0 + 8), xb + 8);
    unpack8(*reinterpret_cast<const uint4*>(a.nw + k0), w);
    unpack8(*reinterpret_cast<const uint4*>(a.nw + k0 + 8), w + 8);
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = round_bf16(round_bf16(xa[j] + xb[j]) * inv * w[j]);
  } else if constexpr (PRO == kProSiluMul) {
    float xb[16];
    unpack8(*reinterpret_cast<const uint4*>(a.b + k0), xb);
    unpack8(*reinterpret_cast<const uint4*>(a.b + k0 + 8), xb + 8);
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = siluf_(xa[j]) * xb[j];
  } else {  // kProHeadNormSilu: a = y, b = z
    float xb[16], w[16];
    const uint32_t d0 = k0 % a.head_dim;
    const float hi = hinv[k0 / a.head_dim];
    unpack8(*reinterpret_cast<const uint4*>(a.b + k0), xb);
    unpack8(*reinterpret_cast<const uint4*>(a.b + k0 + 8), xb + 8);
    unpack8(*reinterpret_cast<const uint4*>(a.nw + d0), w);
    unpack8(*reinterpret_cast<const uint4*>(a.nw + d0 + 8), w + 8);
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = siluf_(xb[j]) * round_bf16(xa[j] * hi * w[j]);
  }
}

// ---- fp32 dot: a code byte becomes a float by placing it in the mantissa of
// 2^23 and subtracting 2^23 (exact), then one FMA; four partial sums.
__device__ __forceinline__ float code_f(uint32_t word, uint32_t sel) {
  return __uint_as_float(__byte_perm(word, 0x4B000000u, sel)) - 8388608.0f;
}
__device__ __forceinline__ float dot16_f32(const uint4 w, const float* x) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    a0 = fmaf(code_f(ws[j], 0x7650u), x[4 * j + 0], a0);
    a1 = fmaf(code_f(ws[j], 0x7651u), x[4 * j + 1], a1);
    a2 = fmaf(code_f(ws[j], 0x7652u), x[4 * j + 2], a2);
    a3 = fmaf(code_f(ws[j], 0x7653u), x[4 * j + 3], a3);
  }
  return (a0 + a1) + (a2 + a3);
}

// ---- integer dot: x as 16-bit fixed point per chunk (x ~= q * 2^(e-15), q =
// 256*hi + lo, hi signed byte, lo unsigned byte), sum c*q exact in int32 by dp4a.
struct XQ {
  uint32_t hi[4], lo[4];
  float scale;
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
  int e = 0;
  if (amax > 0.f) frexpf(amax, &e);  // amax = m * 2^e, 0.5 <= m < 1
  const float up = ldexpf(1.0f, 15 - e);
  q.scale = amax > 0.f ? ldexpf(1.0f, e - 15) : 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t hi = 0, lo = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int t = amax > 0.f ? __float2int_rn(v[4 * w + j] * up) : 0;
      t = max(-32768, min(32767, t));
      hi |= (uint32_t)((t >> 8) & 0xFF) << (8 * j);
      lo |= (uint32_t)(t & 0xFF) << (8 * j);
    }
    q.hi[w] = hi;
    q.lo[w] = lo;
  }
}
__device__ __forceinline__ float dot16_dp4a(const uint4 w, const XQ& q) {
  int ah = 0;
  uint32_t al = 0;
  ah = dp4a_us(w.x, q.hi[0], ah);
  ah = dp4a_us(w.y, q.hi[1], ah);
  ah = dp4a_us(w.z, q.hi[2], ah);
  ah = dp4a_us(w.w, q.hi[3], ah);
  al = dp4a_uu(w.x, q.lo[0], al);
  al = dp4a_uu(w.y, q.lo[1], al);
  al = dp4a_uu(w.z, q.lo[2], al);
  al = dp4a_uu(w.w, q.lo[3], al);
  return (float)(ah * 256 + (int)al) * q.scale;
}

template <int PRO, int EPI, int MODE>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_q8g64_kernel(const __grid_constant__ GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.bar_off);
  uint64_t* empty = full + a.nstage;
  float* red = reinterpret_cast<float*>(empty + a.nstage);  // [2][8] cross-warp partials
  float* pro = red + 16;                                    // [128] prologue statistics

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t G = gridDim.x, bid = blockIdx.x;
  const uint32_t rb = (uint32_t)(((uint64_t)a.total_rows * bid) / G);
  const uint32_t re = (uint32_t)(((uint64_t)a.total_rows * (bid + 1)) / G);
  const uint32_t R = kGemvConsumerWarps / a.W;

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

  float inv = 0.f;
  if constexpr (PRO == kProRmsNorm || PRO == kProAddRmsNorm) {
    float ss = 0.f;
    for (uint32_t k = threadIdx.x * 8; k < a.K; k += kGemvConsumerWarps * 32 * 8) {
      float x[8];
      unpack8(*reinterpret_cast<const uint4*>(a.a + k), x);
      if constexpr (PRO == kProAddRmsNorm) {
        float xb[8];
        unpack8(*reinterpret_cast<const uint4*>(a.b + k), xb);
        uint32_t packed[4];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = round_bf16(x[j] + xb[j]);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          packed[j] = (uint32_t)to_bf16(x[2 * j]) | ((uint32_t)to_bf16(x[2 * j + 1]) << 16);
        if (bid == 0) *reinterpret_cast<uint4*>(a.resid_out + k) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(x[j], x[j], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) pro[warp] = ss;
    named_barrier(1, kGemvConsumerWarps * 32);
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kGemvConsumerWarps; ++w) tot += pro[w];
    inv = rsqrtf(tot / (float)a.K + a.eps);
  }
  if constexpr (PRO == kProHeadNormSilu) {
    const uint32_t nh = a.K / a.head_dim;
    for (uint32_t h = warp; h < nh; h += kGemvConsumerWarps) {
      float ss = 0.f;
      for (uint32_t d = lane; d < a.head_dim; d += 32) {
        const float y = bf16f(a.a[h * a.head_dim + d]);
        ss = fmaf(y, y, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) pro[h] = rsqrtf(ss / (float)a.head_dim + a.eps);
    }
    named_barrier(1, kGemvConsumerWarps * 32);
  }

  // Each lane's chunks of x, kept in registers for every row of the kernel.
  const uint32_t kp = warp % a.W, rs = warp / a.W, nchunks = a.K / 16, cpl = a.cpl;
  constexpr int CPL = MODE == 0 ? kGemvCplMaxF32 : kGemvCplMax;
  float xs[CPL];
  float xr[MODE == 0 ? CPL : 1][16];
  XQ xq[MODE == 1 ? CPL : 1];
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    xs[c] = 0.f;
    if (c < (int)cpl) {
      const uint32_t ch = lane + 32 * (kp + a.W * c);
      float v[16];
      if (ch < nchunks) {
        x_chunk<PRO>(a, ch * 16, inv, pro, v);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) xs[c] += v[j];
      if constexpr (MODE == 0) {
#pragma unroll
        for (int j = 0; j < 16; ++j) xr[c][j] = v[j];
      } else {
        quantize16(v, xq[c]);
      }
    }
  }

  TileIter it{rb, re, R, 0};
  Tile t;
  uint32_t i = 0;
  bool dead = false;  // a wait gave up: keep joining the barriers, compute nothing
  while (it.next(a, t)) {
    const uint32_t st = i % a.nstage;
    if (!dead && !mbar_wait(&full[st], (i / a.nstage) & 1)) {
      set_status(a.status, kStatusTimeout);
      dead = true;
    }
    const uint8_t* sbase = smem + st * a.stage_stride;
    float acc = 0.f;
    if (rs < t.nr && !dead) {
      const uint8_t* crow = sbase + rs * a.K;
      const uint16_t* srow = reinterpret_cast<const uint16_t*>(sbase + a.stage_scale_off) + rs * a.gstride;
      const uint16_t* brow = reinterpret_cast<const uint16_t*>(sbase + a.stage_bias_off) + rs * a.gstride;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        if (c < (int)cpl) {
          const uint32_t ch = lane + 32 * (kp + a.W * c);
          if (ch < nchunks) {
            const uint4 w = *reinterpret_cast<const uint4*>(crow + ch * 16);
            const float s = bf16f(srow[ch >> 2]), b = bf16f(brow[ch >> 2]);
            float d;
            if constexpr (MODE == 0) d = dot16_f32(w, xr[c]);
            else d = dot16_dp4a(w, xq[c]);
            acc = fmaf(s, d, acc);
            acc = fmaf(b, xs[c], acc);
          }
        }
      }
      acc = warp_sum(acc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done reading the stage

    bool store = false;
    if (a.W == 1) {
      store = rs < t.nr && lane == 0;
    } else {
      if (lane == 0) red[(i & 1) * kGemvConsumerWarps + warp] = acc;
      named_barrier(1, kGemvConsumerWarps * 32);
      if (kp == 0 && lane == 0 && rs < t.nr) {
        acc = 0.f;
        for (uint32_t j = 0; j < a.W; ++j) acc += red[(i & 1) * kGemvConsumerWarps + rs * a.W + j];
        store = true;
      }
    }
    if (store && !dead) {
      const GemvSeg& s = a.seg[t.seg];
      const uint32_t local = t.r + rs - s.row0;
      float y = acc;
      if constexpr (EPI == kEpiResid) y += bf16f(a.resid_in[local]);
      s.out[local] = to_bf16(y);
    }
    ++i;
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

template <int MODE>
GemvKernel pick(int pro, int epi) {
  if (epi == kEpiResid) return pro == kProSiluMul ? gemv_q8g64_kernel<kProSiluMul, kEpiResid, MODE> : nullptr;
  switch (pro) {
    case kProPlain: return gemv_q8g64_kernel<kProPlain, kEpiStore, MODE>;
    case kProRmsNorm: return gemv_q8g64_kernel<kProRmsNorm, kEpiStore, MODE>;
    case kProAddRmsNorm: return gemv_q8g64_kernel<kProAddRmsNorm, kEpiStore, MODE>;
    case kProSiluMul: return gemv_q8g64_kernel<kProSiluMul, kEpiStore, MODE>;
    case kProHeadNormSilu: return gemv_q8g64_kernel<kProHeadNormSilu, kEpiStore, MODE>;
  }
  return nullptr;
}

GemvKernel pick_kernel(int pro, int epi, int mode) { return mode ? pick<1>(pro, epi) : pick<0>(pro, epi); }

}  // namespace

bool gemv_plan(GemvPlan& p, int num_sms) {
  GemvArgs& a = p.args;
  if (a.K == 0 || a.K % 64 != 0 || a.K > (uint32_t)kGemvMaxK || a.nseg == 0 || a.nseg > kGemvMaxSegs) return false;
  const uint32_t nchunks = a.K / 16;
  const uint32_t cpl_max = g_gemv_mode ? kGemvCplMax : kGemvCplMaxF32;
  a.W = 0;
  for (uint32_t W = 1; W <= 8; W *= 2) {
    const uint32_t cpl = (nchunks + 32 * W - 1) / (32 * W);
    if (cpl <= cpl_max) {
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
  p.smem = a.bar_off + 2 * a.nstage * 8 + 16 * 4 + 128 * 4;
  uint32_t total = 0;
  for (uint32_t s = 0; s < a.nseg; ++s) {
    a.seg[s].row0 = total;
    total += a.seg[s].rows;
  }
  a.total_rows = total;
  if (total == 0) return false;
  if (p.prologue == kProHeadNormSilu && (a.head_dim == 0 || a.head_dim % 16 || a.K % a.head_dim ||
                                         a.K / a.head_dim > 128))
    return false;
  p.grid = total < (uint32_t)num_sms ? total : (uint32_t)num_sms;
  return pick_kernel(p.prologue, p.epilogue, 0) != nullptr;
}

cudaError_t gemv_launch(const GemvPlan& p, cudaStream_t stream, bool pdl) {
  GemvKernel k = pick_kernel(p.prologue, p.epilogue, g_gemv_mode);
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
  for (int mode = 0; mode < 2; ++mode)
    for (int epi = 0; epi < 2; ++epi)
      for (int pi = 0; pi < 5; ++pi) {
        GemvKernel k = pick_kernel(pros[pi], epi, mode);
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
