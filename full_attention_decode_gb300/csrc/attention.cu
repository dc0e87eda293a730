// Decode attention of the full-attention layer ("full_attention.rs",
// forward_full_attention, from the qkv split through sigmoid_gate), on sm_103a.
//
// attn_kernel: split-KV ("flash decoding") over the sequence. CTA s owns tokens
// [s*S/P, (s+1)*S/P) of every kv-head, so each K/V row (all kv-heads of a token,
// contiguous in the [capacity][Hkv][D] cache) is read from HBM exactly once. A
// producer warp streams the cached rows into a shared-memory ring with bulk copies
// before the kernel waits on its predecessor (those rows do not depend on it).
// Each consumer warp owns q-heads that share one kv-head (GQA packing): it reads
// the q_proj output directly with the [Q_h | gate_h] split folded into the
// indexing, applies the per-head RMSNorm and RoPE on the first rotary_dim dims,
// and runs an online softmax over the split. The CTA whose split holds the new
// token forms k (RMSNorm + RoPE) and v itself, appends them at row cache_pos, and
// attends to that token from shared memory, so no CTA reads a row being written.
//
// attn_combine_kernel: merges the P partial (max, sum, output) triples per head
// and applies the output gate: ga = bf16(bf16(attn) * sigmoid(gate)).
#include "common.cuh"
#include "kernels.h"

namespace q35 {
namespace {

// q-heads per consumer warp: the heads are spread over the 8 warps.
__host__ __device__ inline uint32_t hpw_of(uint32_t H) { return H > kAttnConsumerWarps ? H / kAttnConsumerWarps : 1; }

// Position and attended length: host values, or read from device memory.
struct PosInfo {
  uint32_t pos, S;
  bool ok;
};
__device__ __forceinline__ PosInfo read_pos(const AttnArgs& a) {
  PosInfo r;
  if (a.d_pos) {
    const int32_t p = *a.d_pos;
    const uint32_t lim = min(a.capacity, a.max_seq);
    r.ok = p >= 0 && (uint32_t)p < lim;
    r.pos = r.ok ? (uint32_t)p : 0;
    r.S = r.pos + 1;
  } else {
    r.ok = true;
    r.pos = a.cache_pos;
    r.S = a.S;
  }
  return r;
}

template <int EPL>
__device__ __forceinline__ void load_row(const uint16_t* p, float* x) {
  if constexpr (EPL == 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    x[0] = bf16lo(u.x); x[1] = bf16hi(u.x); x[2] = bf16lo(u.y); x[3] = bf16hi(u.y);
    x[4] = bf16lo(u.z); x[5] = bf16hi(u.z); x[6] = bf16lo(u.w); x[7] = bf16hi(u.w);
  } else if constexpr (EPL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    x[0] = bf16lo(u.x); x[1] = bf16hi(u.x); x[2] = bf16lo(u.y); x[3] = bf16hi(u.y);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    x[0] = bf16lo(u); x[1] = bf16hi(u);
  }
}

// RMSNorm over one head (this lane's EPL elements at d = lane*EPL), rounded to
// bf16, then RoPE on dims [0, R) with rotate-half pairing, rounded to bf16.
// buf: this warp's D floats of shared memory.
template <int EPL>
__device__ __forceinline__ void norm_rope(float* x, const uint16_t* w, float eps, uint32_t D, uint32_t R,
                                          uint32_t pos, const float* inv_freq, float* buf, uint32_t lane) {
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) ss = fmaf(x[e], x[e], ss);
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)D + eps);
  float wv[EPL];
  load_row<EPL>(w + lane * EPL, wv);
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    x[e] = round_bf16(x[e] * inv * wv[e]);
    buf[lane * EPL + e] = x[e];
  }
  __syncwarp();
  const uint32_t half = R / 2;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const uint32_t d = lane * EPL + e;
    if (d < R) {
      const uint32_t i = d < half ? d : d - half;
      float sn, cs;
      sincosf((float)pos * inv_freq[i], &sn, &cs);
      x[e] = d < half ? round_bf16(buf[d] * cs - buf[d + half] * sn)
                      : round_bf16(buf[d] * cs + buf[d - half] * sn);
    }
  }
  __syncwarp();
}

// Sum over the 32 lanes of v[0..NV-1] (NV = 8, 16 or 32): each step hands half of
// the remaining values to the partner lane. Lane L ends with the total of
// v[L >> (5 - log2 NV)]; the 32/NV lanes that share an index hold the same value.
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
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      n = h;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
  return v[0];
}

template <int D, int HPW>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int EPL = D / 32;
  constexpr int TS = kAttnTile;              // tokens per stage
  constexpr int NV = HPW * TS;               // scores per stage and warp
  constexpr int SH = NV == 8 ? 2 : NV == 16 ? 1 : 0;
  static_assert(NV == 8 || NV == 16 || NV == 32, "scores per stage");
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.bar_off);
  uint64_t* empty = full + a.nstage;
  float* qbuf = reinterpret_cast<float*>(smem + a.q_off);       // [8 warps][D]
  float* fresh = reinterpret_cast<float*>(smem + a.fresh_off);  // k then v, [Hkv][D] each

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t s = blockIdx.x;
  const uint32_t rowh = a.Hkv * D;  // elements per cache row
  const uint32_t rowbytes = rowh * 2;

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < a.nstage; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kAttnConsumerWarps);
    }
    mbar_fence_init();
  }
  __syncthreads();

  const PosInfo pi = read_pos(a);
  const uint32_t t0 = (uint32_t)(((uint64_t)pi.S * s) / a.P);
  const uint32_t t1 = (uint32_t)(((uint64_t)pi.S * (s + 1)) / a.P);
  const bool has_fresh = pi.S == pi.pos + 1 && pi.pos >= t0 && pi.pos < t1;
  const uint32_t tc_end = has_fresh ? pi.pos : t1;  // cached rows [t0, tc_end)
  const uint32_t ntiles = (pi.ok && tc_end > t0) ? (tc_end - t0 + TS - 1) / TS : 0;

  if (warp == kAttnConsumerWarps) {
    // ------------------------------------------------ producer
    if (lane == 0) {
      if (tc_end > t0 && pi.ok) {  // the cached rows of this split, toward L2 (see the GEMV)
        prefetch_l2(a.kc + (size_t)t0 * rowh, (uint64_t)(tc_end - t0) * rowbytes);
        prefetch_l2(a.vc + (size_t)t0 * rowh, (uint64_t)(tc_end - t0) * rowbytes);
      }
      bool waited = false, ok = true;
      uint32_t i = 0;
      for (; i < ntiles; ++i) {
        const uint32_t st = i % a.nstage;
        if (i >= a.nstage) {
          if (!waited) {
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
        const uint32_t tt = t0 + i * TS;
        const uint32_t n = min((uint32_t)TS, tc_end - tt);
        uint8_t* dst = smem + st * a.stage_stride;
        mbar_arrive_expect_tx(&full[st], 2 * n * rowbytes);
        bulk_g2s(dst, a.kc + (size_t)tt * rowh, n * rowbytes, &full[st]);
        bulk_g2s(dst + TS * rowbytes, a.vc + (size_t)tt * rowh, n * rowbytes, &full[st]);
      }
      if (!waited) {
        pdl_wait();
        pdl_launch();
      }
      if (!ok) {
        const uint32_t first = i > a.nstage ? i - a.nstage : 0;
        for (uint32_t j = first; j < i; ++j) mbar_wait(&full[j % a.nstage], (j / a.nstage) & 1);
      }
    }
    return;
  }

  // -------------------------------------------------- consumers
  pdl_wait();
  pdl_launch();
  if (!pi.ok) {
    if (s == 0 && threadIdx.x == 0) set_status(a.status, kStatusRange);
    return;
  }

  // The new token's k (normed, rotated) and v: needed by the split that attends
  // to it, and appended to the cache by exactly one CTA.
  const bool appender = has_fresh || (pi.S != pi.pos + 1 && s == 0);
  if (appender) {
    for (uint32_t g = warp; g < a.Hkv; g += kAttnConsumerWarps) {
      float kx[EPL], vx[EPL];
      load_row<EPL>(a.k_new + g * D + lane * EPL, kx);
      load_row<EPL>(a.v_new + g * D + lane * EPL, vx);
      norm_rope<EPL>(kx, a.k_norm, a.eps, D, a.R, pi.pos, a.inv_freq, qbuf + warp * D, lane);
      uint16_t* kd = a.kc + (size_t)pi.pos * rowh + g * D + lane * EPL;
      uint16_t* vd = a.vc + (size_t)pi.pos * rowh + g * D + lane * EPL;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        fresh[g * D + lane * EPL + e] = kx[e];
        fresh[rowh + g * D + lane * EPL + e] = vx[e];
        kd[e] = to_bf16(kx[e]);
        vd[e] = to_bf16(vx[e]);
      }
    }
  }

  // This warp's q-heads (consecutive, one kv-head): normed and rotated, in registers.
  const uint32_t h0 = warp * HPW;
  const bool active = h0 < a.H;
  const uint32_t g = active ? h0 / (a.H / a.Hkv) : 0;
  float q[HPW][EPL];
  float m[HPW], l[HPW], acc[HPW][EPL];
#pragma unroll
  for (int j = 0; j < HPW; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      acc[j][e] = 0.f;
      q[j][e] = 0.f;
    }
    if (active) {
      load_row<EPL>(a.q_full + (size_t)(h0 + j) * 2 * D + lane * EPL, q[j]);
      norm_rope<EPL>(q[j], a.q_norm, a.eps, D, a.R, pi.pos, a.inv_freq, qbuf + warp * D, lane);
    }
  }
  named_barrier(1, kAttnConsumerWarps * 32);  // the fresh row is visible to every warp

  // after the transposed reduction this lane holds the score of (head mj, token mt)
  const uint32_t midx = lane >> SH, mj = midx / TS, mt = midx % TS;
  for (uint32_t i = 0; i < ntiles; ++i) {
    const uint32_t st = i % a.nstage;
    if (!mbar_wait(&full[st], (i / a.nstage) & 1)) {
      set_status(a.status, kStatusTimeout);
      return;
    }
    const uint8_t* base = smem + st * a.stage_stride;
    const uint32_t n = min((uint32_t)TS, tc_end - (t0 + i * TS));
    if (active) {
      float d[NV];
#pragma unroll
      for (int t = 0; t < TS; ++t) {  // rows t >= n hold stale data; their scores are masked
        float kf[EPL];
        load_row<EPL>(reinterpret_cast<const uint16_t*>(base + t * rowbytes) + g * D + lane * EPL, kf);
#pragma unroll
        for (int j = 0; j < HPW; ++j) {
          float x = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) x = fmaf(q[j][e], kf[e], x);
          d[j * TS + t] = x;
        }
      }
      float sc = reduce_transposed<NV>(d, lane) * a.scale_log2;
      sc = mt < n ? sc : -INFINITY;
      float mx = sc;
#pragma unroll
      for (int o = 1 << SH; o < (TS << SH); o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float mold = m[0];
#pragma unroll
      for (int j = 1; j < HPW; ++j) mold = mj == (uint32_t)j ? m[j] : mold;
      const float mnew = fmaxf(mold, mx);
      const float p = exp2f(sc - mnew);
      float ps = p;
#pragma unroll
      for (int o = 1 << SH; o < (TS << SH); o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
#pragma unroll
      for (int j = 0; j < HPW; ++j) {
        const float mn = __shfl_sync(0xffffffffu, mnew, (j * TS) << SH);
        const float sum = __shfl_sync(0xffffffffu, ps, (j * TS) << SH);
        const float corr = exp2f(m[j] - mn);
        l[j] = fmaf(l[j], corr, sum);
        m[j] = mn;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[j][e] *= corr;
      }
      for (uint32_t t = 0; t < n; ++t) {
        float vf[EPL];
        load_row<EPL>(reinterpret_cast<const uint16_t*>(base + (TS + t) * rowbytes) + g * D + lane * EPL, vf);
#pragma unroll
        for (int j = 0; j < HPW; ++j) {
          const float pj = __shfl_sync(0xffffffffu, p, (j * TS + t) << SH);
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[j][e] = fmaf(pj, vf[e], acc[j][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  if (has_fresh && active) {
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
      const float sc = warp_sum(x) * a.scale_log2;
      const float mn = fmaxf(m[j], sc);
      const float corr = exp2f(m[j] - mn), p = exp2f(sc - mn);
      l[j] = fmaf(l[j], corr, p);
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[j][e] = fmaf(acc[j][e], corr, p * vf[e]);
      m[j] = mn;
    }
  }
  if (active) {
#pragma unroll
    for (int j = 0; j < HPW; ++j) {
      const uint32_t h = h0 + j;
      float* po = a.part_o + ((size_t)s * a.H + h) * D + lane * EPL;
#pragma unroll
      for (int e = 0; e < EPL; ++e) po[e] = acc[j][e];
      if (lane == 0) {
        a.part_ml[((size_t)s * a.H + h) * 2 + 0] = m[j];
        a.part_ml[((size_t)s * a.H + h) * 2 + 1] = l[j];
      }
    }
  }
}

// grid (H, D / 32), 256 threads: lane = output dim, warp w merges splits w, w+8, ...
// (loads issued together, then an online merge), and warp 0 merges the 8 warps.
__global__ void __launch_bounds__(256) attn_combine_kernel(const __grid_constant__ AttnArgs a) {
  __shared__ float part[3][8][32];
  pdl_wait();
  pdl_launch();
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t h = blockIdx.x, d = blockIdx.y * 32 + lane;
  const PosInfo pi = read_pos(a);
  const size_t oi = (size_t)h * a.D + d;
  if (!pi.ok) {
    if (warp == 0) a.ga[oi] = 0;
    return;
  }
  float M = -INFINITY, L = 0.f, O = 0.f;
  for (uint32_t base = 0; base < a.P; base += 8 * 8) {
    float ms[8], ls[8], os[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t sp = base + warp + 8 * k;
      const bool ok = sp < a.P;
      ms[k] = ok ? a.part_ml[((size_t)sp * a.H + h) * 2] : -INFINITY;
      ls[k] = ok ? a.part_ml[((size_t)sp * a.H + h) * 2 + 1] : 0.f;
      os[k] = ok ? a.part_o[((size_t)sp * a.H + h) * a.D + d] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (ms[k] == -INFINITY) continue;  // a split with no tokens
      const float mn = fmaxf(M, ms[k]);
      const float c0 = exp2f(M - mn), c1 = exp2f(ms[k] - mn);
      L = L * c0 + ls[k] * c1;
      O = O * c0 + os[k] * c1;
      M = mn;
    }
  }
  part[0][warp][lane] = M;
  part[1][warp][lane] = L;
  part[2][warp][lane] = O;
  __syncthreads();
  if (warp != 0) return;
  M = -INFINITY;
#pragma unroll
  for (int w = 0; w < 8; ++w) M = fmaxf(M, part[0][w][lane]);
  L = 0.f;
  O = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const float mw = part[0][w][lane];
    if (mw == -INFINITY) continue;
    const float c = exp2f(mw - M);
    L = fmaf(part[1][w][lane], c, L);
    O = fmaf(part[2][w][lane], c, O);
  }
  const float attn = round_bf16(O / L);
  const float gate = bf16f(a.q_full[(size_t)h * 2 * a.D + a.D + d]);
  a.ga[oi] = to_bf16(attn * sigmoidf_(gate));
}

template <int D, int HPW>
cudaError_t launch_d(const AttnPlan& p, cudaStream_t stream, bool pdl) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.args.P);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_kernel<D, HPW>, p.args);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(p.args.H, D / 32);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.numAttrs = 1;  // the combine always follows the attention kernel
  return cudaLaunchKernelEx(&cfg, attn_combine_kernel, p.args);
}

}  // namespace

bool attn_plan(AttnPlan& p) {
  AttnArgs& a = p.args;
  if (a.D != 64 && a.D != 128 && a.D != 256) return false;
  if (a.Hkv == 0 || a.Hkv > 8 || a.H % a.Hkv) return false;
  const uint32_t hpw = hpw_of(a.H);
  if (a.H > kAttnConsumerWarps && a.H % kAttnConsumerWarps) return false;
  if ((hpw != 1 && hpw != 2 && hpw != 4) || hpw > a.H / a.Hkv) return false;
  if (a.R % 2 || a.R > a.D || a.R / 2 > (uint32_t)kAttnMaxHalfRot) return false;
  if (a.P == 0 || a.P > (uint32_t)kAttnMaxSplits) return false;
  const uint32_t rowbytes = a.Hkv * a.D * 2;
  a.TS = kAttnTile;
  a.stage_stride = (2 * a.TS * rowbytes + 127) / 128 * 128;
  a.nstage = 98304 / a.stage_stride;
  if (a.nstage > 8) a.nstage = 8;
  if (a.nstage < 2) a.nstage = 2;
  a.bar_off = a.nstage * a.stage_stride;
  a.q_off = a.bar_off + 2 * a.nstage * 8;
  a.q_off = (a.q_off + 15) / 16 * 16;
  a.fresh_off = a.q_off + kAttnConsumerWarps * a.D * 4;
  p.smem = a.fresh_off + 2 * a.Hkv * a.D * 4;
  return p.smem <= (uint32_t)kAttnSmemBudget + 32768;
}

template <int D>
cudaError_t launch_h(const AttnPlan& p, cudaStream_t stream, bool pdl) {
  switch (hpw_of(p.args.H)) {
    case 1: return launch_d<D, 1>(p, stream, pdl);
    case 2: return launch_d<D, 2>(p, stream, pdl);
    case 4: return launch_d<D, 4>(p, stream, pdl);
  }
  return cudaErrorInvalidValue;
}

cudaError_t attn_launch(const AttnPlan& p, cudaStream_t stream, bool pdl) {
  switch (p.args.D) {
    case 64: return launch_h<64>(p, stream, pdl);
    case 128: return launch_h<128>(p, stream, pdl);
    case 256: return launch_h<256>(p, stream, pdl);
  }
  return cudaErrorInvalidValue;
}

template <int D>
cudaError_t set_attr_d() {
  const int lim = kAttnSmemBudget + 32768;
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_kernel<D, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_kernel<D, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  return e;
}

cudaError_t attn_set_attributes() {
  cudaError_t e = set_attr_d<64>();
  if (e == cudaSuccess) e = set_attr_d<128>();
  if (e == cudaSuccess) e = set_attr_d<256>();
  return e;
}

}  // namespace q35
