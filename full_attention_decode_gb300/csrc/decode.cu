// Host side of the persistent decode kernel (decode_kernel.cuh): the checks of a
// program's dimensions against the kernel's buffers, the choice of ring and
// phase-buffer sizes, and the launch.
#include "decode_kernel.cuh"

namespace q35 {
namespace {

// The instantiation for a program: attention head dim and q-heads per warp, GDN
// key head dim, and whether it decodes a batch of sequences (the single-sequence
// kernel has no sequence loop).
DecodeKernel pick(uint32_t D, uint32_t hpw, uint32_t Dk, bool batched) {
  switch (D) {
    case 64: return decode_kernel_d64(hpw, Dk, batched);
    case 128: return decode_kernel_d128(hpw, Dk, batched);
    case 256: return decode_kernel_d256(hpw, Dk, batched);
  }
  return nullptr;
}

}  // namespace

bool decode_dims_ok(const Program& p, bool has_fa, bool has_gdn, int num_sms) {
  // a GEMV phase of K columns and N rows: its tile fits a ring tile, its input
  // chunks, the CTA's partial sums and residual rows fit the phase buffer
  const uint32_t room = p.union_bytes;
  if (p.ring_bytes + p.union_bytes + kDecFixed != (uint32_t)kDecSmem || p.ring_bytes % 128 ||
      p.ring_bytes < (uint32_t)kDecTileMax)
    return false;
  // a CTA's row range is computed in 32 bits (rows < 2^24, CTAs <= 256), and the
  // down projection's residual rows of a CTA are one per consumer thread at most
  if (num_sms <= 0 || num_sms > 256 || (p.E + num_sms - 1) / num_sms > (uint32_t)NCT) return false;
  auto gemv_ok = [&](uint32_t K, uint32_t N) {
    if (K == 0 || K % 64 || K > 12288 || N == 0 || N >= (1u << 24)) return false;
    if (p.batch > 1) {  // tensor-core passes: one sequence's staged input fits; a tile fits;
      // the down projection's residual rows of a pass fit their buffer
      if ((p.E + num_sms - 1) / num_sms * kMaxBatch * 4 > kBatchResid) return false;
      const uint32_t R = batch_rows(K), gs = ((K / 64 + 7) / 8) * 8;
      return batch_seq_bytes(K) + kBatchPart <= room &&
             (R * K + 15) / 16 * 16 + 4 * R * gs <= (uint32_t)kDecTileMax;
    }
    const uint32_t nch = K / 16;
    uint32_t W, cpl;
    pick_split(nch, W, cpl);
    if (W == 0) return false;
    const uint32_t R = NCW / W, gs = ((K / 64 + 7) / 8) * 8;
    const uint32_t stage = (R * K + 15) / 16 * 16 + 2 * R * gs * 2;
    const uint32_t rows = (N + num_sms - 1) / num_sms;
    return stage <= (uint32_t)kDecTileMax && nch * 48 + (W + 1) * rows * 4 <= room;
  };
  for (uint32_t l = 0; l < p.n_layers; ++l) {
    const LayerDesc& L = p.layers[l];
    auto n = [&](int i) { return L.m[i].n; };
    bool ok = true;
    if (L.kind == kLayerGemv || L.kind == kLayerHead) {
      ok = gemv_ok(p.E, n(0));
    } else if (L.kind == kLayerFA) {
      ok = gemv_ok(p.E, n(0) + n(1) + n(2)) && gemv_ok(p.H * p.D, n(3)) && gemv_ok(p.E, n(4) + n(5)) &&
           gemv_ok(p.I, n(6));
    } else if (L.kind == kLayerGDN) {
      ok = gemv_ok(p.E, n(0) + n(1) + n(2) + n(3)) && gemv_ok(p.Z, n(7)) && gemv_ok(p.E, n(4) + n(5)) &&
           gemv_ok(p.I, n(6));
    } else {
      ok = false;
    }
    if (!ok) return false;
  }
  if (has_fa) {
    if (p.D != 64 && p.D != 128 && p.D != 256) return false;
    const uint32_t hpw = attn_hpw(p.H, p.Hkv);
    if (hpw == 0 || p.Hkv > 8) return false;
    const uint32_t rowbytes = p.Hkv * p.D * 2;
    if (2 * kTS * rowbytes > (uint32_t)kDecTileMax) return false;
    const uint32_t NG = p.H / hpw, TI = NCW / NG;
    if (TI == 0) return false;
    const uint32_t fresh = 2 * p.Hkv * p.D * 4;
    const uint32_t rope = NCW * p.D * 4, merge = TI > 1 ? NG * hpw * (p.D + 2) * 4 : 0;
    if (1024 + fresh + (rope > merge ? rope : merge) > room) return false;  // angle table, new row, buffers
    if (3 * NCW * 32 * 4 > room) return false;
    if (p.P == 0 || p.P > (uint32_t)kDecMaxSplits) return false;
    if (p.H * (p.D / 32) == 0) return false;
  }
  if (has_gdn) {
    if (p.Dk != 32 && p.Dk != 64 && p.Dk != 128) return false;
    if (p.Dv % 32 || p.Dv == 0 || p.Kc == 0 || p.Kc > (uint32_t)kMaxKc) return false;
    const uint32_t m = p.Dv / 16;
    if (m > 32 || (m & (m - 1))) return false;  // a head's chunks on adjacent lanes
    if ((2 * p.Dk + 32) > (uint32_t)NCT) return false;
    if (gdn_tile_bytes(p.Dk, p.Kc) > (uint32_t)kDecTileMax) return false;  // one ring tile
  }
  return true;
}

bool decode_pick_split(Program& p, bool has_fa, bool has_gdn, int num_sms) {
  bool ok = false;
  if (p.batch <= 1) {
    p.ring_bytes = kDecRingLarge;
    p.union_bytes = kDecUnionSmall;
    ok = decode_dims_ok(p, has_fa, has_gdn, num_sms);
  }
  if (!ok) {
    p.ring_bytes = kDecRing;
    p.union_bytes = kDecUnion;
    ok = decode_dims_ok(p, has_fa, has_gdn, num_sms);
  }
  if (ok) fill_shapes(p);
  return ok;
}

cudaError_t decode_set_attributes() {
  const uint32_t Ds[3] = {64, 128, 256}, Hs[2] = {1, 2}, Dks[3] = {32, 64, 128};
  for (uint32_t d : Ds)
    for (uint32_t h : Hs)
      for (uint32_t k : Dks)
        for (bool bt : {false, true}) {
          DecodeKernel f = pick(d, h, k, bt);
          if (!f) continue;
          cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem);
          if (e != cudaSuccess) return e;
        }
  return cudaSuccess;
}

cudaError_t decode_launch(const Program& p, int num_sms, cudaStream_t stream) {
  // the head dims select the attention and GDN phase code; a program without those
  // phases (a GEMV alone) runs on any instantiation
  const uint32_t hpw = attn_hpw(p.H, p.Hkv);
  const uint32_t D = (p.D == 64 || p.D == 128 || p.D == 256) ? p.D : 256;
  const uint32_t Dk = (p.Dk == 32 || p.Dk == 64 || p.Dk == 128) ? p.Dk : 128;
  DecodeKernel f = pick(D, hpw ? hpw : 1, Dk, p.batch > 1);
  if (!f) return cudaErrorInvalidValue;
  // every sequence's tagged words start the launch at zero (not written yet)
  const uint32_t tb = p.sm.tag_begin, te = p.sm.tag_end;
  if (te > tb) {
    cudaError_t e;
    if (p.batch <= 1)
      e = cudaMemsetAsync(p.scratch + tb, 0, te - tb, stream);
    else
      e = cudaMemset2DAsync(p.scratch + tb, p.seq_stride, 0, te - tb, p.batch, stream);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = kDecSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, f, p);
}

}  // namespace q35
