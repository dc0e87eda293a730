// Device helpers shared by the sm_103a kernels: bf16 conversions, mbarriers,
// bulk (TMA-engine) copies global -> shared, programmatic dependent launch, the
// tagged words through which CTAs hand each other their results, and waits
// bounded in time that report through the device status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace q35 {

constexpr int kStatusTimeout = 5;  // QWEN35_ERR_DEVICE_TIMEOUT
constexpr int kStatusRange = 6;    // QWEN35_ERR_DEVICE_RANGE
constexpr uint64_t kWaitNs = 1000000000ull;  // a bounded wait gives up after 1 s (the default)

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t to_bf16(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
__device__ __forceinline__ float round_bf16(float f) { return bf16f(to_bf16(f)); }
// The two bf16 halves of a 32-bit word as floats (low half first).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return x / (1.0f + expf(-x)); }
// SiLU with the fast exponential and division intrinsics (relative error ~1e-6,
// far below the bf16 rounding of every value it feeds); used where it runs per
// element of a GEMV input.
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Named barrier over the first `nthreads` threads of the block (id 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// n arrivals at once (a team standing in for the warps that skip the tile).
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
// Test the phase. With a nonzero QWEN35_WAIT_HINT_NS the thread may sleep in
// hardware until the phase completes or about that many ns pass; with 0 it uses
// the instruction's own (short) time limit.
#ifndef QWEN35_WAIT_HINT_NS
#define QWEN35_WAIT_HINT_NS 0
#endif
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
#if QWEN35_WAIT_HINT_NS > 0
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"((uint32_t)QWEN35_WAIT_HINT_NS)
      : "memory");
#else
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
#endif
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase with the given parity to complete; false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// ---------------------------------------------------------------- tagged words
//
// A result that other CTAs read travels as 32-bit words, the bf16 value in the
// high half and the writing phase's tag in the low half, stored and loaded at GPU
// scope without going through L1 (a relaxed access: each 32-bit word is read or
// written whole). A reader polls the words themselves until every tag is the one
// it expects, so a result is usable one L2 round trip after it is stored; the
// words are zeroed before each launch, and tags are never zero.
__device__ __forceinline__ uint32_t tag_word(float v, uint32_t tag) { return ((uint32_t)to_bf16(v) << 16) | tag; }
__device__ __forceinline__ uint32_t tag_word_bits(uint16_t b, uint32_t tag) { return ((uint32_t)b << 16) | tag; }
__device__ __forceinline__ float tag_value(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ bool tag_is(uint32_t w, uint32_t tag) { return (w & 0xFFFFu) == tag; }
__device__ __forceinline__ uint4 ld_tagged4(const uint32_t* p) {
  uint4 r;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p)
               : "memory");
  return r;
}
__device__ __forceinline__ uint32_t ld_tagged(const uint32_t* p) {
  uint32_t r;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(r) : "l"(p) : "memory");
  return r;
}
__device__ __forceinline__ void st_tagged(uint32_t* p, uint32_t w) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(w) : "memory");
}
__device__ __forceinline__ void st_tagged4(uint32_t* p, uint4 w) {
  asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(w.x), "r"(w.y), "r"(w.z),
               "r"(w.w)
               : "memory");
}
__device__ __forceinline__ bool tags4_are(const uint4 w, uint32_t tag) {
  return tag_is(w.x, tag) & tag_is(w.y, tag) & tag_is(w.z, tag) & tag_is(w.w, tag);
}
// A timeout already recorded in the status word: later waits give up at once
// (the launch's results are meaningless anyway), so that a launch whose waits run
// out ends after about one wait limit, not one per wait.
__device__ __forceinline__ bool timed_out(const int* status) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(status) : "memory");
  return v == kStatusTimeout;
}
// Load 4 tagged words and poll them until all carry `tag` (bounded); false (and
// whatever was last read) when the wait runs out.
__device__ __forceinline__ bool ld_tagged4_wait(const uint32_t* p, uint32_t tag, uint4& w, uint64_t limit_ns,
                                                const int* status) {
  w = ld_tagged4(p);
  if (tags4_are(w, tag)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t n = 1;; ++n) {
    __nanosleep(64);
    w = ld_tagged4(p);
    if (tags4_are(w, tag)) return true;
    if (global_ns() - t0 > limit_ns || ((n & 15) == 0 && timed_out(status))) return false;
  }
}
__device__ __forceinline__ bool ld_tagged_wait(const uint32_t* p, uint32_t tag, uint32_t& w, uint64_t limit_ns,
                                               const int* status) {
  w = ld_tagged(p);
  if (tag_is(w, tag)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t n = 1;; ++n) {
    __nanosleep(64);
    w = ld_tagged(p);
    if (tag_is(w, tag)) return true;
    if (global_ns() - t0 > limit_ns || ((n & 15) == 0 && timed_out(status))) return false;
  }
}
// Acquire load / release store at GPU scope (a flag that publishes other data).
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t r;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(r) : "l"(p) : "memory");
  return r;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Orders this thread's earlier memory accesses before its later ones at GPU scope
// (both ways): placed after a phase has read its inputs and before it writes, it
// makes the hand-over of tagged words a synchronisation.
__device__ __forceinline__ void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// ---------------------------------------------------------------- bulk copies

// Contiguous global -> shared copy through the bulk-copy (TMA) engine, completing
// `bytes` of transaction count on `bar`. dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// Same with an L2 evict-first policy: for data read once per decode step (weights).
__device__ __forceinline__ void bulk_g2s_stream(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
// Pull [src, src + bytes) toward L2 without staging it anywhere (16-byte aligned,
// bytes % 16 == 0); issued in pieces of at most 64 KiB.
// A hint: a request that is not 16-byte aligned in address and size is dropped.
__device__ __forceinline__ void prefetch_l2(const void* src, uint64_t bytes) {
  if ((reinterpret_cast<uintptr_t>(src) | bytes) & 15) return;
  const char* p = static_cast<const char*>(src);
  while (bytes > 0) {
    const uint32_t n = bytes > 65536 ? 65536u : (uint32_t)bytes;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(n) : "memory");
    p += n;
    bytes -= n;
  }
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- PDL

// Wait until the preceding kernel in the stream has completed and its writes are
// visible (no-op when launched without programmatic serialization).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next kernel in the stream be scheduled early.
__device__ __forceinline__ void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace q35
