// Device helpers for the decode megakernel: PTX wrappers (mbarrier, bulk copy, acquire/release,
// timers) and the register dequantisation of bf16 / FP8-E4M3 / NVFP4 weight words.
// sm_103a only.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace mk {

// ------------------------------------------------------------------ special registers
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint64_t clock64_() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t smid() {
  uint32_t s;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
  return s;
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ------------------------------------------------------------------ gpu-scope ordering
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_acqrel_add(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void fence_acqrel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// 64-bit integer add at gpu scope, no return value (count-word contributions).
__device__ __forceinline__ void red_add_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Activations written by other SMs are read at L2 (never through a possibly stale L1 line).
__device__ __forceinline__ float ld_cg_f32(const float* p) {
  float v;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cg_f32x4(const float* p) {
  float4 v;
  asm volatile("ld.relaxed.gpu.global.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// Named barrier over the consumer warps only (id 1); the producer warp never joins it.
__device__ __forceinline__ void bar_consumers(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ mbarrier + bulk copy
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
// count arrivals at once (a release on behalf of every consumer warp)
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking probe of a phase (never suspends the thread; callers spin on it).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// Global -> this CTA's shared memory, completion counted on `bar` (bytes must be a multiple of
// 16, both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ------------------------------------------------------------------ debug bounds checks
// Built with MK_DEBUG_BOUNDS (libmk_debug.so), a checked access whose index is out of range is
// skipped and recorded: status word 0 = 5 (first failure wins), word 1 = site << 24 | low bits of
// the index, word 2 = 1 (every CTA stops at its next wait). In the normal build the check is
// compiled away (always true). status: the SyncBlock's status words, or null.
__device__ __forceinline__ bool mk_in_bounds(bool ok, uint32_t* status, uint32_t site, uint32_t value) {
#ifdef MK_DEBUG_BOUNDS
  if (!ok && status) {
    if (atomicCAS(&status[0], 0u, 5u) == 0u) st_relaxed_u32(&status[1], (site << 24) | (value & 0xFFFFFFu));
    st_relaxed_u32(&status[2], 1u);
  }
  return ok;
#else
  (void)ok, (void)status, (void)site, (void)value;
  return true;
#endif
}

// ------------------------------------------------------------------ register dequantisation
// E4M3 pair (low byte = first element) -> two floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t pair16) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)pair16));
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}
// E2M1 pair (low nibble = first element) -> two floats (exact).
__device__ __forceinline__ float2 e2m1x2_to_f2(uint32_t byte) {
  uint32_t h;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h) : "r"(byte));
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// (a0, a1) += (w0 * x0, w1 * x1) as one packed instruction; each lane is exactly fmaf.
__device__ __forceinline__ void ffma2(float& a0, float& a1, float w0, float w1, float x0, float x1) {
  asm("{ .reg .b64 A, W, X;\n\t"
      "mov.b64 A, {%0, %1};\n\t"
      "mov.b64 W, {%2, %3};\n\t"
      "mov.b64 X, {%4, %5};\n\t"
      "fma.rn.f32x2 A, W, X, A;\n\t"
      "mov.b64 {%0, %1}, A; }"
      : "+f"(a0), "+f"(a1)
      : "f"(w0), "f"(w1), "f"(x0), "f"(x1));
}

// 16 bytes of weights times the matching activations, accumulated into acc[0..1] (two independent
// chains keep the FMA dependency short: even elements into acc[0], odd into acc[1]).
// bf16: 8 weights, x: 2 float4. FP8: 16 weights, x: 4 float4.
__device__ __forceinline__ void dot_bf16_16B(uint4 w, const float4* x, float* acc) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lo = __uint_as_float(ws[i] << 16), hi = __uint_as_float(ws[i] & 0xFFFF0000u);
    const float4 xv = x[i / 2];
    float xa = (i & 1) ? xv.z : xv.x, xb = (i & 1) ? xv.w : xv.y;
    ffma2(acc[0], acc[1], lo, hi, xa, xb);
  }
}
__device__ __forceinline__ void dot_fp8_16B(uint4 w, const float4* x, float* acc) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 a = e4m3x2_to_f2(ws[i] & 0xFFFFu), b = e4m3x2_to_f2(ws[i] >> 16);
    const float4 xv = x[i];
    ffma2(acc[0], acc[1], a.x, a.y, xv.x, xv.y);
    ffma2(acc[0], acc[1], b.x, b.y, xv.z, xv.w);
  }
}
// NVFP4: 16 bytes = 32 weights = two 16-element scale blocks; x: 8 float4; s0/s1: block scales.
__device__ __forceinline__ void dot_nvfp4_16B(uint4 w, const float4* x, float s0, float s1, float* acc) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  float blk[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float2 v = e2m1x2_to_f2((ws[i] >> (8 * b)) & 0xFFu);
      const int e = i * 8 + b * 2;  // element index within the lane's 32
      const float4 xv = x[e / 4];
      float xa = (e % 4 == 0) ? xv.x : xv.z, xb = (e % 4 == 0) ? xv.y : xv.w;
      ffma2(blk[i / 2][0], blk[i / 2][1], v.x, v.y, xa, xb);
    }
  }
  acc[0] = fmaf(blk[0][0] + blk[0][1], s0, acc[0]);
  acc[1] = fmaf(blk[1][0] + blk[1][1], s1, acc[1]);
}

}  // namespace mk
