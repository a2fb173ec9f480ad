// Auxiliary kernels: the device weight packers (bf16 -> FP8-E4M3 per-row, bf16 -> NVFP4), the
// RoPE cos/sin table, and a probe that runs the hardware format conversions on every input.
#include <cuda_runtime.h>

#include "mk_device.cuh"
#include "mk_internal.h"

namespace mk {

__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Two fp32 values -> two E4M3 codes (round-to-nearest-even, saturating); `lo` lands in the low byte.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}
// Two fp32 values -> two E2M1 codes (round-to-nearest-even, saturating); `lo` in the low nibble.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint32_t d;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ float e4m3_to_f(uint8_t c) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)c));
  return __half2float(__ushort_as_half((uint16_t)(h & 0xFFFFu)));
}

// ---------------------------------------------------------------- FP8 per-row packer
// One warp per row: scale = fp32(absmax / 448), rounded to nearest-even bf16 when bf16_scale;
// code = E4M3_RNE_satfinite(fp32(w / scale)).
__global__ void k_pack_fp8(const uint16_t* __restrict__ w, int rows, int cols, uint8_t* __restrict__ codes,
                           float* __restrict__ scales, int bf16_scale) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const uint16_t* row = w + (size_t)warp * cols;
  float amax = 0.f;
  for (int k = lane; k < cols; k += 32) amax = fmaxf(amax, fabsf(bf16_to_f(row[k])));
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  float s = __fdiv_rn(amax, 448.0f);
  if (bf16_scale) {  // s is finite and non-negative: round the low 16 bits away, ties to even
    const uint32_t u = __float_as_uint(s);
    s = __uint_as_float((u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u);
  }
  if (lane == 0) scales[warp] = s;
  uint8_t* out = codes + (size_t)warp * cols;
  for (int k = 2 * lane; k < cols; k += 64) {
    uint16_t pair = 0;
    if (s != 0.f) pair = f32x2_to_e4m3x2(__fdiv_rn(bf16_to_f(row[k]), s), __fdiv_rn(bf16_to_f(row[k + 1]), s));
    out[k] = (uint8_t)(pair & 0xFF);
    out[k + 1] = (uint8_t)(pair >> 8);
  }
}

// ---------------------------------------------------------------- NVFP4 packer
__global__ void k_amax(const uint16_t* __restrict__ w, size_t n, uint32_t* amax_bits) {
  float m = 0.f;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    m = fmaxf(m, fabsf(bf16_to_f(w[i])));
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));  // non-negative: uint order
}
__global__ void k_tscale(float* t) { t[0] = __fdiv_rn(t[0], 2688.0f); }  // 2688 = 6 * 448

// One thread per 16-element block: b = E4M3_RNE(amax_block / fp32(6 t)); code = E2M1_RNE(w / fp32(b t)).
__global__ void k_pack_nvfp4(const uint16_t* __restrict__ w, int rows, int cols, uint8_t* __restrict__ codes,
                             uint8_t* __restrict__ bscales, const float* __restrict__ tscale) {
  const size_t nb = (size_t)rows * (cols / 16);
  const size_t blk = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= nb) return;
  const float t = tscale[0];
  const float t6 = __fmul_rn(6.0f, t);
  const uint16_t* src = w + blk * 16;
  float v[16];
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    v[j] = bf16_to_f(src[j]);
    amax = fmaxf(amax, fabsf(v[j]));
  }
  uint8_t bcode = 0;
  if (t6 != 0.f) bcode = (uint8_t)(f32x2_to_e4m3x2(__fdiv_rn(amax, t6), 0.f) & 0xFF);
  bscales[blk] = bcode;
  const float denom = __fmul_rn(e4m3_to_f(bcode), t);
  uint8_t* out = codes + blk * 8;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t byte = 0;
    if (denom != 0.f) byte = f32x2_to_e2m1x2(__fdiv_rn(v[2 * j], denom), __fdiv_rn(v[2 * j + 1], denom));
    out[j] = (uint8_t)byte;
  }
}

// The value of an E2M1 code (hardware decode of the low nibble).
__device__ __forceinline__ double e2m1_to_d(uint32_t nib) {
  uint32_t h;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h) : "r"(nib & 0xFu));
  return (double)__half2float(__ushort_as_half((uint16_t)(h & 0xFFFFu)));
}

// Codes of one 16-element block for block-scale code c (same quotient rule as k_pack_nvfp4) and its
// squared reconstruction error, summed in double in element order with no fused multiply-add.
__device__ double nvfp4_block_err(const float* v, uint32_t c, float t, uint8_t* out) {
  const float ef = e4m3_to_f((uint8_t)c);
  const float denom = __fmul_rn(ef, t);
  const double sc = __dmul_rn((double)ef, (double)t);
  double err = 0.0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t byte = 0;
    if (denom != 0.f) byte = f32x2_to_e2m1x2(__fdiv_rn(v[2 * j], denom), __fdiv_rn(v[2 * j + 1], denom));
    out[j] = (uint8_t)byte;
    const double d0 = __dsub_rn((double)v[2 * j], __dmul_rn(e2m1_to_d(byte), sc));
    err = __dadd_rn(err, __dmul_rn(d0, d0));
    const double d1 = __dsub_rn((double)v[2 * j + 1], __dmul_rn(e2m1_to_d(byte >> 4), sc));
    err = __dadd_rn(err, __dmul_rn(d1, d1));
  }
  return err;
}

// NVFP4 with a per-block scale search: one thread per 16-element block tries every E4M3 code
// 0 .. 0x7E as its block scale and keeps the one with the least squared reconstruction error,
// ties to the smaller code (an all-zero block keeps code 0).
__global__ void k_pack_nvfp4_mse(const uint16_t* __restrict__ w, int rows, int cols, uint8_t* __restrict__ codes,
                                 uint8_t* __restrict__ bscales, const float* __restrict__ tscale) {
  const size_t nb = (size_t)rows * (cols / 16);
  const size_t blk = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= nb) return;
  const float t = tscale[0];
  const uint16_t* src = w + blk * 16;
  float v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = bf16_to_f(src[j]);
  uint8_t best[8], cand[8];
  uint32_t bc = 0;
  double be = nvfp4_block_err(v, 0, t, best);
  for (uint32_t c = 1; c <= 0x7Eu; ++c) {
    const double e = nvfp4_block_err(v, c, t, cand);
    if (e < be) {
      be = e;
      bc = c;
#pragma unroll
      for (int j = 0; j < 8; ++j) best[j] = cand[j];
    }
  }
  bscales[blk] = (uint8_t)bc;
  uint8_t* out = codes + blk * 8;
#pragma unroll
  for (int j = 0; j < 8; ++j) out[j] = best[j];
}

// ---------------------------------------------------------------- RoPE table
// cos/sin of pos * theta^(-2i/128), angle and trig in double, stored as fp32.
__global__ void k_rope_table(float* cosb, float* sinb, int max_ctx, double theta) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= max_ctx * (HD / 2)) return;
  const int pos = idx / (HD / 2), i = idx % (HD / 2);
  const double inv = pow(theta, -2.0 * i / (double)HD);
  const double ang = (double)pos * inv;
  double s, c;
  sincos(ang, &s, &c);
  cosb[idx] = (float)c;
  sinb[idx] = (float)s;
}

// ---------------------------------------------------------------- conversion probe
__global__ void k_probe_cvt(uint32_t* f16_e4m3, uint32_t* f16_e2m1, const float* in, int n, uint16_t* e4, uint8_t* e2) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (f16_e4m3 && i < 65536) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)i));
    f16_e4m3[i] = h;
  }
  if (f16_e2m1 && i < 256) {
    uint32_t h;
    asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h) : "r"((uint32_t)i));
    f16_e2m1[i] = h;
  }
  if (in && i < n / 2) {
    const float a = in[2 * i], b = in[2 * i + 1];
    if (e4) e4[i] = f32x2_to_e4m3x2(a, b);
    if (e2) e2[i] = (uint8_t)f32x2_to_e2m1x2(a, b);
  }
}

// ---------------------------------------------------------------- launchers
int launch_pack_fp8(const void* w, int rows, int cols, void* codes, float* scales, int bf16_scale, void* stream) {
  const int threads = 256, warps_per_block = threads / 32;
  const int blocks = (rows + warps_per_block - 1) / warps_per_block;
  k_pack_fp8<<<blocks, threads, 0, (cudaStream_t)stream>>>((const uint16_t*)w, rows, cols, (uint8_t*)codes, scales,
                                                           bf16_scale);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_pack_nvfp4(const void* w, int rows, int cols, void* codes, void* bscales, float* t, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(t, 0, sizeof(float), st) != cudaSuccess) return -1;
  const size_t n = (size_t)rows * cols;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  k_amax<<<blocks, 256, 0, st>>>((const uint16_t*)w, n, (uint32_t*)t);
  k_tscale<<<1, 1, 0, st>>>(t);
  const size_t nb = (size_t)rows * (cols / 16);
  k_pack_nvfp4<<<(unsigned)((nb + 255) / 256), 256, 0, st>>>((const uint16_t*)w, rows, cols, (uint8_t*)codes,
                                                               (uint8_t*)bscales, t);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_pack_nvfp4_mse(const void* w, int rows, int cols, void* codes, void* bscales, float* t, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(t, 0, sizeof(float), st) != cudaSuccess) return -1;
  const size_t n = (size_t)rows * cols;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  k_amax<<<blocks, 256, 0, st>>>((const uint16_t*)w, n, (uint32_t*)t);
  k_tscale<<<1, 1, 0, st>>>(t);
  const size_t nb = (size_t)rows * (cols / 16);
  k_pack_nvfp4_mse<<<(unsigned)((nb + 127) / 128), 128, 0, st>>>((const uint16_t*)w, rows, cols, (uint8_t*)codes,
                                                                   (uint8_t*)bscales, t);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// One layer's W_o [HID rows][QROWS cols] (canonical packed form) -> the folded O-projection's blocks:
// block (head h, slice s) at dst + (h * FOLD_SLICES + s) * wo_block_bytes(fmt) holds rows
// [FOLD_ROWS s, +FOLD_ROWS) and columns [HD h, +HD): bf16 / FP8 codes row-major; NVFP4 codes
// row-major (HD / 2 bytes a row) followed by the rows' E4M3 block scales (HD / 16 bytes a row).
// One thread per destination byte.
__global__ void k_repack_o(const uint8_t* __restrict__ data, const uint8_t* __restrict__ scale, int fmt,
                           uint8_t* __restrict__ dst) {
  const int bb = wo_block_bytes(fmt);
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)NQH * FOLD_SLICES * bb) return;
  const int blk = (int)(i / bb), o = (int)(i % bb);
  const int h = blk / FOLD_SLICES, s = blk % FOLD_SLICES;
  if (fmt == 2) {
    const int cb = HD / 2;  // code bytes of a block row
    if (o < FOLD_ROWS * cb) {
      const int r = o / cb, c = o % cb;
      dst[i] = data[(size_t)(FOLD_ROWS * s + r) * (QROWS / 2) + (size_t)cb * h + c];
    } else {
      const int o2 = o - FOLD_ROWS * cb, sb = HD / 16;
      const int r = o2 / sb, c = o2 % sb;
      dst[i] = scale[(size_t)(FOLD_ROWS * s + r) * (QROWS / 16) + (size_t)sb * h + c];
    }
  } else {
    const int eb = fmt == 0 ? 2 : 1, rb = HD * eb;  // bytes of a block row
    const int r = o / rb, c = o % rb;
    dst[i] = data[(size_t)(FOLD_ROWS * s + r) * QROWS * eb + (size_t)rb * h + c];
  }
}

int launch_repack_o(const void* data, const void* scale, int fmt, void* dst, void* stream) {
  const long long n = (long long)NQH * FOLD_SLICES * wo_block_bytes(fmt);
  k_repack_o<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream>>>((const uint8_t*)data,
                                                                           (const uint8_t*)scale, fmt, (uint8_t*)dst);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_rope_table(float* cosb, float* sinb, int max_ctx, float theta, void* stream) {
  const int n = max_ctx * (HD / 2);
  k_rope_table<<<(n + 255) / 256, 256, 0, (cudaStream_t)stream>>>(cosb, sinb, max_ctx, (double)theta);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_probe_cvt(uint32_t* a, uint32_t* b, const float* in, int n, uint16_t* e4, uint8_t* e2, void* stream) {
  int total = 65536;
  if (in && n / 2 > total) total = n / 2;
  k_probe_cvt<<<(total + 255) / 256, 256, 0, (cudaStream_t)stream>>>(a, b, in, n, e4, e2);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace mk
