// The batched verify step (see mk_verify.h): k <= 8 tokens at positions pos0 .. pos0 + k - 1 run
// through every layer and the LM head in one persistent launch of 128 CTAs.
//
// Each GEMM step computes Y[row][t] = W[row] . x_t for this CTA's weight rows and the k token
// vectors on the tensor cores: A = the CTA's weight rows (M = 128; rows past the CTA's own are
// never read back), B = the k activation vectors split into a 16-bit high part and a 16-bit low
// part (x = hi + lo to about 2^-16 relative for bf16, 2^-22 for f16; B rows 0..7 and 8..15),
// D = fp32 in tensor memory, Y = D[.][t] + D[.][8 + t]. A producer warp streams the repacked weight
// boxes through a ring of shared-memory slots with bulk copies; one thread issues the MMAs of a
// slot and commits them to the slot's empty barrier, so the slot is refilled as soon as the tensor
// core has read it. Activations cross SMs in sentinel exchange buffers (32-bit values, ready once
// they differ from X_EMPTY), one buffer per layer, step and token. Attention runs one (q head,
// token) pair per CTA with causal masking over the k new positions, whose keys and values each
// unit computes from the exchanged q|k|v; the LM head keeps one argmax per token.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "mk_device.cuh"
#include "mk_tc.cuh"
#include "mk_verify.h"

namespace mk {

// ------------------------------------------------------------------ repack into verify blocks
// One 16-bit operand value of row `row`, column `col` of a canonical packed matrix: bf16 bits
// (to_bf16) or the exact f16 of the FP8 code / NVFP4 code x block scale (the row scale and the
// tensor scale are applied after the GEMM).
__device__ uint16_t v_elem(const DMat& m, int K, int row, int col) {
  if (m.fmt == 0) return reinterpret_cast<const uint16_t*>(m.data)[(size_t)row * K + col];
  float v;
  if (m.fmt == 1) {
    v = e4m3x2_to_f2(m.data[(size_t)row * K + col]).x;
  } else {  // even column in the low nibble
    const float2 pr = e2m1x2_to_f2(m.data[(size_t)row * (K / 2) + col / 2]);
    v = ((col & 1) ? pr.y : pr.x) * e4m3x2_to_f2(m.scale[(size_t)row * (K / 16) + col / 16]).x;
  }
  return __half_as_ushort(__float2half_rn(v));
}

// Row r (0 .. R - 1) of CTA c's rows of step s: the source matrix (which) and its row.
__device__ int v_src_row(int s, int c, int r, int& which) {
  if (s == VS_QKV) {  // q rows to CTAs 0..63, k rows to 64..95, v rows to 96..127, 32 each
    which = c < 64 ? M_Q : (c < 96 ? M_K : M_V);
    const int base = c < 64 ? c : (c < 96 ? c - 64 : c - 96);
    return 32 * base + r;
  }
  if (s == VS_GU) {  // 32 gate rows then the same 32 units' up rows
    which = r < 32 ? M_GATE : M_UP;
    return 32 * c + (r % 32);
  }
  which = s == VS_O ? M_O : M_DOWN;
  return 8 * c + r;
}

// One block (layer step s, CTA c): box b, tile row L = seg * R + r, 16-byte chunk cc holds row r's
// inputs seg * KS + 64 b + 8 cc .. + 7. bf16 matrices are copied bit for bit; FP8 and NVFP4 ones
// become f16 (to_bf16 = 0).
__global__ void k_verify_repack_layer(const DLayer L, int to_bf16, uint8_t* __restrict__ dst) {
  (void)to_bf16;
  const int s = blockIdx.y, c = blockIdx.x;
  const int nbox = v_nbox(s, c);
  if (nbox == 0) return;
  const VStepGeom g = v_step_geom(s);
  const int K = v_cols(s);
  uint8_t* blk = dst + v_block_offset(s, c);
  const int nchunk = nbox * 128 * 8;  // 16-byte chunks of the block
  for (int i = threadIdx.x; i < nchunk; i += blockDim.x) {
    const int bx = i / 1024, rem = i % 1024, tr = rem / 8, cc = rem % 8;
    const int seg = tr / g.R, r = tr % g.R;
    int which;
    const int row = v_src_row(s, c, r, which);
    const DMat& m = L.m[which];
    const int col0 = seg * g.KS + 64 * bx + 8 * cc;
    uint16_t v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = v_elem(m, K, row, col0 + e);
    uint4 w;
    w.x = v[0] | ((uint32_t)v[1] << 16);
    w.y = v[2] | ((uint32_t)v[3] << 16);
    w.z = v[4] | ((uint32_t)v[5] << 16);
    w.w = v[6] | ((uint32_t)v[7] << 16);
    *reinterpret_cast<uint4*>(blk + (size_t)bx * V_BOX + sw128_offset(tr, cc)) = w;
  }
}

__global__ void k_verify_repack_head(const DMat e, int vocab, int to_bf16, uint8_t* __restrict__ dst) {
  (void)to_bf16;
  const int c = blockIdx.x, q = blockIdx.y;
  const int v0 = (int)((long long)vocab * c / V_GRID), v1 = (int)((long long)vocab * (c + 1) / V_GRID);
  const int r0 = v0 + V_HEAD_CHUNK * q;
  const int nr = min(V_HEAD_CHUNK, v1 - r0);
  if (nr <= 0) return;
  const int R8 = (nr + 7) & ~7;
  uint8_t* blk = dst + (size_t)c * v_head_cta_bytes(vocab) + (size_t)q * V_HEAD_CHUNK * HID * 2;
  const int nchunk = R8 * HID / 8;
  for (int i = threadIdx.x; i < nchunk; i += blockDim.x) {
    const int j = i / (R8 * 8), rem = i % (R8 * 8), r = rem / 8, cc = rem % 8;
    uint16_t v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = r < nr ? v_elem(e, HID, r0 + r, 64 * j + 8 * cc + k) : (uint16_t)0;
    uint4 w;
    w.x = v[0] | ((uint32_t)v[1] << 16);
    w.y = v[2] | ((uint32_t)v[3] << 16);
    w.z = v[4] | ((uint32_t)v[5] << 16);
    w.w = v[6] | ((uint32_t)v[7] << 16);
    *reinterpret_cast<uint4*>(blk + (size_t)j * R8 * 128 + sw128_offset(r, cc)) = w;
  }
}

int launch_verify_repack_layer(const DLayer& L, int to_bf16, uint8_t* dst, void* stream) {
  k_verify_repack_layer<<<dim3(V_GRID, VS_COUNT), 256, 0, (cudaStream_t)stream>>>(L, to_bf16, dst);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_verify_repack_head(const DMat& e, int vocab, int to_bf16, uint8_t* dst, void* stream) {
  k_verify_repack_head<<<dim3(V_GRID, v_head_chunks(vocab)), 256, 0, (cudaStream_t)stream>>>(e, vocab, to_bf16, dst);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// ------------------------------------------------------------------ kernel layout
constexpr int V_RING = V_NSLOT * SLOT;  // weight ring (96 KB)
// B operand: KB boxes of N rows x 128 bytes; the largest is down_proj's (3 x 256 rows, 96 KB), the
// LM head's is 16 x 16 rows
__host__ __device__ constexpr int v_xb_bytes(int kb, int n) { return kb * n * 128; }
constexpr int V_XB = v_xb_bytes(3, 256);
static_assert(v_xb_bytes(4, 64) <= V_XB && v_xb_bytes(2, 256) <= V_XB && v_xb_bytes(8, 32) <= V_XB &&
                  v_xb_bytes(HID / 64, VN) <= V_XB,
              "a step's B operand exceeds the staging buffer");
constexpr uint32_t V_TMEM_COLS = 512;  // two accumulators of 128 lanes x N (<= 256) fp32 columns

struct __align__(16) VSmem {
  uint64_t full[V_NSLOT];
  uint64_t empty[V_NSLOT];  // arrived by tcgen05.commit when the MMAs reading the slot completed
  uint64_t done;            // arrived by both issuers' tcgen05.commit when a step's MMAs completed
  uint32_t tmem;            // tensor memory base address
  volatile int flag;         // stays 0: the wait for the MMAs' completion after an abort
  volatile int abort;
  float red[VK][4];         // per-token partial sums of squares (four staging warps a token)
  float inv[VK];            // per-token RMSNorm factors
  float hres[VK][8];        // this CTA's rows of the layer input (o_proj's residual)
  float hres2[VK][8];       // this CTA's rows of h_attn (down_proj's residual)
  float gu[VK][64];         // gate and up outputs before SwiGLU
  float part[128][VK];      // per-segment partial sums of an epilogue (tile row seg * R + r)
  float q[HD];              // attention: the unit's normalised, rotated query
  __align__(16) uint16_t knew[VK][HD];  // keys and values of the new positions (bf16, as cached)
  __align__(16) uint16_t vnew[VK][HD];
  float sc[V_MAXPOS];       // scores, then softmax numerators
  float wo[NCW][HD];        // per-warp attention output partials
  float wst[NCW][2];        // per-warp (max, sum)
  float hb[4][VK];          // LM head: per-warp best logit and index of each token
  int hbi[4][VK];
};
constexpr int V_SMEM_BYTES = 1024 + V_RING + V_XB + (int)sizeof(VSmem);  // 1024: alignment slack
static_assert(V_SMEM_BYTES <= 232448, "verify kernel shared memory exceeds one CTA's budget");

__device__ __forceinline__ uint4 v_ld4(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ bool v_ready(const uint4& v) {
  return v.x != X_EMPTY && v.y != X_EMPTY && v.z != X_EMPTY && v.w != X_EMPTY;
}
// Sentinel exchange words of layer l, token t (see V_XL): q|k|v, attention output, h_attn, SwiGLU
// output, layer output.
__device__ __forceinline__ uint32_t* vx(const VParams& p, int l, int t) { return p.x + ((size_t)l * VK + t) * V_XL; }
constexpr int VX_QKV = 0, VX_ATT = QKV_ROWS, VX_HA = QKV_ROWS + QROWS, VX_ACT = VX_HA + HID, VX_H = VX_ACT + FFN;

// Boxes (64 input columns, R8 rows) of one GEMM step of this CTA and how they fill ring slots.
struct VGeom {
  int R8, nbox, bps;  // rows, boxes, boxes per slot
  __device__ int slots() const { return (nbox + bps - 1) / bps; }
};
__device__ __forceinline__ VGeom v_geom(int R8, int K) {
  VGeom g;
  g.R8 = R8;
  g.nbox = K / 64;
  g.bps = SLOT / (R8 * 128);
  return g;
}

// Bounded wait on an mbarrier phase; false on abort or timeout (the caller reports it).
__device__ bool v_wait(uint64_t* b, uint32_t par, volatile int* abort, unsigned long long timeout_ns) {
  if (mbar_test_wait(b, par)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(b, par)) {
    if (*abort) return false;
    if (globaltimer() - t0 > timeout_ns) return false;
  }
  return true;
}

// Record a failure (first one wins) and tell every CTA to stop. Consumer threads also raise this
// CTA's abort flag, which the consumers read only right after a CTA barrier, so they all take the
// same path; the producer warp leaves the flag alone (it runs outside those barriers).
__device__ void v_fail_global(const VParams& p, uint32_t code, uint32_t detail) {
  if (atomicCAS(&p.sync->status[0], 0u, code) == 0u) st_relaxed_u32(&p.sync->status[1], detail);
  st_relaxed_u32(&p.sync->status[2], 1u);
}
__device__ void v_fail(const VParams& p, VSmem* s, uint32_t code, uint32_t detail) {
  v_fail_global(p, code, detail);
  s->abort = 1;
}

// ------------------------------------------------------------------ producer
// Streams this CTA's boxes of every step of every layer, then of its LM-head chunks, in the order
// the MMA issuer consumes them (a run of up to bps boxes per slot, one bulk copy each).
__device__ void v_producer(const VParams& p, VSmem* s, uint8_t* ring) {
  const int c = blockIdx.x;
  const uint64_t pol = l2_evict_first_policy();
  uint32_t n = 0;
  auto issue = [&](const uint8_t* src, uint32_t bytes) -> bool {
    const uint32_t slot = n % V_NSLOT;
    if (n >= V_NSLOT && !v_wait(&s->empty[slot], ((n / V_NSLOT) - 1) & 1, &s->abort, p.timeout_ns)) {
      if (!s->abort) v_fail_global(p, 3u, (uint32_t)PH_WAIT | ((uint32_t)c << 16) | 0x80000000u);
      return false;
    }
    mbar_expect_tx(&s->full[slot], bytes);
    bulk_g2s(ring + (size_t)slot * SLOT, src, bytes, &s->full[slot], pol);
    ++n;
    return true;
  };
  bool ok = true;
  for (int l = 0; l < p.n_layers && ok; ++l) {
    for (int st = 0; st < VS_COUNT && ok; ++st) {
      const uint8_t* blk = p.vw + (size_t)l * v_layer_bytes() + v_block_offset(st, c);
      for (int j = 0; j < v_nbox(st, c) && ok; ++j) ok = issue(blk + (size_t)j * V_BOX, (uint32_t)V_BOX);
    }
  }
  const int v0 = (int)((long long)p.vocab * c / V_GRID), v1 = (int)((long long)p.vocab * (c + 1) / V_GRID);
  for (int q = 0; ok && v0 + V_HEAD_CHUNK * q < v1; ++q) {
    const int nr = min(V_HEAD_CHUNK, v1 - v0 - V_HEAD_CHUNK * q), R8 = (nr + 7) & ~7;
    const uint8_t* blk = p.vhead + (size_t)c * v_head_cta_bytes(p.vocab) + (size_t)q * V_HEAD_CHUNK * HID * 2;
    const VGeom g = v_geom(R8, HID);  // the same runs of boxes the MMA issuer expects
    for (int j = 0; j < g.nbox && ok; j += g.bps)
      ok = issue(blk + (size_t)j * R8 * 128, (uint32_t)(min(g.bps, g.nbox - j) * R8 * 128));
  }
  // every copy issued has landed before the producer leaves (after an abort the consumers may have
  // stopped waiting for them); a copy still in flight after 200 ms is recorded in status word 3
  for (uint32_t i = n > V_NSLOT ? n - V_NSLOT : 0; i < n; ++i) {
    const uint64_t t0 = globaltimer();
    while (!mbar_test_wait(&s->full[i % V_NSLOT], (i / V_NSLOT) & 1)) {
      if (globaltimer() - t0 > 200000000ull) {
        st_relaxed_u32(&p.sync->status[3], 1u);
        return;
      }
    }
  }
}

// ------------------------------------------------------------------ consumers
// 16-bit high and low parts of x (bf16 or f16): x - hi is exact in fp32 and lo rounds it.
// Two elements at once (packed conversions, the same roundings): hw and lw hold the high and low
// parts of a in their low halves and of b in their high halves.
__device__ __forceinline__ void v_split2(float a, float b, int ab_bf16, uint32_t& hw, uint32_t& lw) {
  if (ab_bf16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
    hw = *reinterpret_cast<const uint32_t*>(&h);
    lw = *reinterpret_cast<const uint32_t*>(&l);
  } else {
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
    hw = *reinterpret_cast<const uint32_t*>(&h);
    lw = *reinterpret_cast<const uint32_t*>(&l);
  }
}

struct VCons {
  const VParams* P;
  VSmem* s;
  uint8_t* ring;
  uint8_t* xb;
  int tid, lane, warp;
  uint32_t n;      // ring slots consumed
  uint32_t ndone;  // GEMM steps completed (parity of `done`)
  bool acc2;       // the last GEMM step used the second accumulator

  // Stage the k input vectors of a GEMM step into the B operand of a step with segments of KS inputs
  // and N rows: input e of token t, in segment seg = e / KS, goes to box (e % KS) / 64, high part in
  // row 16 seg + t, low part in row 16 seg + 8 + t. The inputs are the sentinel words at
  // vx(l, t) + xoff (embed: the embedding rows of the tokens instead); w (normed inputs,
  // K == HID): the bf16 norm weights, multiplied in, and each token's sum of squares left in
  // red[t][0..3]; res (optional): elements [8 res_chunk, +8) of each token saved un-normed.
  __device__ void stage(int l, int xoff, int K, const uint16_t* w, float (*res)[8], int res_chunk, int ab_bf16,
                        bool embed, int KS, int N) {
    const VParams& p = *P;
    const int cpt = K / 8, total = p.k * cpt;  // 8-element chunks per token, in all
    constexpr int BATCH = 4;
    for (int i0 = 0; i0 < total; i0 += BATCH * NCT) {
      uint4 a[BATCH], b[BATCH];
      int tt[BATCH], ch[BATCH];
#pragma unroll
      for (int m = 0; m < BATCH; ++m) {
        const int i = i0 + m * NCT + tid;
        tt[m] = i < total ? i / cpt : -1;
        ch[m] = i % cpt;
        if (tt[m] >= 0 && !embed) {
          const uint32_t* src = vx(p, l, tt[m]) + xoff + 8 * ch[m];
          a[m] = v_ld4(src);
          b[m] = v_ld4(src + 4);
        }
      }
      if (!embed) {  // poll the words that were still empty
        const uint64_t t0 = globaltimer();
        uint32_t it = 0;
        while (true) {
          bool ready = true;
#pragma unroll
          for (int m = 0; m < BATCH; ++m) {
            if (tt[m] >= 0 && !(v_ready(a[m]) && v_ready(b[m]))) {
              const uint32_t* src = vx(p, l, tt[m]) + xoff + 8 * ch[m];
              a[m] = v_ld4(src);
              b[m] = v_ld4(src + 4);
              ready = ready && v_ready(a[m]) && v_ready(b[m]);
            }
          }
          if (ready || s->abort) break;  // after an abort the operand is garbage and never used
          if ((++it & 255u) == 0u && ld_relaxed_u32(&p.sync->status[2]) != 0u) {
            s->abort = 1;
            break;
          }
          if (globaltimer() - t0 > p.timeout_ns) {
            v_fail(p, s, 3u, (uint32_t)(PH_WAIT | (l << 8) | (blockIdx.x << 16)));
            break;
          }
        }
      }
#pragma unroll
      for (int m = 0; m < BATCH; ++m) {
        const int t = tt[m];
        float v[8];
        if (t >= 0) {
          const int e0 = 8 * ch[m];
          if (embed) {
            const int tok = p.tokens[t];
            if (p.embed.fmt == 0) {
              const uint4 q = __ldg(reinterpret_cast<const uint4*>(p.embed.data + ((size_t)tok * HID + e0) * 2));
              const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                v[2 * e] = __uint_as_float(qq[e] << 16);
                v[2 * e + 1] = __uint_as_float(qq[e] & 0xFFFF0000u);
              }
            } else {
              const float sc = __ldg(reinterpret_cast<const float*>(p.embed.scale) + tok);
              const uint2 q = __ldg(reinterpret_cast<const uint2*>(p.embed.data + (size_t)tok * HID + e0));
              const uint32_t qq[2] = {q.x, q.y};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = e4m3x2_to_f2((qq[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
                v[2 * e] = f.x * sc;
                v[2 * e + 1] = f.y * sc;
              }
            }
          } else {
            v[0] = __uint_as_float(a[m].x), v[1] = __uint_as_float(a[m].y);
            v[2] = __uint_as_float(a[m].z), v[3] = __uint_as_float(a[m].w);
            v[4] = __uint_as_float(b[m].x), v[5] = __uint_as_float(b[m].y);
            v[6] = __uint_as_float(b[m].z), v[7] = __uint_as_float(b[m].w);
          }
          if (res && ch[m] == res_chunk) {
#pragma unroll
            for (int e = 0; e < 8; ++e) res[t][e] = v[e];
          }
          float ss = 0.f;
          if (w) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              ss = fmaf(v[e], v[e], ss);
              v[e] *= __uint_as_float((uint32_t)__ldg(w + e0 + e) << 16);
            }
          }
          uint4 H, L;
          v_split2(v[0], v[1], ab_bf16, H.x, L.x);
          v_split2(v[2], v[3], ab_bf16, H.y, L.y);
          v_split2(v[4], v[5], ab_bf16, H.z, L.z);
          v_split2(v[6], v[7], ab_bf16, H.w, L.w);
          const int seg = e0 / KS, j = e0 - seg * KS, n0 = VN * seg;
          uint8_t* box = xb + (size_t)(j / 64) * (N * 128);
          if (mk_in_bounds((j / 64 + 1) * N * 128 <= V_XB && n0 + VN <= N && t < VK, p.sync->status, 11,
                           (uint32_t)e0)) {
            *reinterpret_cast<uint4*>(box + sw128_offset(n0 + t, (j % 64) / 8)) = H;
            *reinterpret_cast<uint4*>(box + sw128_offset(n0 + 8 + t, (j % 64) / 8)) = L;
          }
          if (w) {  // a warp's 32 chunks of a round belong to one token (cpt is a multiple of 32)
#pragma unroll
            for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) s->red[t][(ch[m] / 32) & 3] = ss;
          }
        }
      }
    }
    fence_proxy_async_smem();  // the staged operand, visible to the tensor core
  }
  // 1 / rms of token t's staged input (HID elements), the partial sums in a fixed order.
  __device__ __forceinline__ float inv_rms(int t) const {
    const float tot = ((s->red[t][0] + s->red[t][1]) + s->red[t][2]) + s->red[t][3];
    return rsqrtf(tot * (1.0f / (float)HID) + P->eps);
  }

  // The MMAs of one GEMM step: D[row][n] = sum over the step's boxes of A (ring slots) x B (xb, boxes
  // of N rows). One thread issuing MMAs sets the pace (each costs it tens of cycles whatever its
  // size), so two issue them: thread 0 the even ring slots of the step into accumulator 0 (tensor
  // memory columns 0 .. N - 1), thread 32 the odd ones into accumulator 1 (columns N .. 2N - 1).
  // Each commits its slots to their empty barriers, so a slot is refilled as soon as the tensor
  // core has read it, and finally commits `done` (two arrivals); every thread then waits for it.
  // The epilogue adds the two accumulators (read_seg). Returns false after an abort.
  __device__ bool mma_step(VGeom g, int N, uint32_t idesc, int phase, int layer) {
    const VParams& p = *P;
    const int nslots = g.slots();
    acc2 = nslots > 1;
    bar_consumers(NCT);  // the staged operand and the previous step's tensor-memory reads
    if (tid == 0 || tid == 32) {
      const int who = tid >> 5;
      tc_fence_after();
      const uint32_t xbase = smem_u32(xb), d = s->tmem + (uint32_t)(who * N);
      bool first = true;
      for (int sl = who; sl < nslots; sl += 2) {
        const uint32_t m = n + (uint32_t)sl, slot = m % V_NSLOT, par = (m / V_NSLOT) & 1;
        if (s->abort) break;
        if (!v_wait(&s->full[slot], par, &s->abort, p.timeout_ns)) {
          if (!s->abort) v_fail(p, s, 3u, (uint32_t)(phase | (layer << 8) | (blockIdx.x << 16)) | 0x80000000u);
          break;
        }
        const uint32_t sbase = smem_u32(ring + (size_t)slot * SLOT);
        const int j0 = sl * g.bps;  // the slot's first box
        // the MMA reads 128 rows (16 KB) from a box's start, which end inside the ring and xb, and
        // N rows of each B box
        if (!mk_in_bounds(slot < V_NSLOT && (slot + 1) * SLOT + (g.bps - 1) * g.R8 * 128 <= V_RING + V_XB - 16384 + SLOT &&
                              (min(g.nbox, j0 + g.bps)) * N * 128 <= V_XB,
                          p.sync->status, 14, slot))
          break;
        for (int b = 0, j = j0; b < g.bps && j < g.nbox; ++b, ++j) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            umma_f16(d, umma_desc_sw128(sbase + (uint32_t)(b * g.R8 * 128 + 32 * kk)),
                     umma_desc_sw128(xbase + (uint32_t)(j * N * 128 + 32 * kk)), idesc, first ? 0u : 1u);
            first = false;
          }
        }
        umma_commit(&s->empty[slot]);
      }
      umma_commit(&s->done);  // also after an abort: the issued MMAs finish before the CTA exits
    }
    n += (uint32_t)nslots;
    // every thread waits for the MMAs (they were committed even after an abort, so they end first)
    const bool ok = v_wait(&s->done, ndone & 1, &s->abort, p.timeout_ns) || v_wait(&s->done, ndone & 1, &s->flag, p.timeout_ns);
    ++ndone;
    tc_fence_after();
    if (!ok) v_fail(p, s, 3u, (uint32_t)(phase | (layer << 8) | (blockIdx.x << 16)) | 0x40000000u);
    bar_consumers(NCT);  // every consumer thread is past its writes of the abort flag
    return s->abort == 0;
  }
  // This thread's accumulator row (warps 0..3: tensor-memory lane L = 32 warp + lane, tile row
  // seg * R + r with seg = L / R) on its own segment's diagonal block, both accumulators added
  // (the second only where the step had more than one ring slot): y[t] = D[L][16 seg + t] +
  // D[L][16 seg + 8 + t] (high and low parts). A warp's lanes may lie in several segments (R < 32):
  // the warp loads each of their column blocks and every lane keeps its own.
  __device__ void read_seg(int R, int N, float* y) {
    const int L = 32 * warp + lane, seg = L / R;
    const int s0 = (32 * warp) / R, s1 = (32 * warp + 31) / R;
    const uint32_t base = s->tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll
    for (int t = 0; t < VK; ++t) y[t] = 0.f;
    for (int sg = s0; sg <= s1; ++sg) {  // warp-uniform; per token: hi0 + lo0, then + hi1, + lo1
      uint32_t r0[8], r1[8], r2[8], r3[8];
      tmem_ld8_issue(base + (uint32_t)(VN * sg), r0);  // the segment's loads in flight together
      tmem_ld8_issue(base + (uint32_t)(VN * sg + 8), r1);
      if (acc2) {
        tmem_ld8_issue(base + (uint32_t)(N + VN * sg), r2);
        tmem_ld8_issue(base + (uint32_t)(N + VN * sg + 8), r3);
      }
      tmem_wait_ld8(r0);
      tmem_wait_ld8(r1);
      if (acc2) {
        tmem_wait_ld8(r2);
        tmem_wait_ld8(r3);
      }
      float h[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) h[t] = __uint_as_float(r0[t]) + __uint_as_float(r1[t]);
      if (acc2) {
#pragma unroll
        for (int t = 0; t < 8; ++t) h[t] = (h[t] + __uint_as_float(r2[t])) + __uint_as_float(r3[t]);
      }
      if (sg == seg) {
#pragma unroll
        for (int t = 0; t < VK; ++t) y[t] = h[t];
      }
    }
    tc_fence_before();
  }
  // Warps 0..3: this thread's diagonal-block row into part[L] (see read_seg).
  __device__ void read_part(int R, int N) {
    float y[VK];
    read_seg(R, N, y);
#pragma unroll
    for (int t = 0; t < VK; ++t) s->part[32 * warp + lane][t] = y[t];
  }
  // Row r's result for token t: its segments' partial sums added in segment order.
  __device__ __forceinline__ float seg_sum(int R, int S, int r, int t) const {
    float a = s->part[r][t];
    for (int sg = 1; sg < S; ++sg) a += s->part[sg * R + r][t];
    return a;
  }
  // Row scale of a canonical matrix after the 16-bit GEMM: FP8 row scale, NVFP4 tensor scale, 1.
  __device__ __forceinline__ float row_scale(const DMat& m, int row) const {
    return m.fmt == 1 ? __ldg(reinterpret_cast<const float*>(m.scale) + row) : (m.fmt == 2 ? m.tscale : 1.f);
  }
};

// ------------------------------------------------------------------ attention unit
// CTA b < 16 k attends for q head b % 16 and token t = b / 16 over positions 0 .. pos0 + t: the cached
// ones from the KV cache, the new ones pos0 .. pos0 + t from the keys and values the unit computes
// itself from the exchanged q|k|v (QK-norm, RoPE at their positions, bf16 as cached). The unit of
// the first q head of a KV head also writes token t's key and value to the cache.
__device__ bool v_attention(VCons& C, int l) {
  const VParams& p = *C.P;
  VSmem* s = C.s;
  const int h = blockIdx.x % NQH, t = blockIdx.x / NQH, g = h / GQA;
  const DLayer& L = p.layers[l];
  const int lane = C.lane, warp = C.warp;
  // vector vi: 0 = q of token t, 1 .. t + 1 = k of token vi - 1, t + 2 .. 2 t + 2 = v of token vi - t - 2
  for (int vi = warp; vi < 2 * t + 3; vi += NCW) {
    const bool isq = vi == 0, isk = vi >= 1 && vi <= t + 1;
    const int tok = isq ? t : (isk ? vi - 1 : vi - t - 2);
    const int off = isq ? h * HD : (isk ? QROWS + g * HD : QROWS + KVROWS + g * HD);
    const uint32_t* src = vx(p, l, tok) + VX_QKV + off;
    uint32_t wv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) wv[j] = ld_relaxed_u32(src + lane + 32 * j);
    const uint64_t t0 = globaltimer();
    while (wv[0] == X_EMPTY || wv[1] == X_EMPTY || wv[2] == X_EMPTY || wv[3] == X_EMPTY) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (wv[j] == X_EMPTY) wv[j] = ld_relaxed_u32(src + lane + 32 * j);
      if (s->abort) break;
      if (globaltimer() - t0 > p.timeout_ns) {
        v_fail(p, s, 3u, (uint32_t)(PH_ATTN | (l << 8) | (blockIdx.x << 16)));
        break;
      }
    }
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = __uint_as_float(wv[j]);
    if (isq || isk) {  // QK-norm over the head, then RoPE at the token's position
      const uint16_t* nw = isq ? L.q_norm : L.k_norm;
      float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
#pragma unroll
      for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float inv = 1.0f / sqrtf(ss / (float)HD + p.eps);
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = v[j] * inv * __uint_as_float((uint32_t)__ldg(nw + lane + 32 * j) << 16);
      const int pos = p.pos0 + tok;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float cs = __ldg(p.rope_cos + (size_t)pos * (HD / 2) + lane + 32 * j);
        const float sn = __ldg(p.rope_sin + (size_t)pos * (HD / 2) + lane + 32 * j);
        const float a = v[j], b = v[j + 2];
        v[j] = a * cs - b * sn;
        v[j + 2] = b * cs + a * sn;
      }
    }
    if (isq) {
#pragma unroll
      for (int j = 0; j < 4; ++j) s->q[lane + 32 * j] = v[j];
    } else {
      uint16_t* dst = isk ? s->knew[tok] : s->vnew[tok];
      uint16_t* cache = isk ? p.kc : p.vc;
      const size_t row = (((size_t)l * NKVH + g) * p.max_ctx + p.pos0 + tok) * HD;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint16_t bits = __bfloat16_as_ushort(__float2bfloat16_rn(v[j]));
        dst[lane + 32 * j] = bits;
        if (h % GQA == 0 && tok == t && mk_in_bounds(p.pos0 + tok < p.max_ctx, p.sync->status, 13, (uint32_t)tok))
          cache[row + lane + 32 * j] = bits;
      }
    }
  }
  bar_consumers(NCT);
  if (s->abort) return false;
  const int np = p.pos0 + t + 1;  // positions attended
  const int per = (np + NCW - 1) / NCW;
  const int ws0 = min(np, warp * per), ws1 = min(np, ws0 + per);
  const float scale = 0.08838834764831845f;  // 1 / sqrt(128)
  const uint16_t* kbase = p.kc + ((size_t)l * NKVH + g) * p.max_ctx * HD;
  const uint16_t* vbase = p.vc + ((size_t)l * NKVH + g) * p.max_ctx * HD;
  // scores: eight lanes a position (16 dimensions each), four positions a pass
  const int gp = lane >> 3, sl = lane & 7;
  float qr[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) qr[j] = s->q[16 * sl + j];
  float m = -INFINITY;
  for (int b0 = ws0; b0 < ws1; b0 += 4) {
    const int pp = b0 + gp;
    float a = 0.f;
    if (pp < ws1) {
      const uint16_t* row = pp < p.pos0 ? kbase + (size_t)pp * HD : s->knew[pp - p.pos0];
      uint4 k0, k1;
      if (pp < p.pos0) {
        k0 = __ldg(reinterpret_cast<const uint4*>(row + 16 * sl));
        k1 = __ldg(reinterpret_cast<const uint4*>(row + 16 * sl + 8));
      } else {
        k0 = *reinterpret_cast<const uint4*>(row + 16 * sl);
        k1 = *reinterpret_cast<const uint4*>(row + 16 * sl + 8);
      }
      const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        a = fmaf(qr[2 * e], __uint_as_float(kw[e] << 16), a);
        a = fmaf(qr[2 * e + 1], __uint_as_float(kw[e] & 0xFFFF0000u), a);
      }
    }
#pragma unroll
    for (int o = 4; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (pp < ws1 && mk_in_bounds(pp < V_MAXPOS, p.sync->status, 12, (uint32_t)pp)) {
      a *= scale;
      if (sl == 0) s->sc[pp] = a;
      m = fmaxf(m, a);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __syncwarp();
  float lsum = 0.f;
  for (int pp = ws0 + lane; pp < ws1; pp += 32) {
    const float e = expf(s->sc[pp] - m);
    s->sc[pp] = e;
    lsum += e;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
  __syncwarp();
  float o4[4] = {0.f, 0.f, 0.f, 0.f};
  for (int pp = ws0; pp < ws1; ++pp) {
    uint2 vw;
    if (pp < p.pos0) vw = __ldg(reinterpret_cast<const uint2*>(vbase + (size_t)pp * HD + 4 * lane));
    else vw = *reinterpret_cast<const uint2*>(s->vnew[pp - p.pos0] + 4 * lane);
    const float pr = s->sc[pp];
    o4[0] = fmaf(pr, __uint_as_float(vw.x << 16), o4[0]);
    o4[1] = fmaf(pr, __uint_as_float(vw.x & 0xFFFF0000u), o4[1]);
    o4[2] = fmaf(pr, __uint_as_float(vw.y << 16), o4[2]);
    o4[3] = fmaf(pr, __uint_as_float(vw.y & 0xFFFF0000u), o4[3]);
  }
  *reinterpret_cast<float4*>(&s->wo[warp][4 * lane]) = make_float4(o4[0], o4[1], o4[2], o4[3]);
  if (lane == 0) {
    s->wst[warp][0] = m;
    s->wst[warp][1] = lsum;
  }
  bar_consumers(NCT);
  if (C.tid < HD) {  // merge the warps (an empty slice has max -inf and sum 0: weight 0)
    const int d = C.tid;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NCW; ++w) M = fmaxf(M, s->wst[w][0]);
    float ls = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) {
      const float f = expf(s->wst[w][0] - M);
      ls = fmaf(f, s->wst[w][1], ls);
      acc = fmaf(f, s->wo[w][d], acc);
    }
    st_relaxed_u32(vx(p, l, t) + VX_ATT + h * HD + d, __float_as_uint(acc / ls));
  }
  return true;
}

// ------------------------------------------------------------------ the launch
__device__ void v_run(VCons& C) {
  const VParams& p = *C.P;
  VSmem* s = C.s;
  const int c = blockIdx.x, tid = C.tid, lane = C.lane, warp = C.warp;
  for (int t = 0; t < p.k; ++t) {  // an invalid token ends the launch in every CTA alike
    const int tok = p.tokens[t];
    if ((unsigned)tok >= (unsigned)p.vocab) {
      if (tid == 0) v_fail(p, s, 4u, (uint32_t)c << 16);
      bar_consumers(NCT);
      return;
    }
  }
  const VStepGeom gq = v_step_geom(VS_QKV), go = v_step_geom(VS_O), gg = v_step_geom(VS_GU), gd = v_step_geom(VS_DOWN);
  const uint32_t id_q = umma_idesc_f16(p.layer_bf16, gq.N), id_o = umma_idesc_f16(p.layer_bf16, go.N);
  const uint32_t id_g = umma_idesc_f16(p.layer_bf16, gg.N), id_d = umma_idesc_f16(p.layer_bf16, gd.N);
  const uint32_t id_h = umma_idesc_f16(p.head_bf16, VN);
  const bool epi = warp < 4;         // warps 0..3 read the accumulator (tensor-memory lane quarters)
  const int row = 32 * warp + lane;  // this thread's accumulator row
  const bool gu_cta = c < V_GU_CTAS;
  float y[VK];
  for (int l = 0; l < p.n_layers; ++l) {
    const DLayer& L = p.layers[l];
    // ---- q|k|v: this CTA's 32 rows (CTA c writes q|k|v elements 32 c .. 32 c + 31)
    C.stage(l == 0 ? 0 : l - 1, VX_H, HID, L.ln_in, s->hres, c, p.layer_bf16, l == 0, gq.KS, gq.N);
    if (!C.mma_step(v_geom(128, gq.KS), gq.N, id_q, PH_QKV, l)) return;
    if (epi) C.read_part(gq.R, gq.N);
    bar_consumers(NCT);
    for (int i = tid; i < gq.R * p.k; i += NCT) {
      const int r = i % gq.R, t = i / gq.R;
      const int which = c < 64 ? M_Q : (c < 96 ? M_K : M_V);
      const int mrow = 32 * (c < 64 ? c : (c < 96 ? c - 64 : c - 96)) + r;
      const float v = C.seg_sum(gq.R, gq.S, r, t) * C.row_scale(L.m[which], mrow) * C.inv_rms(t);
      st_relaxed_u32(vx(p, l, t) + VX_QKV + 32 * c + r, __float_as_uint(v));
    }
    // ---- attention, one (q head, token) pair per CTA
    if (c < NQH * p.k && !v_attention(C, l)) return;
    // ---- o_proj: rows 8 c .. 8 c + 7, plus the residual
    C.stage(l, VX_ATT, QROWS, nullptr, nullptr, -1, p.layer_bf16, false, go.KS, go.N);
    if (!C.mma_step(v_geom(128, go.KS), go.N, id_o, PH_O, l)) return;
    if (epi) C.read_part(go.R, go.N);
    bar_consumers(NCT);
    for (int i = tid; i < go.R * p.k; i += NCT) {
      const int r = i % go.R, t = i / go.R;
      const float v = s->hres[t][r] + C.seg_sum(go.R, go.S, r, t) * C.row_scale(L.m[M_O], 8 * c + r);
      st_relaxed_u32(vx(p, l, t) + VX_HA + 8 * c + r, __float_as_uint(v));
    }
    // ---- gate/up (CTAs 0..95): FFN units 32 c .. 32 c + 31 (rows 0..31 gate, 32..63 up), SwiGLU;
    // every CTA stages (its rows of h_attn are down_proj's residual)
    C.stage(l, VX_HA, HID, L.ln_post, s->hres2, c, p.layer_bf16, false, gg.KS, gg.N);
    if (gu_cta) {
      if (!C.mma_step(v_geom(128, gg.KS), gg.N, id_g, PH_GATEUP, l)) return;
      if (epi) C.read_part(gg.R, gg.N);
    }
    bar_consumers(NCT);
    for (int i = tid; gu_cta && i < gg.R * p.k; i += NCT) {
      const int r = i % gg.R, t = i / gg.R;
      const float sc = C.row_scale(L.m[r < 32 ? M_GATE : M_UP], 32 * c + (r % 32));
      s->gu[t][r] = C.seg_sum(gg.R, gg.S, r, t) * sc * C.inv_rms(t);
    }
    bar_consumers(NCT);
    for (int i = tid; gu_cta && i < 32 * p.k; i += NCT) {
      const int u = i % 32, t = i / 32;
      const float gt = s->gu[t][u], up = s->gu[t][32 + u];
      st_relaxed_u32(vx(p, l, t) + VX_ACT + 32 * c + u, __float_as_uint(gt / (1.0f + expf(-gt)) * up));
    }
    // ---- down_proj: rows 8 c .. 8 c + 7, plus the residual
    C.stage(l, VX_ACT, FFN, nullptr, nullptr, -1, p.layer_bf16, false, gd.KS, gd.N);
    if (!C.mma_step(v_geom(128, gd.KS), gd.N, id_d, PH_DOWN, l)) return;
    if (epi) C.read_part(gd.R, gd.N);
    bar_consumers(NCT);
    for (int i = tid; i < gd.R * p.k; i += NCT) {
      const int r = i % gd.R, t = i / gd.R;
      const float v = s->hres2[t][r] + C.seg_sum(gd.R, gd.S, r, t) * C.row_scale(L.m[M_DOWN], 8 * c + r);
      st_relaxed_u32(vx(p, l, t) + VX_H + 8 * c + r, __float_as_uint(v));
    }
  }
  // ---- final RMSNorm + LM head in chunks of 128 rows, one running argmax per token
  C.stage(p.n_layers - 1, VX_H, HID, p.final_norm, nullptr, -1, p.head_bf16, false, HID, VN);
  float best[VK];
  int besti[VK];
#pragma unroll
  for (int t = 0; t < VK; ++t) best[t] = -INFINITY, besti[t] = 0x7FFFFFFF;
  const int v0 = (int)((long long)p.vocab * c / V_GRID), v1 = (int)((long long)p.vocab * (c + 1) / V_GRID);
  for (int q = 0; v0 + V_HEAD_CHUNK * q < v1; ++q) {
    const int r0 = v0 + V_HEAD_CHUNK * q, nr = min(V_HEAD_CHUNK, v1 - r0);
    if (!C.mma_step(v_geom((nr + 7) & ~7, HID), VN, id_h, PH_HEAD, p.n_layers)) return;
    if (epi) {
      C.read_seg(128, VN, y);
      if (row < nr) {
        const int r = r0 + row;
        const float sc = C.row_scale(p.embed, r);
#pragma unroll
        for (int t = 0; t < VK; ++t) {
          if (t < p.k) {
            const float lg = y[t] * sc * C.inv_rms(t);
            if (p.logits) p.logits[(size_t)t * p.vocab + r] = lg;
            if (lg > best[t] || (lg == best[t] && r < besti[t])) best[t] = lg, besti[t] = r;
          }
        }
      }
    }
  }
  // CTA argmax per token (lowest index among equal maxima), then the grid's through one 64-bit
  // atomicMax key per token; the last CTA to finish publishes the tokens and resets the keys
  if (epi) {
#pragma unroll
    for (int t = 0; t < VK; ++t) {
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best[t], o);
        const int oi = __shfl_xor_sync(0xffffffffu, besti[t], o);
        if (ob > best[t] || (ob == best[t] && oi < besti[t])) best[t] = ob, besti[t] = oi;
      }
      if (lane == 0) s->hb[warp][t] = best[t], s->hbi[warp][t] = besti[t];
    }
  }
  bar_consumers(NCT);
  if (tid == 0) {
    for (int t = 0; t < p.k; ++t) {
      float b = s->hb[0][t];
      int bi = s->hbi[0][t];
      for (int w = 1; w < 4; ++w)
        if (s->hb[w][t] > b || (s->hb[w][t] == b && s->hbi[w][t] < bi)) b = s->hb[w][t], bi = s->hbi[w][t];
      if (bi == 0x7FFFFFFF) continue;  // a CTA without LM-head rows
      const uint32_t u = __float_as_uint(b);
      const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
      atomicMax(&p.sync->key[t], ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)bi));
    }
    fence_acqrel_gpu();
    const uint32_t old = atom_acqrel_add(&p.sync->c[PH_HEAD][0], 1u);
    if (old == (uint32_t)(gridDim.x - 1)) {
      for (int t = 0; t < p.k; ++t) {
        const unsigned long long kk = ld_relaxed_u64(&p.sync->key[t]);
        p.next_out[t] = (int32_t)(0xFFFFFFFFu - (uint32_t)(kk & 0xFFFFFFFFull));
        st_relaxed_u64(&p.sync->key[t], 0ull);
      }
      st_relaxed_u32(&p.sync->c[PH_HEAD][0], 0u);
    }
  }
}

__global__ void __launch_bounds__(NTHREADS, 1) k_verify(const VParams p) {
  extern __shared__ uint8_t vsm_raw[];
  uint8_t* base = vsm_raw + ((1024u - (smem_u32(vsm_raw) & 1023u)) & 1023u);  // 1024-byte aligned
  uint8_t* ring = base;
  uint8_t* xb = base + V_RING;
  VSmem* s = reinterpret_cast<VSmem*>(base + V_RING + V_XB);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    for (int i = 0; i < V_NSLOT; ++i) {
      mbar_init(&s->full[i], 1);
      mbar_init(&s->empty[i], 1);
    }
    mbar_init(&s->done, 2);  // one arrival per MMA issuer
    s->abort = 0;
    s->flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&s->tmem, V_TMEM_COLS);
    tmem_relinquish();
  }
  {  // the next launch's exchange set starts empty (this launch uses the other one)
    uint4* x4 = reinterpret_cast<uint4*>(p.x_reset);
    const uint4 e4 = make_uint4(X_EMPTY, X_EMPTY, X_EMPTY, X_EMPTY);
    const size_t n4 = v_x_words(p.n_layers) / 4;
    for (size_t i = (size_t)blockIdx.x * NTHREADS + tid; i < n4; i += (size_t)gridDim.x * NTHREADS) x4[i] = e4;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid >= NCT) {
    if (tid == NCT) v_producer(p, s, ring);
    return;
  }
  VCons C;
  C.P = &p;
  C.s = s;
  C.ring = ring;
  C.xb = xb;
  C.tid = tid;
  C.lane = tid & 31;
  C.warp = warp;
  C.n = 0;
  C.ndone = 0;
  v_run(C);
  tc_fence_before();
  bar_consumers(NCT);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(s->tmem, V_TMEM_COLS);
  }
}

int verify_smem_bytes() { return V_SMEM_BYTES; }

static bool g_vattr[64] = {};
int launch_verify(const VParams& p, void* stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  if (!g_vattr[dev]) {
    if (cudaFuncSetAttribute(k_verify, cudaFuncAttributeMaxDynamicSharedMemorySize, V_SMEM_BYTES) != cudaSuccess)
      return -1;
    g_vattr[dev] = true;
  }
  void* args[] = {(void*)&p};
  return cudaLaunchCooperativeKernel((const void*)k_verify, dim3(V_GRID), dim3(NTHREADS), args, V_SMEM_BYTES,
                                     (cudaStream_t)stream) == cudaSuccess
             ? 0
             : -1;
}

}  // namespace mk
