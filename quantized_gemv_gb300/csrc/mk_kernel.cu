// The decode megakernel: one persistent cooperative launch runs every layer of a
// Qwen3-0.6B-shaped decoder and the LM-head argmax, producing one token.
//
// Structure (per CTA, one CTA per SM):
//   * a producer warp streams this CTA's weight rows (and, for attention units, its slice of the
//     bf16 KV cache) with cp.async.bulk into an 11-slot shared-memory ring. Weights do not depend
//     on the token, so the stream runs ahead across every wait ("productive spin", monolith page,
//     "Upstream facts"; generalised from an L2 prefetch into staging in the SM's own memory);
//   * 16 consumer warps dequantise the staged rows in registers (cvt e4m3x2 / e2m1x2 -> f16x2 ->
//     fp32) and accumulate in fp32 with warp-shuffle reductions;
//   * grid barriers are replaced by per-phase arrival counters written with release and polled
//     with acquire at gpu scope ("Hazy-style counters", monolith page, "Design decisions", sync
//     experiment 2), each wait bounded by a %globaltimer deadline;
//   * the RMSNorm factor is recomputed by every CTA instead of meeting at a barrier (monolith
//     page, "Upstream facts", tricks already in upstream);
//   * attention is split over (KV head, position chunk) units; the last unit of a KV head to
//     finish merges the partial softmaxes, so no CTA waits for it;
//   * the LM head rows are spread over all CTAs, each CTA folds its (max, index) into one 64-bit
//     atomicMax, and the last CTA to finish writes the token (folding the two LM-head kernels
//     into the same launch, monolith page, "Design decisions", sync experiment 5).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mk_device.cuh"
#include "mk_internal.h"

namespace mk {

struct __align__(16) Smem {
  uint64_t full[NSLOT];
  uint64_t empty[NSLOT];
  float xs[XS_MAX];
  float hs[HID];
  float part[2][32][NCW];
  float gs[64];
  float us[64];
  float red[64];
  float qs[2][HD];
  float kn[HD];
  float vn[HD];
  float sc[2][UNIT_POS];
  float stat[4];
  int flag;
  volatile int abort;
};
constexpr int RING_BYTES = SLOT * NSLOT;
constexpr int SMEM_BYTES = RING_BYTES + (int)sizeof(Smem);

// ------------------------------------------------------------------ format geometry
__device__ __forceinline__ int epl_of(int fmt) { return fmt == 0 ? 8 : (fmt == 1 ? 16 : 32); }
__device__ __forceinline__ int code_bytes(int fmt, int K) { return fmt == 0 ? 2 * K : (fmt == 1 ? K : K / 2); }
__device__ __forceinline__ int scale_bytes(int fmt, int K) { return fmt == 2 ? K / 16 : 0; }
__device__ __forceinline__ int tile_rows(int fmt, int K) {
  int r = SLOT / (code_bytes(fmt, K) + scale_bytes(fmt, K));
  return r > 32 ? 32 : r;
}
// Position of input element k in the staged vector, laid out so that lane l of a warp reads the
// activations of its 16-byte weight slice as conflict-free float4 loads.
__device__ __forceinline__ int xs_index(int k, int epl) {
  int per_chunk = 32 * epl;
  int ch = k / per_chunk, r = k % per_chunk;
  int lane = r / epl, e = r % epl;
  return ((ch * (epl / 4) + e / 4) * 32 + lane) * 4 + (e & 3);
}
__device__ __forceinline__ void split_range(int n, int parts, int i, int& a, int& b) {
  a = (int)((long long)n * i / parts);
  b = (int)((long long)n * (i + 1) / parts);
}
__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ float ldg_bf16(const uint16_t* p) { return bf16f(__ldg(p)); }

// ------------------------------------------------------------------ X-ray
template <bool XR>
struct Xray {
  TraceRec* base;
  int n;
  __device__ void init(TraceRec* t) {
    base = t ? t + (size_t)blockIdx.x * TRACE_PER_CTA : nullptr;
    n = 0;
  }
  __device__ __forceinline__ void stamp(int phase, int kind) {
    if (XR && base && n < TRACE_PER_CTA) {
      TraceRec r;
      r.gtime = globaltimer();
      r.clk = clock64_();
      r.smid = smid();
      r.cta = (uint16_t)blockIdx.x;
      r.phase = (uint8_t)phase;
      r.kind = (uint8_t)kind;
      base[n++] = r;
    }
  }
  __device__ void finish() {
    if (XR && base && n < TRACE_PER_CTA) {
      TraceRec r = {};
      r.kind = 255;  // end marker
      base[n] = r;
    }
  }
};

// ------------------------------------------------------------------ per-CTA schedule
// Both the producer and the consumers derive the same ranges, so they agree on the tile order.
struct Sched {
  int q0, q1;    // rows of the virtual q|k|v matrix
  int o0, o1;    // o_proj output rows
  int j0, j1;    // FFN units (gate and up rows)
  int d0, d1;    // down_proj output rows
  int v0, v1;    // LM-head rows
  bool unit;     // this CTA runs an attention unit
  int ug, uc;    // its KV head and chunk
  int t0, t1;    // positions [t0, t1) of the chunk
  int ncached;   // positions of the chunk already in the cache (read through the ring)
  __device__ void make(const KParams& P) {
    const int G = gridDim.x, b = blockIdx.x;
    split_range(QKV_ROWS, G, b, q0, q1);
    split_range(HID, G, b, o0, o1);
    split_range(FFN, G, b, j0, j1);
    split_range(HID, G, b, d0, d1);
    split_range(P.vocab, G, b, v0, v1);
    unit = b < NKVH * P.units;
    ug = unit ? b / P.units : 0;
    uc = unit ? b % P.units : 0;
    split_range(P.pos + 1, P.units, uc, t0, t1);
    int c_end = t1 < P.pos ? t1 : P.pos;
    ncached = unit ? (c_end > t0 ? c_end - t0 : 0) : 0;
  }
};

// QKV segment s (0 = q, 1 = k, 2 = v) of the virtual row range.
__device__ __forceinline__ void qkv_segment(int s, int q0, int q1, int& r0, int& r1, int& base) {
  const int lo[3] = {0, QROWS, QROWS + KVROWS};
  const int hi[3] = {QROWS, QROWS + KVROWS, QKV_ROWS};
  base = lo[s];
  r0 = max(q0, lo[s]) - lo[s];
  r1 = min(q1, hi[s]) - lo[s];
}

// ------------------------------------------------------------------ producer
struct Producer {
  Smem* s;
  uint8_t* ring;
  const KParams* P;
  uint32_t n;
  uint64_t pol;
  bool ok;
  uint64_t deadline_ns;

  __device__ bool take_slot(uint32_t& slot) {
    slot = n % NSLOT;
    if (n >= NSLOT) {
      uint32_t par = ((n / NSLOT) - 1) & 1;
      if (!mbar_try_wait(&s->empty[slot], par)) {
        uint64_t t0 = globaltimer();
        while (!mbar_try_wait(&s->empty[slot], par)) {
          if (s->abort) return false;
          if (globaltimer() - t0 > deadline_ns) return false;
        }
      }
    }
    return true;
  }
  __device__ void issue(const uint8_t* src0, uint32_t b0, const uint8_t* src1, uint32_t b1) {
    if (!ok) return;
    uint32_t slot;
    if (!take_slot(slot)) {
      ok = false;
      return;
    }
    uint8_t* dst = ring + (size_t)slot * SLOT;
    mbar_expect_tx(&s->full[slot], b0 + b1);
    bulk_g2s(dst, src0, b0, &s->full[slot], pol);
    if (b1) bulk_g2s(dst + b0, src1, b1, &s->full[slot], pol);
    ++n;
  }
  __device__ void rows(const DMat& m, int K, int r0, int r1) {
    const int cb = code_bytes(m.fmt, K), sb = scale_bytes(m.fmt, K), rpt = tile_rows(m.fmt, K);
    for (int r = r0; r < r1 && ok; r += rpt) {
      int nr = min(rpt, r1 - r);
      issue(m.data + (size_t)r * cb, (uint32_t)(nr * cb), sb ? m.scale + (size_t)r * sb : nullptr,
            (uint32_t)(nr * sb));
    }
  }
  __device__ void kv(int layer, int g, int t0, int ncached) {
    for (int t = 0; t < ncached && ok; t += KVT) {
      int np = min(KVT, ncached - t);
      size_t off = (((size_t)layer * NKVH + g) * P->max_ctx + t0 + t) * HD;
      // K at slot offset 0, V at slot offset SLOT/2
      if (!ok) return;
      uint32_t slot;
      if (!take_slot(slot)) {
        ok = false;
        return;
      }
      uint8_t* dst = ring + (size_t)slot * SLOT;
      uint32_t bytes = (uint32_t)(np * HD * 2);
      mbar_expect_tx(&s->full[slot], 2 * bytes);
      bulk_g2s(dst, P->kc + off, bytes, &s->full[slot], pol);
      bulk_g2s(dst + SLOT / 2, P->vc + off, bytes, &s->full[slot], pol);
      ++n;
    }
  }
  // Wait until every copy this producer issued has landed (used on abort, before the CTA exits).
  __device__ void drain() {
    uint32_t first = n > NSLOT ? n - NSLOT : 0;
    for (uint32_t i = first; i < n; ++i) {
      uint32_t slot = i % NSLOT, par = (i / NSLOT) & 1;
      uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&s->full[slot], par))
        if (globaltimer() - t0 > 200000000ull) break;
    }
  }
};

__device__ void run_producer(const KParams& P, Smem* s, uint8_t* ring) {
  if ((threadIdx.x & 31) != 0) return;
  Producer pr;
  pr.s = s;
  pr.ring = ring;
  pr.P = &P;
  pr.n = 0;
  pr.pol = l2_evict_first_policy();
  pr.ok = true;
  pr.deadline_ns = P.timeout_ns;
  Sched S;
  S.make(P);
  for (int l = 0; l < P.n_layers && pr.ok; ++l) {
    const DLayer& L = P.layers[l];
    for (int sg = 0; sg < 3; ++sg) {
      int r0, r1, base;
      qkv_segment(sg, S.q0, S.q1, r0, r1, base);
      if (r0 < r1) pr.rows(L.m[M_Q + sg], HID, r0, r1);
    }
    if (S.unit) pr.kv(l, S.ug, S.t0, S.ncached);
    pr.rows(L.m[M_O], QROWS, S.o0, S.o1);
    pr.rows(L.m[M_GATE], HID, S.j0, S.j1);
    pr.rows(L.m[M_UP], HID, S.j0, S.j1);
    pr.rows(L.m[M_DOWN], FFN, S.d0, S.d1);
  }
  if (pr.ok) pr.rows(P.embed, HID, S.v0, S.v1);
  if (!pr.ok) pr.drain();
}

// ------------------------------------------------------------------ consumer
template <bool XR>
struct Consumer {
  Smem* s;
  uint8_t* ring;
  const KParams* P;
  uint32_t n;  // tiles consumed
  int tid, lane, warp;
  Xray<XR> xr;

  __device__ void fail(uint32_t code, uint32_t detail) {
    // first failure wins; tell every CTA to stop
    if (P->sync) {
      if (atomicCAS(&P->sync->status[0], 0u, code) == 0u) st_relaxed_u32(&P->sync->status[1], detail);
      st_relaxed_u32(&P->sync->status[2], 1u);
    }
    s->abort = 1;
  }
  __device__ __forceinline__ void st(int phase, int kind) {
    if (tid == 0) xr.stamp(phase, kind);
  }
  __device__ void wait_full(uint32_t slot, uint32_t par, int phase, int layer) {
    if (mbar_try_wait(&s->full[slot], par)) return;
    uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&s->full[slot], par)) {
      if (s->abort) return;
      if (globaltimer() - t0 > P->timeout_ns) {
        fail(3u, (uint32_t)(phase | (layer << 8) | (blockIdx.x << 16)) | 0x80000000u);
        return;
      }
    }
  }
  // Thread 0 polls `ctr` until it reaches `target`; returns false (CTA-uniformly) on abort.
  __device__ bool wait_ctr(const uint32_t* ctr, uint32_t target, int phase, int layer) {
    if (tid == 0) {
      xr.stamp(phase, 2);
      if (ld_acquire(ctr) < target) {
        uint64_t t0 = globaltimer();
        while (true) {
          if (ld_acquire(ctr) >= target) break;
          if (ld_relaxed_u32(&P->sync->status[2]) != 0u) {
            s->abort = 1;
            break;
          }
          if (globaltimer() - t0 > P->timeout_ns) {
            fail(3u, (uint32_t)(phase | (layer << 8) | (blockIdx.x << 16)));
            break;
          }
        }
      }
      xr.stamp(phase, 3);
    }
    bar_consumers(NCT);
    return s->abort == 0;
  }
  __device__ void signal(uint32_t* ctr, int phase, int layer) {
    bar_consumers(NCT);
    if (tid == 0) {
      bool skip = (P->fault_cta == (int)blockIdx.x) && (P->fault_phase == phase) && layer == 0;
      if (!skip) red_release_add(ctr, 1u);
    }
  }

  // RMSNorm of hs (HID values) with weight w, staged into xs for a matrix of format fmt.
  __device__ void stage_rmsnorm(const uint16_t* w, int fmt) {
    float a = s->hs[tid], b = s->hs[tid + NCT];
    float ss = a * a + b * b;
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) s->red[warp] = ss;
    bar_consumers(NCT);
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < NCW; ++i) tot += s->red[i];
    float inv = 1.0f / sqrtf(tot / (float)HID + P->eps);
    int epl = epl_of(fmt);
    s->xs[xs_index(tid, epl)] = a * inv * ldg_bf16(w + tid);
    s->xs[xs_index(tid + NCT, epl)] = b * inv * ldg_bf16(w + tid + NCT);
    bar_consumers(NCT);
  }
  // Load HID floats written by other CTAs into hs.
  __device__ void load_h(const float* src) {
    s->hs[tid] = ld_cg_f32(src + tid);
    s->hs[tid + NCT] = ld_cg_f32(src + tid + NCT);
    bar_consumers(NCT);
  }
  // Load n floats written by other CTAs straight into the staged layout for format fmt.
  __device__ void stage_global(const float* src, int n, int fmt) {
    int epl = epl_of(fmt);
    for (int k = tid; k < n; k += NCT) s->xs[xs_index(k, epl)] = ld_cg_f32(src + k);
    bar_consumers(NCT);
  }

  // Dequant-GEMV over rows [r0, r1) of m (K inputs), streamed through the ring; calls
  // epi(row, y) on threads 0..rows-in-tile-1 for every finished row. Returns false on abort.
  template <class Epi>
  __device__ bool rows(const DMat& m, int K, int r0, int r1, int phase, int layer, Epi epi) {
    const int fmt = m.fmt, epl = epl_of(fmt), nchunk = K / (32 * epl);
    const int cb = code_bytes(fmt, K), sbytes = scale_bytes(fmt, K), rpt = tile_rows(fmt, K);
    for (int r = r0; r < r1; r += rpt) {
      const int nr = min(rpt, r1 - r);
      const uint32_t slot = n % NSLOT, par = (n / NSLOT) & 1;
      wait_full(slot, par, phase, layer);
      const uint8_t* tile = ring + (size_t)slot * SLOT;
      const int items = nr * nchunk;
      const int i0 = warp * items / NCW, i1 = (warp + 1) * items / NCW;
      float(*part)[NCW] = s->part[n & 1];
      float acc = 0.f;
      int cur = -1;
      for (int i = i0; i < i1; ++i) {
        const int row = i / nchunk, ch = i - row * nchunk;
        if (row != cur) {
          if (cur >= 0) {
#pragma unroll
            for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) part[cur][warp] = acc;
          }
          acc = 0.f;
          cur = row;
        }
        const uint4 w = *reinterpret_cast<const uint4*>(tile + (size_t)row * cb + ch * 512 + lane * 16);
        const float4* xv = reinterpret_cast<const float4*>(s->xs) + ch * (epl / 4) * 32 + lane;
        if (fmt == 0) {
          float4 x[2] = {xv[0], xv[32]};
          acc = dot_bf16_16B(w, x, acc);
        } else if (fmt == 1) {
          float4 x[4] = {xv[0], xv[32], xv[64], xv[96]};
          acc = dot_fp8_16B(w, x, acc);
        } else {
          float4 x[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) x[j] = xv[32 * j];
          const uint16_t sp = *reinterpret_cast<const uint16_t*>(tile + (size_t)nr * cb + (size_t)row * sbytes +
                                                                 ch * 64 + lane * 2);
          const float2 sc = e4m3x2_to_f2(sp);
          acc = dot_nvfp4_16B(w, x, sc.x, sc.y, acc);
        }
      }
      if (cur >= 0) {
#pragma unroll
        for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) part[cur][warp] = acc;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s->empty[slot]);
      ++n;
      bar_consumers(NCT);
      if (s->abort) return false;
      if (tid < nr) {
        const int row = tid;
        float y = 0.f;
        for (int w = 0; w < NCW; ++w) {
          const int a = w * items / NCW, b = (w + 1) * items / NCW;
          if (a < b && a < (row + 1) * nchunk && b > row * nchunk) y += part[row][w];
        }
        if (fmt == 1) y *= __ldg(reinterpret_cast<const float*>(m.scale) + r + row);
        else if (fmt == 2) y *= m.tscale;
        epi(r + row, y);
      }
    }
    return true;
  }

  // One attention unit: KV head g, positions [S.t0, S.t1) of layer l.
  __device__ bool attention(const Sched& S, const DLayer& L, int l) {
    const KParams& p = *P;
    const int g = S.ug;
    // raw q (two heads), k, v of KV head g
    float val;
    if (tid < 2 * HD) val = ld_cg_f32(p.qkv + GQA * HD * g + tid);
    else if (tid < 3 * HD) val = ld_cg_f32(p.qkv + QROWS + HD * g + (tid - 2 * HD));
    else val = ld_cg_f32(p.qkv + QROWS + KVROWS + HD * g + (tid - 3 * HD));
    float ss = val * val;
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) s->red[warp] = ss;
    bar_consumers(NCT);
    const int vec = warp / 4, d = tid & (HD - 1);
    float nv = val;
    if (vec < 3) {  // QK-norm: RMSNorm over the head
      float tot = s->red[4 * vec] + s->red[4 * vec + 1] + s->red[4 * vec + 2] + s->red[4 * vec + 3];
      float inv = 1.0f / sqrtf(tot / (float)HD + p.eps);
      nv = val * inv * ldg_bf16((vec < 2 ? L.q_norm : L.k_norm) + d);
    }
    float* dst = vec == 0 ? s->qs[0] : (vec == 1 ? s->qs[1] : (vec == 2 ? s->kn : s->vn));
    dst[d] = nv;
    bar_consumers(NCT);
    if (tid < 3 * (HD / 2)) {  // RoPE, half-split pairs (i, i + 64)
      const int which = tid / (HD / 2), i = tid % (HD / 2);
      float* x = which == 0 ? s->qs[0] : (which == 1 ? s->qs[1] : s->kn);
      const float c = __ldg(p.rope_cos + (size_t)p.pos * (HD / 2) + i);
      const float sn = __ldg(p.rope_sin + (size_t)p.pos * (HD / 2) + i);
      const float a = x[i], b = x[i + HD / 2];
      x[i] = a * c - b * sn;
      x[i + HD / 2] = b * c + a * sn;
    }
    bar_consumers(NCT);
    if (tid < 2 * HD) {  // the cache holds bf16: round the new key and value
      const int which = tid / HD, dd = tid % HD;
      float* x = which ? s->vn : s->kn;
      const __nv_bfloat16 hb = __float2bfloat16_rn(x[dd]);
      const uint16_t bits = __bfloat16_as_ushort(hb);
      x[dd] = bf16f(bits);
      if (S.uc == p.units - 1) {
        uint16_t* cache = which ? p.vc : p.kc;
        cache[(((size_t)l * NKVH + g) * p.max_ctx + p.pos) * HD + dd] = bits;
      }
    }
    bar_consumers(NCT);
    // scores
    const int np = S.t1 - S.t0, ntiles = (S.ncached + KVT - 1) / KVT;
    for (int i = 0; i < ntiles; ++i) wait_full((n + i) % NSLOT, ((n + i) / NSLOT) & 1, PH_ATTN, l);
    bar_consumers(NCT);
    if (s->abort) return false;
    const float scale = 0.08838834764831845f;  // 1/sqrt(128)
    float q0[4], q1[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      q0[e] = s->qs[0][4 * lane + e];
      q1[e] = s->qs[1][4 * lane + e];
    }
    for (int t = warp; t < np; t += NCW) {
      float k4[4];
      if (t < S.ncached) {
        const uint8_t* tile = ring + (size_t)((n + t / KVT) % NSLOT) * SLOT;
        const uint2 raw = *reinterpret_cast<const uint2*>(tile + (t % KVT) * HD * 2 + lane * 8);
        k4[0] = __uint_as_float(raw.x << 16);
        k4[1] = __uint_as_float(raw.x & 0xFFFF0000u);
        k4[2] = __uint_as_float(raw.y << 16);
        k4[3] = __uint_as_float(raw.y & 0xFFFF0000u);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) k4[e] = s->kn[4 * lane + e];
      }
      float a = 0.f, b = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        a = fmaf(q0[e], k4[e], a);
        b = fmaf(q1[e], k4[e], b);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
      }
      if (lane == 0) {
        s->sc[0][t] = a * scale;
        s->sc[1][t] = b * scale;
      }
    }
    bar_consumers(NCT);
    if (warp < 2) {  // softmax numerators and partial sums of this chunk
      float m = -INFINITY;
      for (int t = lane; t < np; t += 32) m = fmaxf(m, s->sc[warp][t]);
#pragma unroll
      for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float sum = 0.f;
      for (int t = lane; t < np; t += 32) {
        const float e = expf(s->sc[warp][t] - m);
        s->sc[warp][t] = e;
        sum += e;
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) {
        s->stat[warp] = m;
        s->stat[2 + warp] = sum;
      }
    }
    bar_consumers(NCT);
    {
      const int h = tid >> 8, dd = (tid & 255) >> 1, half = tid & 1;
      float acc = 0.f;
      for (int t = half; t < np; t += 2) {
        float vv;
        if (t < S.ncached) {
          const uint8_t* tile = ring + (size_t)((n + t / KVT) % NSLOT) * SLOT;
          vv = bf16f(*reinterpret_cast<const uint16_t*>(tile + SLOT / 2 + (t % KVT) * HD * 2 + dd * 2));
        } else {
          vv = s->vn[dd];
        }
        acc = fmaf(s->sc[h][t], vv, acc);
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      if (half == 0) {
        float* part = p.attp + (((size_t)g * MAXC + S.uc) * 2 + h) * PART_STRIDE;
        part[4 + dd] = acc;
        if (dd == 0) {
          part[0] = s->stat[h];
          part[1] = s->stat[2 + h];
        }
      }
    }
    bar_consumers(NCT);
    for (int i = 0; i < ntiles; ++i)
      if (lane == 0) mbar_arrive(&s->empty[(n + i) % NSLOT]);
    n += ntiles;
    // the last unit of this KV head to finish merges the chunks
    if (tid == 0) {
      fence_acqrel_gpu();
      const uint32_t old = atom_acqrel_add(&p.sync->grp[g][0], 1u);
      s->flag = (old == (uint32_t)((l + 1) * p.units - 1)) ? 1 : 0;
    }
    bar_consumers(NCT);
    if (s->flag) {
      if (tid < 2 * HD) {
        const int h = tid / HD, dd = tid % HD;
        float M = -INFINITY;
        for (int c = 0; c < p.units; ++c)
          M = fmaxf(M, ld_cg_f32(p.attp + (((size_t)g * MAXC + c) * 2 + h) * PART_STRIDE));
        float Lsum = 0.f, o = 0.f;
        for (int c = 0; c < p.units; ++c) {
          const float* part = p.attp + (((size_t)g * MAXC + c) * 2 + h) * PART_STRIDE;
          const float w = expf(ld_cg_f32(part) - M);
          Lsum = fmaf(w, ld_cg_f32(part + 1), Lsum);
          o = fmaf(w, ld_cg_f32(part + 4 + dd), o);
        }
        p.att[GQA * HD * g + tid] = o / Lsum;
      }
      signal(&p.sync->c[PH_ATTN][0], PH_ATTN, l);
    }
    return true;
  }

  __device__ void run(const KParams& p) {
    const int G = gridDim.x;
    Sched S;
    S.make(p);
    // ---------------- embedding: h = row `token` of the tied matrix (every CTA, no wait)
    st(PH_EMBED, 0);
    const int token = p.token_ptr ? *(volatile const int32_t*)p.token_ptr : p.token;
    if ((unsigned)token >= (unsigned)p.vocab) {  // e.g. the previous greedy step was abandoned
      if (tid == 0) fail(4u, (uint32_t)blockIdx.x << 16);
      bar_consumers(NCT);
      return;
    }
    {
      const DMat& E = p.embed;
      for (int k = tid; k < HID; k += NCT) {
        float v;
        if (E.fmt == 0) {
          v = bf16f(__ldg(reinterpret_cast<const uint16_t*>(E.data) + (size_t)token * HID + k));
        } else {
          const uint8_t c = __ldg(E.data + (size_t)token * HID + k);
          const float2 f = e4m3x2_to_f2(c);
          v = f.x * __ldg(reinterpret_cast<const float*>(E.scale) + token);
        }
        s->hs[k] = v;
        if (p.hidden_dbg && blockIdx.x == 0) p.hidden_dbg[k] = v;
      }
    }
    bar_consumers(NCT);
    st(PH_EMBED, 1);
    for (int l = 0; l < p.n_layers; ++l) {
      const DLayer& L = p.layers[l];
      // ---------------- QKV
      if (l > 0) {
        if (!wait_ctr(&p.sync->c[PH_DOWN][0], (uint32_t)(l * G), PH_DOWN, l)) return;
        load_h(p.h_mlp);
      }
      st(PH_QKV, 0);
      stage_rmsnorm(L.ln_in, L.m[M_Q].fmt);
      for (int sg = 0; sg < 3; ++sg) {
        int r0, r1, base;
        qkv_segment(sg, S.q0, S.q1, r0, r1, base);
        if (r0 >= r1) continue;
        float* out = p.qkv + base;
        if (!rows(L.m[M_Q + sg], HID, r0, r1, PH_QKV, l, [&](int r, float y) { out[r] = y; })) return;
      }
      signal(&p.sync->c[PH_QKV][0], PH_QKV, l);
      st(PH_QKV, 1);
      // ---------------- attention
      if (S.unit) {
        if (!wait_ctr(&p.sync->c[PH_QKV][0], (uint32_t)((l + 1) * G), PH_QKV, l)) return;
        st(PH_ATTN, 0);
        if (!attention(S, L, l)) return;
        st(PH_ATTN, 1);
      }
      // ---------------- o_proj + residual
      if (!wait_ctr(&p.sync->c[PH_ATTN][0], (uint32_t)((l + 1) * NKVH), PH_ATTN, l)) return;
      st(PH_O, 0);
      stage_global(p.att, QROWS, L.m[M_O].fmt);
      {
        float* hout = p.h_attn;
        const float* hin = s->hs;
        if (!rows(L.m[M_O], QROWS, S.o0, S.o1, PH_O, l, [&](int r, float y) { hout[r] = hin[r] + y; })) return;
      }
      signal(&p.sync->c[PH_O][0], PH_O, l);
      st(PH_O, 1);
      // ---------------- post-attention RMSNorm + gate/up + SwiGLU
      if (!wait_ctr(&p.sync->c[PH_O][0], (uint32_t)((l + 1) * G), PH_O, l)) return;
      st(PH_GATEUP, 0);
      load_h(p.h_attn);
      stage_rmsnorm(L.ln_post, L.m[M_GATE].fmt);
      {
        float* gs = s->gs;
        float* us = s->us;
        const int j0 = S.j0;
        if (!rows(L.m[M_GATE], HID, S.j0, S.j1, PH_GATEUP, l, [&](int r, float y) { gs[r - j0] = y; })) return;
        if (!rows(L.m[M_UP], HID, S.j0, S.j1, PH_GATEUP, l, [&](int r, float y) { us[r - j0] = y; })) return;
      }
      bar_consumers(NCT);
      if (tid < S.j1 - S.j0) {
        const float gv = s->gs[tid];
        p.act[S.j0 + tid] = gv / (1.0f + expf(-gv)) * s->us[tid];
      }
      signal(&p.sync->c[PH_GATEUP][0], PH_GATEUP, l);
      st(PH_GATEUP, 1);
      // ---------------- down_proj + residual
      if (!wait_ctr(&p.sync->c[PH_GATEUP][0], (uint32_t)((l + 1) * G), PH_GATEUP, l)) return;
      st(PH_DOWN, 0);
      stage_global(p.act, FFN, L.m[M_DOWN].fmt);
      {
        float* hout = p.h_mlp;
        const float* hin = s->hs;
        float* dbg = p.hidden_dbg ? p.hidden_dbg + (size_t)(l + 1) * HID : nullptr;
        if (!rows(L.m[M_DOWN], FFN, S.d0, S.d1, PH_DOWN, l, [&](int r, float y) {
              const float v = hin[r] + y;
              hout[r] = v;
              if (dbg) dbg[r] = v;
            }))
          return;
      }
      signal(&p.sync->c[PH_DOWN][0], PH_DOWN, l);
      st(PH_DOWN, 1);
    }
    // ---------------- final RMSNorm + LM head + argmax
    if (!wait_ctr(&p.sync->c[PH_DOWN][0], (uint32_t)(p.n_layers * G), PH_DOWN, p.n_layers)) return;
    st(PH_HEAD, 0);
    load_h(p.h_mlp);
    stage_rmsnorm(p.final_norm, p.embed.fmt);
    float best = -INFINITY;
    int besti = 0x7FFFFFFF;
    {
      float* lg = p.logits;
      if (!rows(p.embed, HID, S.v0, S.v1, PH_HEAD, p.n_layers, [&](int r, float y) {
            if (lg) lg[r] = y;
            if (y > best || (y == best && r < besti)) {
              best = y;
              besti = r;
            }
          }))
        return;
    }
    // CTA argmax (lowest index among equal maxima)
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, besti, o);
      if (ob > best || (ob == best && oi < besti)) {
        best = ob;
        besti = oi;
      }
    }
    if (lane == 0) {
      s->red[warp] = best;
      s->red[32 + warp] = __int_as_float(besti);
    }
    bar_consumers(NCT);
    if (tid == 0) {
      for (int w = 1; w < NCW; ++w) {
        const float ob = s->red[w];
        const int oi = __float_as_int(s->red[32 + w]);
        if (ob > best || (ob == best && oi < besti)) {
          best = ob;
          besti = oi;
        }
      }
      const uint32_t u = __float_as_uint(best);
      const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
      const unsigned long long key = ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)besti);
      atomicMax(&p.sync->key[0], key);
      fence_acqrel_gpu();
      const uint32_t old = atom_acqrel_add(&p.sync->c[PH_HEAD][0], 1u);
      if (old == (uint32_t)(G - 1)) {  // last CTA: publish the token, reset the step's counters
        const unsigned long long k = ld_relaxed_u64(&p.sync->key[0]);
        const int32_t nxt = (int32_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
        p.sync->tok[0] = nxt;
        if (p.next_out) *p.next_out = nxt;
        for (int i = 0; i < 8; ++i) st_relaxed_u32(&p.sync->c[i][0], 0u);
        for (int i = 0; i < NKVH; ++i) st_relaxed_u32(&p.sync->grp[i][0], 0u);
        st_relaxed_u64(&p.sync->key[0], 0ull);
      }
    }
    st(PH_HEAD, 1);
  }
};

template <bool XR>
__global__ void __launch_bounds__(NTHREADS, 1) k_decode(const KParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = smem_raw;
  Smem* s = reinterpret_cast<Smem*>(smem_raw + RING_BYTES);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&s->full[i], 1);
      mbar_init(&s->empty[i], NCW);
    }
    s->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x >= NCT) {
    run_producer(p, s, ring);
  } else {
    Consumer<XR> c;
    c.s = s;
    c.ring = ring;
    c.P = &p;
    c.n = 0;
    c.tid = threadIdx.x;
    c.lane = threadIdx.x & 31;
    c.warp = threadIdx.x >> 5;
    c.xr.init(p.trace);
    c.run(p);
    if (c.tid == 0) c.xr.finish();
  }
}

// ------------------------------------------------------------------ standalone GEMV
__global__ void __launch_bounds__(NTHREADS, 1) k_gemv(const DMat m, int rows, int cols, const float* x, float* y,
                                                      SyncBlock* sync) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = smem_raw;
  Smem* s = reinterpret_cast<Smem*>(smem_raw + RING_BYTES);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&s->full[i], 1);
      mbar_init(&s->empty[i], NCW);
    }
    s->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  int r0, r1;
  split_range(rows, gridDim.x, blockIdx.x, r0, r1);
  KParams p = {};
  p.sync = sync;
  p.timeout_ns = 2000000000ull;
  p.fault_cta = -1;
  if (threadIdx.x >= NCT) {
    if ((threadIdx.x & 31) != 0) return;
    Producer pr;
    pr.s = s;
    pr.ring = ring;
    pr.P = &p;
    pr.n = 0;
    pr.pol = l2_evict_first_policy();
    pr.ok = true;
    pr.deadline_ns = p.timeout_ns;
    pr.rows(m, cols, r0, r1);
    if (!pr.ok) pr.drain();
  } else {
    Consumer<false> c;
    c.s = s;
    c.ring = ring;
    c.P = &p;
    c.n = 0;
    c.tid = threadIdx.x;
    c.lane = threadIdx.x & 31;
    c.warp = threadIdx.x >> 5;
    c.xr.init(nullptr);
    c.stage_global(x, cols, m.fmt);
    c.rows(m, cols, r0, r1, PH_HEAD, 0, [&](int r, float v) { y[r] = v; });
  }
}

// ------------------------------------------------------------------ streaming-read probe
__global__ void __launch_bounds__(NTHREADS, 1) k_stream_read(const uint8_t* buf, size_t per_cta, uint32_t* sink) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = smem_raw;
  Smem* s = reinterpret_cast<Smem*>(smem_raw + RING_BYTES);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&s->full[i], 1);
      mbar_init(&s->empty[i], NCW);
    }
    s->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const uint8_t* base = buf + (size_t)blockIdx.x * per_cta;
  const uint32_t nt = (uint32_t)(per_cta / SLOT);
  if (threadIdx.x >= NCT) {
    if ((threadIdx.x & 31) != 0) return;
    KParams p = {};
    Producer pr;
    pr.s = s;
    pr.ring = ring;
    pr.P = &p;
    pr.n = 0;
    pr.pol = l2_evict_first_policy();
    pr.ok = true;
    pr.deadline_ns = 2000000000ull;
    for (uint32_t i = 0; i < nt && pr.ok; ++i) pr.issue(base + (size_t)i * SLOT, SLOT, nullptr, 0);
    if (!pr.ok) pr.drain();
  } else {
    const int lane = threadIdx.x & 31;
    uint32_t acc = 0;
    for (uint32_t i = 0; i < nt; ++i) {
      const uint32_t slot = i % NSLOT, par = (i / NSLOT) & 1;
      uint64_t t0 = globaltimer();
      bool ok = true;
      while (!mbar_try_wait(&s->full[slot], par))
        if (globaltimer() - t0 > 2000000000ull) {
          ok = false;
          break;
        }
      if (!ok) break;
      const uint4 v = *reinterpret_cast<const uint4*>(ring + (size_t)slot * SLOT + threadIdx.x * 16);
      acc ^= v.x ^ v.y ^ v.z ^ v.w;
      __syncwarp();
      if (lane == 0) mbar_arrive(&s->empty[slot]);
    }
    if (sink && acc == 0x9E3779B9u) sink[0] = acc;
  }
}

// ------------------------------------------------------------------ launchers
int decode_smem_bytes() { return SMEM_BYTES; }

static bool g_attr_done = false;
static int set_attrs() {
  if (g_attr_done) return 0;
  cudaError_t e;
  e = cudaFuncSetAttribute(k_decode<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return -1;
  e = cudaFuncSetAttribute(k_decode<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return -1;
  e = cudaFuncSetAttribute(k_gemv, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return -1;
  e = cudaFuncSetAttribute(k_stream_read, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return -1;
  g_attr_done = true;
  return 0;
}

int decode_occupancy(int* blocks_per_sm) {
  if (set_attrs()) return -1;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k_decode<false>, NTHREADS, SMEM_BYTES) ==
                 cudaSuccess
             ? 0
             : -1;
}

int launch_decode(const KParams& p, int grid, bool xray, void* stream) {
  if (set_attrs()) return -1;
  void* args[] = {(void*)&p};
  cudaError_t e = cudaLaunchCooperativeKernel(xray ? (const void*)k_decode<true> : (const void*)k_decode<false>,
                                              dim3(grid), dim3(NTHREADS), args, SMEM_BYTES, (cudaStream_t)stream);
  return e == cudaSuccess ? 0 : -1;
}

int launch_gemv(const DMat& m, int rows, int cols, const float* x, float* y, int grid, void* stream) {
  if (set_attrs()) return -1;
  k_gemv<<<grid, NTHREADS, SMEM_BYTES, (cudaStream_t)stream>>>(m, rows, cols, x, y, nullptr);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_stream_read(const void* buf, size_t bytes, int grid, void* stream) {
  if (set_attrs()) return -1;
  size_t per = bytes / grid;
  k_stream_read<<<grid, NTHREADS, SMEM_BYTES, (cudaStream_t)stream>>>((const uint8_t*)buf, per, nullptr);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace mk
