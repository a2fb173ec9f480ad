// ORACLE -- test infrastructure, not part of the product.
//
// A plain, slow, obviously-correct CPU implementation of one batch-1 decode step of a
// Qwen3-0.6B-shaped transformer whose linear layers are stored as bf16, FP8-E4M3 with one
// fp32 scale per output row, or NVFP4 (E2M1 codes, one E4M3 scale per 16 consecutive inputs,
// one fp32 scale per tensor). Everything is computed in double precision, in the order the
// definitions state; the only intermediate rounding is the bf16 KV cache, which is part of
// the definition (the KV cache is kept in bf16: monolith page, "Design decisions", KV cache).
//
// Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg may load this library.
// It shares no code, header, table or constant generator with the CUDA path.
//
// Sources (monolith page = "monolith" project plan, projects.dotslasha.me/p/monolith/):
//   model shape, tied embeddings, QK-norm, RoPE ........ monolith page, "Upstream facts" (Model bullet)
//   FP8 format (E4M3, fp32 per-output-row scale, RTN) .. monolith page, "Design decisions" (FP8 format)
//   NVFP4 format (E2M1 + E4M3 per 16 + fp32 tensor) ..... monolith page, "Design decisions" (NVFP4 format)
//   E2M1 value grid {0,+-0.5,+-1,+-1.5,+-2,+-3,+-4,+-6} .. TSCT super-kernel page, section 3b, path 2
//   LM head = embedding matrix, argmax ................... monolith page, "Upstream facts" (Launch structure)
//   bf16 KV cache ........................................ monolith page, "Design decisions" (KV cache)
// Readings where the pages are silent (RoPE pairing, GQA mapping, eps, theta, scale formulas,
// tie rules) are stated at each function below.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

// ------------------------------------------------------------------------------------------
// Number formats
// ------------------------------------------------------------------------------------------

// Round |a| (finite, >= 0) to the nearest value with `p` significant bits whose exponent is
// at least `emin` (values below 2^emin are on the fixed subnormal grid of spacing 2^(emin-p+1)).
// Ties go to the neighbour with an even last significand bit. Uses nearbyint under the default
// round-to-nearest-even mode; every scaling below is by a power of two and therefore exact.
double round_sig(double a, int p, int emin) {
  if (a == 0.0) return 0.0;
  int ex;
  std::frexp(a, &ex);  // a = f * 2^ex, f in [0.5, 1)
  int e = ex - 1;      // a in [2^e, 2^(e+1))
  if (e < emin) e = emin;
  double quantum = std::ldexp(1.0, e - (p - 1));
  return std::nearbyint(a / quantum) * quantum;
}

// OCP FP8 E4M3 ("e4m3fn"): sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities,
// S.1111.111 is NaN, largest finite magnitude 448.
double e4m3_value(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  double mag = (e == 0) ? std::ldexp((double)m, -9) : std::ldexp((double)(8 + m), e - 10);
  return s ? -mag : mag;
}

// Round-to-nearest-even into E4M3 with saturation to +-448 (the "satfinite" behaviour);
// the sign of the input is kept even when the magnitude rounds to zero.
uint8_t e4m3_encode(double v) {
  uint8_t s = std::signbit(v) ? 0x80 : 0x00;
  double a = std::fabs(v);
  if (std::isnan(v)) return 0x7F;
  if (a >= 448.0) return s | 0x7E;
  double r = round_sig(a, 4, -6);  // 1 implicit + 3 stored bits, smallest normal 2^-6
  if (r == 0.0) return s;
  if (r >= 448.0) return s | 0x7E;
  int ex;
  std::frexp(r, &ex);
  int e = ex - 1;
  if (e < -6) {  // subnormal: value = m * 2^-9
    return s | (uint8_t)std::lrint(std::ldexp(r, 9));
  }
  int m = (int)std::lrint(std::ldexp(r, 3 - e)) - 8;
  return s | (uint8_t)(((e + 7) << 3) | m);
}

// FP4 E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit, no inf/NaN.
// Magnitudes by code 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6.
double e2m1_value(uint8_t nib) {
  int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
  double mag = (e == 0) ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

// Round-to-nearest-even into E2M1 with saturation to +-6; sign kept on zero.
uint8_t e2m1_encode(double v) {
  uint8_t s = std::signbit(v) ? 0x8 : 0x0;
  double a = std::fabs(v);
  if (a >= 6.0) return s | 0x7;
  double r = round_sig(a, 2, 0);  // 1 implicit + 1 stored bit, smallest normal 2^0
  if (r >= 6.0) return s | 0x7;
  if (r < 1.0) return s | (uint8_t)std::lrint(2.0 * r);  // 0 or 0.5
  int ex;
  std::frexp(r, &ex);
  int e = ex - 1;                                         // 0, 1 or 2
  int m = (int)std::lrint(std::ldexp(r, 1 - e)) - 2;      // 0 or 1
  return s | (uint8_t)(((e + 1) << 1) | m);
}

// bf16: the top 16 bits of an IEEE binary32.
double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// Round-to-nearest-even of a finite double into bf16 (8 significant bits, binary32 exponent range).
uint16_t bf16_encode(double v) {
  uint16_t s = std::signbit(v) ? 0x8000 : 0;
  double a = std::fabs(v);
  double r = round_sig(a, 8, -126);
  if (r == 0.0) return s;
  if (r >= std::ldexp(1.0, 128)) return s | 0x7F80;  // overflow to infinity
  int ex;
  std::frexp(r, &ex);
  int e = ex - 1;
  if (e < -126) return s | (uint16_t)std::lrint(std::ldexp(r, 133));  // subnormal: m * 2^-133
  int m = (int)std::lrint(std::ldexp(r, 7 - e)) - 128;
  return s | (uint16_t)(((e + 127) << 7) | m);
}

// Run f(r0, r1) over [0, rows) split into nthreads contiguous ranges.
template <class F>
void parallel_rows(int rows, int nthreads, F f) {
  int nt = std::max(1, std::min(nthreads, rows));
  if (nt == 1) {
    f(0, rows);
    return;
  }
  std::vector<std::thread> th;
  for (int t = 0; t < nt; ++t)
    th.emplace_back(f, (int)((long long)rows * t / nt), (int)((long long)rows * (t + 1) / nt));
  for (auto& x : th) x.join();
}

double e4m3_table[256];
double e2m1_table[16];
struct TableInit {
  TableInit() {
    for (int c = 0; c < 256; ++c) e4m3_table[c] = e4m3_value((uint8_t)c);
    for (int c = 0; c < 16; ++c) e2m1_table[c] = e2m1_value((uint8_t)c);
  }
} table_init;

float bf16_as_float(uint16_t b) { return (float)bf16_value(b); }

// ------------------------------------------------------------------------------------------
// Weight formats (canonical, row-major) and their dequantisation
// ------------------------------------------------------------------------------------------
enum Fmt { FMT_BF16 = 0, FMT_FP8_ROW = 1, FMT_NVFP4 = 2 };

struct OrMat {           // mirrors the packed arrays a caller hands to the decoder
  const void* data;      // bf16 [rows][cols] | e4m3 [rows][cols] | e2m1 pairs [rows][cols/2]
  const void* scale;     // NULL | fp32 [rows] | e4m3 [rows][cols/16]
  float tensor_scale;    // NVFP4 only
  int fmt;
};

// Dequantise row r of an R x C matrix into `out` (double, exact for every format).
void dequant_row(const OrMat& m, int cols, int r, double* out) {
  if (m.fmt == FMT_BF16) {
    const uint16_t* p = (const uint16_t*)m.data + (size_t)r * cols;
    for (int k = 0; k < cols; ++k) out[k] = bf16_value(p[k]);
  } else if (m.fmt == FMT_FP8_ROW) {
    const uint8_t* p = (const uint8_t*)m.data + (size_t)r * cols;
    double s = (double)((const float*)m.scale)[r];
    for (int k = 0; k < cols; ++k) out[k] = e4m3_table[p[k]] * s;
  } else {
    const uint8_t* p = (const uint8_t*)m.data + (size_t)r * (cols / 2);
    const uint8_t* bs = (const uint8_t*)m.scale + (size_t)r * (cols / 16);
    double t = (double)m.tensor_scale;
    for (int k = 0; k < cols; ++k) {
      uint8_t byte = p[k / 2];
      uint8_t nib = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);  // even element in the low nibble
      out[k] = e2m1_table[nib] * e4m3_table[bs[k / 16]] * t;
    }
  }
}

// y[r] = sum_k W[r][k] * x[k], each row summed serially in k order (so the result does not
// depend on the thread count). Rows are split over `nthreads` std::threads.
void gemv(const OrMat& m, int rows, int cols, const double* x, double* y, int nthreads) {
  auto work = [&](int r0, int r1) {
    std::vector<double> w(cols);
    for (int r = r0; r < r1; ++r) {
      dequant_row(m, cols, r, w.data());
      double acc = 0.0;
      for (int k = 0; k < cols; ++k) acc += w[k] * x[k];
      y[r] = acc;
    }
  };
  bool small = (long long)rows * cols < (1 << 20);
  parallel_rows(rows, small ? 1 : nthreads, work);
}

// RMSNorm with a multiplicative weight: out = x / sqrt(mean(x^2) + eps) * w  (no "1 + w").
void rmsnorm(const double* x, const uint16_t* w, int n, double eps, double* out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / std::sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) out[i] = x[i] * inv * bf16_value(w[i]);
}

// Rotary embedding, half-split pairing: (x_i, x_{i+D/2}) is rotated by angle
// pos * theta^(-2i/D), i = 0..D/2-1. Angle, cos and sin in double.
void rope(double* x, int d, int pos, double theta) {
  int half = d / 2;
  for (int i = 0; i < half; ++i) {
    double inv_freq = std::pow(theta, -2.0 * i / d);
    double ang = (double)pos * inv_freq;
    double c = std::cos(ang), s = std::sin(ang);
    double a = x[i], b = x[i + half];
    x[i] = a * c - b * s;
    x[i + half] = b * c + a * s;
  }
}

double silu(double z) { return z / (1.0 + std::exp(-z)); }

// Single-query softmax attention over n cached positions (bf16 rows of length d):
// s_t = q . K_t / sqrt(d); p = softmax(s); out = sum_t p_t V_t.
void attend(const double* q, const uint16_t* K, const uint16_t* V, int n, int d, double* out) {
  const double scale = 1.0 / std::sqrt((double)d);
  std::vector<double> s(n);
  double mx = -std::numeric_limits<double>::infinity();
  for (int t = 0; t < n; ++t) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i) acc += q[i] * bf16_value(K[(size_t)t * d + i]);
    s[t] = acc * scale;
    mx = std::max(mx, s[t]);
  }
  double den = 0.0;
  for (int t = 0; t < n; ++t) {
    s[t] = std::exp(s[t] - mx);
    den += s[t];
  }
  for (int i = 0; i < d; ++i) out[i] = 0.0;
  for (int t = 0; t < n; ++t) {
    double p = s[t] / den;
    for (int i = 0; i < d; ++i) out[i] += p * bf16_value(V[(size_t)t * d + i]);
  }
}

// Index of the largest value; the lowest index wins among equal maxima.
int argmax_lowest(const double* x, int n) {
  int best = 0;
  for (int i = 1; i < n; ++i)
    if (x[i] > x[best]) best = i;
  return best;
}


// ------------------------------------------------------------------------------------------
// Quantisers (produce the canonical packed arrays)
// ------------------------------------------------------------------------------------------
// The quotients that decide each code are formed in binary32, as the device packer forms them:
//   FP8:   s = fp32(absmax_row / 448);  code = E4M3_RNE_satfinite(fp32(w / s)).
//   NVFP4: t = fp32(amax_tensor / 2688)            (2688 = 6 * 448)
//          b = E4M3_RNE_satfinite(fp32(amax_block / fp32(6 * t)))
//          code = E2M1_RNE_satfinite(fp32(w / fp32(value(b) * t)))
// A zero scale (all-zero row, block or tensor) gives all-zero codes.
// bf16_scale: the row scale is a bf16 number (the monolith page, "Design decisions", FP8 format,
// allows an fp32 or a bf16 scale): fp32(absmax / 448) rounded to nearest-even bf16; the elements
// are then divided by that scale, so the row maximum may saturate at 448.
void quant_fp8_row(const uint16_t* w, int rows, int cols, uint8_t* codes, float* scales,
                   int nthreads, bool bf16_scale = false) {
  parallel_rows(rows, nthreads, [&](int r0, int r1) {
  for (int r = r0; r < r1; ++r) {
    const uint16_t* p = w + (size_t)r * cols;
    float amax = 0.0f;
    for (int k = 0; k < cols; ++k) amax = std::max(amax, (float)std::fabs(bf16_value(p[k])));
    volatile float s = amax / 448.0f;
    if (bf16_scale) s = (float)bf16_value(bf16_encode((double)s));
    scales[r] = s;
    for (int k = 0; k < cols; ++k) {
      if (s == 0.0f) {
        codes[(size_t)r * cols + k] = 0;
        continue;
      }
      volatile float q = bf16_as_float(p[k]) / s;
      codes[(size_t)r * cols + k] = e4m3_encode((double)q);
    }
  }
  });
}

// The E2M1 codes of one 16-element block for block-scale code `bc` (binary32 quotient, as in
// quant_nvfp4) and the block's squared reconstruction error, summed in double in element order.
double nvfp4_block(const uint16_t* p, uint8_t bc, float t, uint8_t* nib) {
  volatile float bval = (float)e4m3_value(bc);
  volatile float denom = bval * t;
  double err = 0.0;
  for (int j = 0; j < 16; ++j) {
    nib[j] = 0;
    if (denom != 0.0f) {
      volatile float q = bf16_as_float(p[j]) / denom;
      nib[j] = e2m1_encode((double)q);
    }
    const double rec = e2m1_value(nib[j]) * e4m3_value(bc) * (double)t;
    const double d = bf16_value(p[j]) - rec;
    err += d * d;
  }
  return err;
}

// NVFP4 with the per-block scale search the pages ask for (round-to-nearest codes, and per block
// the scale that gives the least squared error: monolith page, "Design decisions", NVFP4 format).
// Reading:
// the tensor scale is the amax one of quant_nvfp4; every E4M3 code 0 .. 0x7E (all non-negative
// finite block scales) is a candidate; a candidate's E2M1 codes are round-to-nearest as in
// quant_nvfp4 and its error is the summed squared reconstruction error of the block; the least
// error wins, ties to the smaller code (so an all-zero block keeps code 0).
void quant_nvfp4_mse(const uint16_t* w, int rows, int cols, uint8_t* codes, uint8_t* bscales,
                     float* tscale_out, int nthreads) {
  float amax_t = 0.0f;
  for (size_t i = 0; i < (size_t)rows * cols; ++i)
    amax_t = std::max(amax_t, (float)std::fabs(bf16_value(w[i])));
  volatile float t = amax_t / 2688.0f;
  *tscale_out = t;
  parallel_rows(rows, nthreads, [&](int r0, int r1) {
  for (int r = r0; r < r1; ++r) {
    for (int b = 0; b < cols / 16; ++b) {
      const uint16_t* p = w + (size_t)r * cols + (size_t)b * 16;
      uint8_t best = 0, nib[16], bnib[16];
      double besterr = nvfp4_block(p, 0, t, bnib);
      for (int c = 1; c <= 0x7E; ++c) {
        const double e = nvfp4_block(p, (uint8_t)c, t, nib);
        if (e < besterr) {
          besterr = e;
          best = (uint8_t)c;
          std::memcpy(bnib, nib, 16);
        }
      }
      bscales[(size_t)r * (cols / 16) + b] = best;
      for (int j = 0; j < 16; ++j) {
        size_t k = (size_t)b * 16 + j;
        uint8_t& byte = codes[(size_t)r * (cols / 2) + k / 2];
        if (k % 2 == 0) byte = (uint8_t)((byte & 0xF0) | bnib[j]);
        else byte = (uint8_t)((byte & 0x0F) | (bnib[j] << 4));
      }
    }
  }
  });
}

void quant_nvfp4(const uint16_t* w, int rows, int cols, uint8_t* codes, uint8_t* bscales,
                 float* tscale_out, int nthreads) {
  float amax_t = 0.0f;
  for (size_t i = 0; i < (size_t)rows * cols; ++i)
    amax_t = std::max(amax_t, (float)std::fabs(bf16_value(w[i])));
  volatile float t = amax_t / 2688.0f;
  *tscale_out = t;
  volatile float t6 = 6.0f * t;
  parallel_rows(rows, nthreads, [&](int r0, int r1) {
  for (int r = r0; r < r1; ++r) {
    for (int b = 0; b < cols / 16; ++b) {
      const uint16_t* p = w + (size_t)r * cols + (size_t)b * 16;
      float amax_b = 0.0f;
      for (int j = 0; j < 16; ++j) amax_b = std::max(amax_b, (float)std::fabs(bf16_value(p[j])));
      uint8_t bcode = 0;
      if (t6 != 0.0f) {
        volatile float ratio = amax_b / t6;
        bcode = e4m3_encode((double)ratio);
      }
      bscales[(size_t)r * (cols / 16) + b] = bcode;
      volatile float bval = (float)e4m3_value(bcode);
      volatile float denom = bval * t;
      for (int j = 0; j < 16; ++j) {
        uint8_t nib = 0;
        if (denom != 0.0f) {
          volatile float q = bf16_as_float(p[j]) / denom;
          nib = e2m1_encode((double)q);
        }
        size_t k = (size_t)b * 16 + j;
        uint8_t& byte = codes[(size_t)r * (cols / 2) + k / 2];
        if (k % 2 == 0) byte = (uint8_t)((byte & 0xF0) | nib);
        else byte = (uint8_t)((byte & 0x0F) | (nib << 4));
      }
    }
  }
  });
}

// ------------------------------------------------------------------------------------------
// The decoder
// ------------------------------------------------------------------------------------------
struct OrLayer {
  OrMat q, k, v, o, gate, up, down;
  const uint16_t* ln_in;    // bf16 [hidden]
  const uint16_t* ln_post;  // bf16 [hidden]
  const uint16_t* q_norm;   // bf16 [head_dim]
  const uint16_t* k_norm;   // bf16 [head_dim]
};

struct OrDesc {
  int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab, max_ctx;
  double rope_theta, rms_eps;
  const OrLayer* layers;
  OrMat embed;               // tied embedding / LM head [vocab][hidden]
  const uint16_t* final_norm;
  int n_threads;
};

struct OrModel {
  OrDesc d;
  std::vector<OrLayer> layers;
  std::vector<uint16_t> kcache, vcache;  // bf16 [layer][kv_head][max_ctx][head_dim]
  size_t kv_index(int l, int h, int t) const {
    return (((size_t)l * d.n_kv_heads + h) * d.max_ctx + t) * d.head_dim;
  }
};

// One decode step: writes K/V at `pos`, attends over positions 0..pos, returns argmax of the
// logits (lowest index among equal maxima). Optional outputs: logits [vocab], hidden
// [(n_layers+1) * hidden] (embedding output, then the residual stream after each layer),
// top2 = {best logit, second-best logit}.
int decode_step(OrModel& M, int token, int pos, double* logits_out, double* hidden_out,
                double* top2) {
  const OrDesc& d = M.d;
  const int H = d.hidden, D = d.head_dim, HQ = d.n_q_heads, HKV = d.n_kv_heads, F = d.ffn;
  const int group = HQ / HKV;
  const int nt = d.n_threads;
  std::vector<double> h(H), xn(H), q(HQ * D), k(HKV * D), v(HKV * D), att(HQ * D), tmp(H),
      g(F), u(F), a(F);

  dequant_row(d.embed, H, token, h.data());  // embedding = row `token` of the tied matrix
  if (hidden_out) std::copy(h.begin(), h.end(), hidden_out);

  for (int l = 0; l < d.n_layers; ++l) {
    const OrLayer& L = M.layers[l];
    rmsnorm(h.data(), L.ln_in, H, d.rms_eps, xn.data());
    gemv(L.q, HQ * D, H, xn.data(), q.data(), nt);
    gemv(L.k, HKV * D, H, xn.data(), k.data(), nt);
    gemv(L.v, HKV * D, H, xn.data(), v.data(), nt);
    for (int hh = 0; hh < HQ; ++hh) {  // QK-norm, then RoPE
      std::vector<double> t(D);
      rmsnorm(&q[hh * D], L.q_norm, D, d.rms_eps, t.data());
      std::copy(t.begin(), t.end(), &q[hh * D]);
      rope(&q[hh * D], D, pos, d.rope_theta);
    }
    for (int hh = 0; hh < HKV; ++hh) {
      std::vector<double> t(D);
      rmsnorm(&k[hh * D], L.k_norm, D, d.rms_eps, t.data());
      std::copy(t.begin(), t.end(), &k[hh * D]);
      rope(&k[hh * D], D, pos, d.rope_theta);
      for (int i = 0; i < D; ++i) {  // the cache holds bf16
        M.kcache[M.kv_index(l, hh, pos) + i] = bf16_encode(k[hh * D + i]);
        M.vcache[M.kv_index(l, hh, pos) + i] = bf16_encode(v[hh * D + i]);
      }
    }
    for (int hh = 0; hh < HQ; ++hh) {  // GQA: q head hh reads kv head hh / group
      int kvh = hh / group;
      attend(&q[hh * D], &M.kcache[M.kv_index(l, kvh, 0)], &M.vcache[M.kv_index(l, kvh, 0)],
             pos + 1, D, &att[hh * D]);
    }
    gemv(L.o, H, HQ * D, att.data(), tmp.data(), nt);
    for (int i = 0; i < H; ++i) h[i] += tmp[i];
    rmsnorm(h.data(), L.ln_post, H, d.rms_eps, xn.data());
    gemv(L.gate, F, H, xn.data(), g.data(), nt);
    gemv(L.up, F, H, xn.data(), u.data(), nt);
    for (int i = 0; i < F; ++i) a[i] = silu(g[i]) * u[i];
    gemv(L.down, H, F, a.data(), tmp.data(), nt);
    for (int i = 0; i < H; ++i) h[i] += tmp[i];
    if (hidden_out) std::copy(h.begin(), h.end(), hidden_out + (size_t)(l + 1) * H);
  }
  rmsnorm(h.data(), d.final_norm, H, d.rms_eps, xn.data());
  std::vector<double> logits(d.vocab);
  gemv(d.embed, d.vocab, H, xn.data(), logits.data(), nt);
  int best = argmax_lowest(logits.data(), d.vocab);
  if (top2) {
    double second = -std::numeric_limits<double>::infinity();
    for (int i = 0; i < d.vocab; ++i)
      if (i != best) second = std::max(second, logits[i]);
    top2[0] = logits[best];
    top2[1] = second;
  }
  if (logits_out) std::copy(logits.begin(), logits.end(), logits_out);
  return best;
}

}  // namespace

// ------------------------------------------------------------------------------------------
// C entry points used by the Python test harness (oracle/oracle.py)
// ------------------------------------------------------------------------------------------
extern "C" {

double or_e4m3_value(int code) { return e4m3_value((uint8_t)code); }
int or_e4m3_encode(double v) { return e4m3_encode(v); }
double or_e2m1_value(int code) { return e2m1_value((uint8_t)code); }
int or_e2m1_encode(double v) { return e2m1_encode(v); }
double or_bf16_value(int bits) { return bf16_value((uint16_t)bits); }
int or_bf16_encode(double v) { return bf16_encode(v); }

void or_quant_fp8_row(const uint16_t* w, int rows, int cols, uint8_t* codes, float* scales,
                      int nthreads) {
  quant_fp8_row(w, rows, cols, codes, scales, nthreads);
}
void or_quant_fp8_row_bf16scale(const uint16_t* w, int rows, int cols, uint8_t* codes, float* scales,
                                int nthreads) {
  quant_fp8_row(w, rows, cols, codes, scales, nthreads, true);
}
void or_quant_nvfp4(const uint16_t* w, int rows, int cols, uint8_t* codes, uint8_t* bscales,
                    float* tscale, int nthreads) {
  quant_nvfp4(w, rows, cols, codes, bscales, tscale, nthreads);
}
void or_quant_nvfp4_mse(const uint16_t* w, int rows, int cols, uint8_t* codes, uint8_t* bscales,
                        float* tscale, int nthreads) {
  quant_nvfp4_mse(w, rows, cols, codes, bscales, tscale, nthreads);
}
void or_attend(const double* q, const uint16_t* K, const uint16_t* V, int n, int d, double* out) {
  attend(q, K, V, n, d, out);
}
int or_argmax(const double* x, int n) { return argmax_lowest(x, n); }
void or_dequant(const OrMat* m, int rows, int cols, double* out) {
  for (int r = 0; r < rows; ++r) dequant_row(*m, cols, r, out + (size_t)r * cols);
}
void or_gemv(const OrMat* m, int rows, int cols, const double* x, double* y, int nthreads) {
  gemv(*m, rows, cols, x, y, nthreads);
}
void or_rmsnorm(const double* x, const uint16_t* w, int n, double eps, double* out) {
  rmsnorm(x, w, n, eps, out);
}
void or_rope(double* x, int d, int pos, double theta) { rope(x, d, pos, theta); }
double or_silu(double z) { return silu(z); }

void* or_model_create(const OrDesc* d) {
  if (!d || d->n_layers <= 0 || d->hidden <= 0 || d->head_dim <= 0 || d->n_kv_heads <= 0 ||
      d->n_q_heads % d->n_kv_heads != 0 || d->head_dim % 2 != 0 || d->max_ctx <= 0)
    return nullptr;
  OrModel* M = new OrModel();
  M->d = *d;
  M->layers.assign(d->layers, d->layers + d->n_layers);
  M->d.layers = M->layers.data();
  size_t n = (size_t)d->n_layers * d->n_kv_heads * d->max_ctx * d->head_dim;
  M->kcache.assign(n, 0);
  M->vcache.assign(n, 0);
  return M;
}
void or_model_destroy(void* m) { delete (OrModel*)m; }

// Copy a prefilled bf16 cache for positions [0, n_pos) of every layer and kv head.
// Layout of k and v: [n_layers][n_kv_heads][n_pos][head_dim].
int or_model_set_kv(void* m, const uint16_t* k, const uint16_t* v, int n_pos) {
  OrModel* M = (OrModel*)m;
  if (n_pos < 0 || n_pos > M->d.max_ctx) return -1;
  const OrDesc& d = M->d;
  for (int l = 0; l < d.n_layers; ++l)
    for (int h = 0; h < d.n_kv_heads; ++h)
      for (int t = 0; t < n_pos; ++t) {
        size_t src = (((size_t)l * d.n_kv_heads + h) * n_pos + t) * d.head_dim;
        std::memcpy(&M->kcache[M->kv_index(l, h, t)], k + src, d.head_dim * 2);
        std::memcpy(&M->vcache[M->kv_index(l, h, t)], v + src, d.head_dim * 2);
      }
  return 0;
}

// Read back positions [0, n_pos) of the cache in the same layout.
int or_model_get_kv(void* m, uint16_t* k, uint16_t* v, int n_pos) {
  OrModel* M = (OrModel*)m;
  if (n_pos < 0 || n_pos > M->d.max_ctx) return -1;
  const OrDesc& d = M->d;
  for (int l = 0; l < d.n_layers; ++l)
    for (int h = 0; h < d.n_kv_heads; ++h)
      for (int t = 0; t < n_pos; ++t) {
        size_t dst = (((size_t)l * d.n_kv_heads + h) * n_pos + t) * d.head_dim;
        std::memcpy(k + dst, &M->kcache[M->kv_index(l, h, t)], d.head_dim * 2);
        std::memcpy(v + dst, &M->vcache[M->kv_index(l, h, t)], d.head_dim * 2);
      }
  return 0;
}

int or_model_step(void* m, int token, int pos, double* logits, double* hidden, double* top2) {
  OrModel* M = (OrModel*)m;
  if (token < 0 || token >= M->d.vocab || pos < 0 || pos >= M->d.max_ctx) return -1;
  return decode_step(*M, token, pos, logits, hidden, top2);
}

}  // extern "C"
