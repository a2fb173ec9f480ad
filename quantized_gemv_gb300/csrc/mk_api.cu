// Host implementation of the C ABI declared in include/mk.h.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "mk_host.h"
#include "mk_verify.h"

using namespace mk;

struct mk_model {
  mk_config cfg;
  unsigned flags;
  cudaStream_t stream;
  int grid;
  int max_units;
  // workspace carve-up (device)
  SyncBlock* sync;
  DLayer* dlayers;
  llword *h_mlp, *h_attn, *qkv, *att, *act;
  float* attp;
  uint32_t steps;  // launches so far; tags of a launch start at 64 * steps
  float *rope_cos, *rope_sin;
  uint16_t *kc, *vc;
  float* hidden_dbg;
  TraceRec* trace;
  bool fold_o;                 // W_o repacked for the folded O-projection (used at short contexts)
  uint8_t* wo_rep;
  size_t wo_lbytes;
  unsigned long long* acc;     // count words, two sets of [n_layers][HID] (launch parity)
  DMat embed;
  const uint16_t* final_norm;
  // host
  uint32_t* host_status;  // pinned: SyncBlock::status and ::tok lines (64 words)
  unsigned long long timeout_ns;
  int fault_cta, fault_phase;
  uint32_t stress_seed = 0;
  std::string err;
  // batched verify (mk_verify_attach)
  std::vector<DLayer> hlayers;  // host copy of the layer table
  uint8_t* vw = nullptr;        // repacked layer blocks
  uint8_t* vhead = nullptr;     // repacked LM-head blocks
  uint32_t* vx = nullptr;       // two sentinel exchange sets (launch parity)
  int vlayer_bf16 = 0, vhead_bf16 = 0;
  uint32_t vsteps = 0;
};

static thread_local std::string g_create_err;

static int set_err(mk_model* m, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (m) m->err = buf;
  else g_create_err = buf;
  return code;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

void mk::set_global_error(const char* msg) { g_create_err = msg; }

struct Layout {
  size_t sync, layers, h_mlp, h_attn, qkv, att, act, attp, rope_cos, rope_sin, kc, vc, hidden, trace, acc, wo, total;
};

static int device_grid(int* grid) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  *grid = decode_grid_for(sms);
  return 0;
}

static int max_units_for(int grid) {
  int u = grid / NKVH;
  return u > MAXC ? MAXC : u;
}

static bool layout_of(const mk_config* c, unsigned flags, int grid, Layout* L) {
  if (!c || c->n_layers < 1 || c->max_ctx < 1 || c->vocab < 1) return false;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  const size_t kv = (size_t)c->n_layers * NKVH * c->max_ctx * HD * sizeof(uint16_t);
  L->sync = take(sizeof(SyncBlock));
  L->layers = take(sizeof(DLayer) * c->n_layers);
  L->h_mlp = take(HID * sizeof(llword));
  L->h_attn = take(HID * sizeof(llword));
  L->qkv = take(QKV_ROWS * sizeof(llword));
  L->att = take(QROWS * sizeof(llword));
  L->act = take(FFN * sizeof(llword));
  L->attp = take((size_t)NKVH * MAXC * 2 * PART_STRIDE * 4);
  L->rope_cos = take((size_t)c->max_ctx * (HD / 2) * 4);
  L->rope_sin = take((size_t)c->max_ctx * (HD / 2) * 4);
  L->hidden = take((size_t)(c->n_layers + 1) * HID * 4);
  L->trace = take((flags & (MK_FLAG_XRAY | MK_FLAG_XRAY_MARKS)) ? (size_t)grid * TRACE_PER_CTA * sizeof(TraceRec) : 0);
  L->kc = take(kv);
  L->vc = take(kv);
  // folded O-projection: count words (two sets) and W_o repacked per (head, slice) block, sized
  // for bf16, the widest format
  const bool fold = !(flags & MK_FLAG_NO_FOLD) && grid == FOLD_GRID;
  L->acc = take(fold ? 2 * (size_t)c->n_layers * HID * sizeof(unsigned long long) : 0);
  L->wo = take(fold ? (size_t)c->n_layers * NQH * FOLD_SLICES * wo_block_bytes(0) : 0);
  L->total = o;
  return true;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static int check_mat(const mk_mat& m, int rows, int cols, const char* name, bool allow_nvfp4) {
  if (m.fmt < MK_BF16 || m.fmt > MK_NVFP4) return set_err(nullptr, MK_EINVAL, "%s: bad format %d", name, m.fmt);
  if (m.fmt == MK_NVFP4 && !allow_nvfp4) return set_err(nullptr, MK_EINVAL, "%s: NVFP4 not allowed here", name);
  if (!m.data || !aligned16(m.data)) return set_err(nullptr, MK_EINVAL, "%s: data NULL or not 16-byte aligned", name);
  if (m.fmt != MK_BF16 && (!m.scale || !aligned16(m.scale)))
    return set_err(nullptr, MK_EINVAL, "%s: scale NULL or not 16-byte aligned", name);
  if (cols % 1024 != 0 || rows < 1) return set_err(nullptr, MK_EINVAL, "%s: unsupported shape", name);
  return MK_OK;
}

static DMat to_dmat(const mk_mat& m) {
  DMat d;
  d.data = (const uint8_t*)m.data;
  d.scale = (const uint8_t*)m.scale;
  d.tscale = m.tensor_scale;
  d.fmt = m.fmt;
  return d;
}

// ------------------------------------------------------------------ checks shared by the entry points
// (mk_create and mk_decode_step_static reject the same inputs with the same codes and messages)
int mk::check_config(const mk_config* c, int max_layers) {
  if (!c) return set_err(nullptr, MK_EINVAL, "config NULL");
  if (c->hidden != HID || c->n_q_heads != NQH || c->n_kv_heads != NKVH || c->head_dim != HD || c->ffn != FFN)
    return set_err(nullptr, MK_EINVAL, "only the Qwen3-0.6B shape family (1024/16/8/128/3072) is supported");
  if (c->n_layers < 1 || c->n_layers > max_layers || c->vocab < 1 || c->vocab >= (1 << 24) || c->max_ctx < 1)
    return set_err(nullptr, MK_EINVAL, "bad n_layers/vocab/max_ctx");
  if (!(c->rms_eps > 0.f) || !(c->rope_theta > 0.f)) return set_err(nullptr, MK_EINVAL, "bad eps/theta");
  return MK_OK;
}

int mk::check_device(const mk_config* c, int* grid_out, int* max_units_out) {
  int grid;
  if (device_grid(&grid)) return set_err(nullptr, MK_ECUDA, "cannot query the device");
  if (grid < 64) return set_err(nullptr, MK_ENORESIDENT, "need at least 64 SMs, device has %d", grid);
  const int max_units = max_units_for(grid);
  if (c->max_ctx > max_units * UNIT_POS)
    return set_err(nullptr, MK_EINVAL, "max_ctx %d exceeds %d on this device", c->max_ctx, max_units * UNIT_POS);
  int dev = 0, coop = 0, bps = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return set_err(nullptr, MK_ECUDA, "no current device");
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (!coop) return set_err(nullptr, MK_ENORESIDENT, "device lacks cooperative launch");
  if (decode_occupancy(&bps) || bps < 1)
    return set_err(nullptr, MK_ENORESIDENT, "persistent CTA (%d threads, %d B smem) does not fit an SM", NTHREADS,
                   decode_smem_bytes());
  *grid_out = grid;
  *max_units_out = max_units;
  return MK_OK;
}

int mk::check_weights(const mk_config* c, const mk_weights* w, DLayer* dl) {
  if (!w || !w->layers) return set_err(nullptr, MK_EINVAL, "weights NULL");
  int rc;
  for (int l = 0; l < c->n_layers; ++l) {
    const mk_layer& ly = w->layers[l];
    const mk_mat* mats[7] = {&ly.q, &ly.k, &ly.v, &ly.o, &ly.gate, &ly.up, &ly.down};
    const int rws[7] = {QROWS, KVROWS, KVROWS, HID, FFN, FFN, HID};
    const int cls[7] = {HID, HID, HID, QROWS, HID, HID, FFN};
    const char* names[7] = {"q", "k", "v", "o", "gate", "up", "down"};
    for (int i = 0; i < 7; ++i) {
      if ((rc = check_mat(*mats[i], rws[i], cls[i], names[i], true)) != MK_OK) return rc;
      dl[l].m[i] = to_dmat(*mats[i]);
    }
    if (ly.q.fmt != ly.k.fmt || ly.q.fmt != ly.v.fmt)
      return set_err(nullptr, MK_EINVAL, "layer %d: q, k, v must share one format", l);
    if (ly.gate.fmt != ly.up.fmt) return set_err(nullptr, MK_EINVAL, "layer %d: gate and up must share one format", l);
    if (!ly.ln_in || !ly.ln_post || !ly.q_norm || !ly.k_norm)
      return set_err(nullptr, MK_EINVAL, "layer %d: norm weight NULL", l);
    dl[l].ln_in = (const uint16_t*)ly.ln_in;
    dl[l].ln_post = (const uint16_t*)ly.ln_post;
    dl[l].q_norm = (const uint16_t*)ly.q_norm;
    dl[l].k_norm = (const uint16_t*)ly.k_norm;
  }
  if ((rc = check_mat(w->embed, c->vocab, HID, "embed", false)) != MK_OK) return rc;
  if (!w->final_norm) return set_err(nullptr, MK_EINVAL, "final_norm NULL");
  return MK_OK;
}

extern "C" {

int mk_decode_grid(void) {
  int grid;
  return device_grid(&grid) ? 0 : grid;
}

int mk_max_context(void) {
  int grid;
  if (device_grid(&grid)) return 0;
  return max_units_for(grid) * UNIT_POS;
}

size_t mk_workspace_bytes(const mk_config* cfg, unsigned flags) {
  int grid;
  if (device_grid(&grid)) return 0;
  Layout L = {};
  if (!layout_of(cfg, flags, grid, &L)) return 0;
  return L.total;
}

const char* mk_last_error(const mk_model* m) { return m ? m->err.c_str() : g_create_err.c_str(); }

int mk_create(const mk_config* c, const mk_weights* w, void* ws, size_t ws_bytes, void* stream, unsigned flags,
              mk_model** out) {
  if (!out) return set_err(nullptr, MK_EINVAL, "out is NULL");
  *out = nullptr;
  int rc, grid, max_units;
  if ((rc = check_config(c, MAX_LAYERS)) != MK_OK) return rc;
  if ((rc = check_device(c, &grid, &max_units)) != MK_OK) return rc;
  Layout L = {};
  layout_of(c, flags, grid, &L);
  if (!ws || ws_bytes < L.total || !aligned16(ws))
    return set_err(nullptr, MK_EINVAL, "workspace too small or unaligned (%zu < %zu)", ws_bytes, L.total);
  std::vector<DLayer> dl(c->n_layers);
  if ((rc = check_weights(c, w, dl.data())) != MK_OK) return rc;

  mk_model* m = new mk_model();
  m->hlayers = dl;
  m->cfg = *c;
  m->flags = flags;
  m->stream = (cudaStream_t)stream;
  m->grid = grid;
  m->max_units = max_units;
  uint8_t* base = (uint8_t*)ws;
  m->sync = (SyncBlock*)(base + L.sync);
  m->dlayers = (DLayer*)(base + L.layers);
  m->h_mlp = (llword*)(base + L.h_mlp);
  m->h_attn = (llword*)(base + L.h_attn);
  m->qkv = (llword*)(base + L.qkv);
  m->att = (llword*)(base + L.att);
  m->act = (llword*)(base + L.act);
  m->steps = 0;
  m->attp = (float*)(base + L.attp);
  m->rope_cos = (float*)(base + L.rope_cos);
  m->rope_sin = (float*)(base + L.rope_sin);
  m->kc = (uint16_t*)(base + L.kc);
  m->vc = (uint16_t*)(base + L.vc);
  m->hidden_dbg = (float*)(base + L.hidden);
  m->trace = (flags & (MK_FLAG_XRAY | MK_FLAG_XRAY_MARKS)) ? (TraceRec*)(base + L.trace) : nullptr;
  m->embed = to_dmat(w->embed);
  m->final_norm = (const uint16_t*)w->final_norm;
  // the folded O-projection needs the grid of 128 and one W_o format in every layer
  m->fold_o = !(flags & MK_FLAG_NO_FOLD) && grid == FOLD_GRID;
  for (int l = 1; m->fold_o && l < c->n_layers; ++l) m->fold_o = w->layers[l].o.fmt == w->layers[0].o.fmt;
  m->acc = m->fold_o ? (unsigned long long*)(base + L.acc) : nullptr;
  m->wo_rep = m->fold_o ? base + L.wo : nullptr;
  m->wo_lbytes = m->fold_o ? (size_t)NQH * FOLD_SLICES * wo_block_bytes(w->layers[0].o.fmt) : 0;
  m->timeout_ns = 500000000ull;
  m->fault_cta = -1;
  m->fault_phase = -1;
  if (cudaMallocHost(&m->host_status, 64 * sizeof(uint32_t)) != cudaSuccess) {
    delete m;
    return set_err(nullptr, MK_ECUDA, "cudaMallocHost failed");
  }
  cudaError_t e = cudaMemsetAsync(ws, 0, L.total, m->stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(m->dlayers, dl.data(), sizeof(DLayer) * c->n_layers, cudaMemcpyHostToDevice, m->stream);
  if (e == cudaSuccess && launch_rope_table(m->rope_cos, m->rope_sin, c->max_ctx, c->rope_theta, m->stream))
    e = cudaGetLastError();
  for (int l = 0; m->fold_o && e == cudaSuccess && l < c->n_layers; ++l)
    if (launch_repack_o(w->layers[l].o.data, w->layers[l].o.scale, w->layers[l].o.fmt, m->wo_rep + l * m->wo_lbytes,
                        m->stream))
      e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaStreamSynchronize(m->stream);
  if (e != cudaSuccess) {
    set_err(nullptr, MK_ECUDA, "mk_create: %s", cudaGetErrorString(e));
    cudaFreeHost(m->host_status);
    delete m;
    return MK_ECUDA;
  }
  *out = m;
  return MK_OK;
}

void mk_destroy(mk_model* m) {
  if (!m) return;
  if (m->host_status) cudaFreeHost(m->host_status);
  delete m;
}

// Attention units per KV head for a step at `pos`: one unit when the whole context fits one
// unit's shared-memory window (no merge step), else one unit per (SM / KV head).
static int units_for(const mk_model* m, int pos) {
  return (pos + 1 <= UNIT_POS) ? 1 : m->max_units;
}

static KParams base_params(mk_model* m) {
  KParams p = {};
  p.layers = m->dlayers;
  p.n_layers = m->cfg.n_layers;
  p.embed = m->embed;
  p.final_norm = m->final_norm;
  p.vocab = m->cfg.vocab;
  p.max_ctx = m->cfg.max_ctx;
  p.eps = m->cfg.rms_eps;
  p.kc = m->kc;
  p.vc = m->vc;
  p.rope_cos = m->rope_cos;
  p.rope_sin = m->rope_sin;
  p.h_mlp = m->h_mlp;
  p.h_attn = m->h_attn;
  p.qkv = m->qkv;
  p.att = m->att;
  p.act = m->act;
  p.attp = m->attp;
  p.sync = m->sync;
  p.hidden_dbg = m->hidden_dbg;
  p.trace = m->trace;
  p.timeout_ns = m->timeout_ns;
  p.fault_cta = m->fault_cta;
  p.fault_phase = m->fault_phase;
  p.stress_seed = m->stress_seed;
  return p;
}

// X-ray level of the model's launches (see launch_decode).
static int xray_level(const mk_model* m) {
  return m->trace == nullptr ? 0 : ((m->flags & MK_FLAG_XRAY_MARKS) ? 2 : 1);
}

// Tags of one launch: 64 * (launch number) + layer; never 0 (the workspace starts zeroed).
// Also sets the launch's folded O-projection parameters: folded where the context fits one
// attention unit; the count words alternate between two sets by launch parity, and every launch
// clears the set the next one uses.
static uint32_t next_tagbase(mk_model* m, KParams& p) {
  m->steps = (m->steps + 1) & 0x03FFFFFFu;
  if (m->steps == 0) m->steps = 1;
  p.fold_o = (m->fold_o && p.units == 1) ? 1 : 0;
  p.wo_rep = m->wo_rep;
  p.wo_lbytes = m->wo_lbytes;
  const size_t set = (size_t)m->cfg.n_layers * HID;
  p.acc = m->acc ? m->acc + (m->steps & 1u) * set : nullptr;
  p.acc_zero = m->acc ? m->acc + ((m->steps + 1u) & 1u) * set : nullptr;
  return m->steps * 64u;
}

// Read the device status; on a failed step clear the sync block so the model stays usable.
static int collect_status(mk_model* m, int32_t* next_token) {
  cudaError_t e = cudaMemcpyAsync(m->host_status, m->sync->status, 64 * sizeof(uint32_t), cudaMemcpyDeviceToHost,
                                  m->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(m->stream);
  if (e != cudaSuccess) return set_err(m, MK_ECUDA, "decode: %s", cudaGetErrorString(e));
  const uint32_t st = m->host_status[0];
  if (st == 4) {
    set_err(m, MK_EINVAL, "a device step read an out-of-range input token");
    cudaMemsetAsync(m->sync, 0, sizeof(SyncBlock), m->stream);
    if (m->acc) cudaMemsetAsync(m->acc, 0, 2 * (size_t)m->cfg.n_layers * HID * sizeof(unsigned long long), m->stream);
    if (m->vx) cudaMemsetAsync(m->vx, 0xFF, 2 * v_x_words(m->cfg.n_layers) * sizeof(uint32_t), m->stream);
    cudaStreamSynchronize(m->stream);
    return MK_EINVAL;
  }
  if (st == 5) {
    const uint32_t d = m->host_status[1];
    set_err(m, MK_EBOUNDS, "out-of-range device access skipped (bounds-checking build): site %u index %u", d >> 24,
            d & 0xFFFFFFu);
    cudaMemsetAsync(m->sync, 0, sizeof(SyncBlock), m->stream);
    if (m->acc) cudaMemsetAsync(m->acc, 0, 2 * (size_t)m->cfg.n_layers * HID * sizeof(unsigned long long), m->stream);
    if (m->vx) cudaMemsetAsync(m->vx, 0xFF, 2 * v_x_words(m->cfg.n_layers) * sizeof(uint32_t), m->stream);
    cudaStreamSynchronize(m->stream);
    return MK_EBOUNDS;
  }
  if (st != 0) {
    const uint32_t d = m->host_status[1];
    set_err(m, MK_ETIMEOUT, "device wait timed out: phase %u layer %u cta %u%s%s", d & 0xFF, (d >> 8) & 0xFF,
            (d >> 16) & 0x7FFF, (d & 0x80000000u) ? " (weight stream)" : "",
            m->host_status[3] ? "; a CTA exited with bulk copies still in flight" : "");
    cudaMemsetAsync(m->sync, 0, sizeof(SyncBlock), m->stream);
    if (m->acc) cudaMemsetAsync(m->acc, 0, 2 * (size_t)m->cfg.n_layers * HID * sizeof(unsigned long long), m->stream);
    if (m->vx) cudaMemsetAsync(m->vx, 0xFF, 2 * v_x_words(m->cfg.n_layers) * sizeof(uint32_t), m->stream);
    cudaStreamSynchronize(m->stream);
    return MK_ETIMEOUT;
  }
  if (next_token) *next_token = (int32_t)m->host_status[32];
  return MK_OK;
}

int mk_decode_step(mk_model* m, int32_t token, int32_t pos, int32_t* next_token_host, float* logits_dev) {
  if (!m) return MK_EINVAL;
  if (token < 0 || token >= m->cfg.vocab) return set_err(m, MK_EINVAL, "token %d out of range", token);
  if (pos < 0 || pos >= m->cfg.max_ctx) return set_err(m, MK_EINVAL, "pos %d out of range", pos);
  KParams p = base_params(m);
  p.token = token;
  p.token_ptr = nullptr;
  p.pos = pos;
  p.next_out = nullptr;
  p.logits = logits_dev;
  p.units = units_for(m, pos);
  p.tagbase = next_tagbase(m, p);
  if (launch_decode(p, m->grid, xray_level(m), m->stream))
    return set_err(m, MK_ECUDA, "launch: %s", cudaGetErrorString(cudaGetLastError()));
  return collect_status(m, next_token_host);
}

int mk_decode_greedy(mk_model* m, int32_t first_token, int32_t pos0, int32_t n, int32_t* tokens_dev) {
  if (!m || n < 0 || !tokens_dev) return MK_EINVAL;
  if (first_token < 0 || first_token >= m->cfg.vocab) return set_err(m, MK_EINVAL, "token out of range");
  if (pos0 < 0 || (long long)pos0 + n > m->cfg.max_ctx) return set_err(m, MK_EINVAL, "positions out of range");
  KParams p = base_params(m);
  for (int i = 0; i < n; ++i) {
    p.token = first_token;
    p.token_ptr = i == 0 ? nullptr : tokens_dev + (i - 1);
    p.pos = pos0 + i;
    p.next_out = tokens_dev + i;
    p.logits = nullptr;
    p.units = units_for(m, p.pos);
    p.tagbase = next_tagbase(m, p);
    if (launch_decode(p, m->grid, xray_level(m), m->stream))
      return set_err(m, MK_ECUDA, "launch: %s", cudaGetErrorString(cudaGetLastError()));
  }
  return MK_OK;
}

int mk_decode_next(mk_model* m, const int32_t* token_dev, int32_t pos, int32_t* next_dev, float* logits_dev) {
  if (!m || !token_dev || !next_dev) return MK_EINVAL;
  if (pos < 0 || pos >= m->cfg.max_ctx) return set_err(m, MK_EINVAL, "pos %d out of range", pos);
  KParams p = base_params(m);
  p.token = 0;
  p.token_ptr = token_dev;
  p.pos = pos;
  p.next_out = next_dev;
  p.logits = logits_dev;
  p.units = units_for(m, pos);
  p.tagbase = next_tagbase(m, p);
  if (launch_decode(p, m->grid, xray_level(m), m->stream))
    return set_err(m, MK_ECUDA, "launch: %s", cudaGetErrorString(cudaGetLastError()));
  return MK_OK;
}

int mk_sync(mk_model* m) {
  if (!m) return MK_EINVAL;
  return collect_status(m, nullptr);
}

int mk_kv_cache(mk_model* m, int layer, void** k, void** v) {
  if (!m || layer < 0 || layer >= m->cfg.n_layers) return MK_EINVAL;
  const size_t off = (size_t)layer * NKVH * m->cfg.max_ctx * HD;
  if (k) *k = m->kc + off;
  if (v) *v = m->vc + off;
  return MK_OK;
}

int mk_debug_hidden(mk_model* m, float* out) {
  if (!m || !out) return MK_EINVAL;
  cudaError_t e = cudaMemcpyAsync(out, m->hidden_dbg, (size_t)(m->cfg.n_layers + 1) * HID * 4,
                                  cudaMemcpyDeviceToDevice, m->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(m->stream);
  return e == cudaSuccess ? MK_OK : set_err(m, MK_ECUDA, "%s", cudaGetErrorString(e));
}

int mk_trace_dump(mk_model* m, void* host_buf, size_t cap, size_t* written) {
  if (!m) return MK_EINVAL;
  if (!m->trace) return set_err(m, MK_ENOTRACE, "model created without MK_FLAG_XRAY");
  const size_t bytes = (size_t)m->grid * TRACE_PER_CTA * sizeof(TraceRec);
  if (!host_buf || cap < bytes) return set_err(m, MK_EINVAL, "trace buffer needs %zu bytes", bytes);
  cudaError_t e = cudaMemcpyAsync(host_buf, m->trace, bytes, cudaMemcpyDeviceToHost, m->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(m->stream);
  if (e != cudaSuccess) return set_err(m, MK_ECUDA, "%s", cudaGetErrorString(e));
  if (written) *written = bytes;
  return MK_OK;
}

int mk_debug_fault(mk_model* m, int cta, int phase, int timeout_ms) {
  if (!m) return MK_EINVAL;
  m->fault_cta = cta;
  m->fault_phase = phase;
  if (timeout_ms > 0) m->timeout_ns = (unsigned long long)timeout_ms * 1000000ull;
  return MK_OK;
}

int mk_debug_stress(mk_model* m, uint32_t seed) {
  if (!m) return MK_EINVAL;
  m->stress_seed = seed;
  return MK_OK;
}

// ------------------------------------------------------------------ batched verify
// Workspace layout of the verify path: repacked layer blocks, repacked LM-head blocks, two sentinel
// exchange sets.
static size_t verify_layout(const mk_model* m, size_t* head_off, size_t* x_off) {
  const size_t lw = align_up((size_t)m->cfg.n_layers * v_layer_bytes(), 256);
  const size_t hw = align_up((size_t)V_GRID * v_head_cta_bytes(m->cfg.vocab), 256);
  if (head_off) *head_off = lw;
  if (x_off) *x_off = lw + hw;
  return lw + hw + 2 * v_x_words(m->cfg.n_layers) * sizeof(uint32_t);
}

size_t mk_verify_workspace_bytes(const mk_model* m) { return m ? verify_layout(m, nullptr, nullptr) : 0; }

int mk_verify_attach(mk_model* m, void* ws, size_t ws_bytes) {
  if (!m) return MK_EINVAL;
  if (m->grid != V_GRID) return set_err(m, MK_ENORESIDENT, "the verify step needs a decode grid of %d CTAs", V_GRID);
  // one operand type per part: bf16 matrices stay bf16, FP8 and NVFP4 ones become exact f16
  const int lb = m->hlayers[0].m[0].fmt == MK_BF16;
  for (const DLayer& L : m->hlayers)
    for (int i = 0; i < 7; ++i)
      if ((L.m[i].fmt == MK_BF16) != (lb != 0))
        return set_err(m, MK_EINVAL, "verify: the layers mix bf16 and quantised matrices");
  size_t head_off, x_off;
  const size_t need = verify_layout(m, &head_off, &x_off);
  if (!ws || ws_bytes < need || !aligned16(ws))
    return set_err(m, MK_EINVAL, "verify workspace too small or unaligned (%zu < %zu)", ws_bytes, need);
  uint8_t* base = (uint8_t*)ws;
  m->vw = base;
  m->vhead = base + head_off;
  m->vx = (uint32_t*)(base + x_off);
  m->vlayer_bf16 = lb;
  m->vhead_bf16 = m->embed.fmt == MK_BF16;
  m->vsteps = 0;
  cudaError_t e = cudaSuccess;
  for (int l = 0; l < m->cfg.n_layers && e == cudaSuccess; ++l)
    if (launch_verify_repack_layer(m->hlayers[l], lb, m->vw + (size_t)l * v_layer_bytes(), m->stream))
      e = cudaGetLastError();
  if (e == cudaSuccess && launch_verify_repack_head(m->embed, m->cfg.vocab, m->vhead_bf16, m->vhead, m->stream))
    e = cudaGetLastError();
  if (e == cudaSuccess)
    e = cudaMemsetAsync(m->vx, 0xFF, 2 * v_x_words(m->cfg.n_layers) * sizeof(uint32_t), m->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(m->stream);
  if (e != cudaSuccess) {
    m->vw = nullptr, m->vhead = nullptr, m->vx = nullptr;
    return set_err(m, MK_ECUDA, "mk_verify_attach: %s", cudaGetErrorString(e));
  }
  return MK_OK;
}

int mk_verify_step(mk_model* m, const int32_t* tokens_dev, int32_t k, int32_t pos0, int32_t* next_dev,
                   float* logits_dev) {
  if (!m || !tokens_dev || !next_dev) return MK_EINVAL;
  if (!m->vw) return set_err(m, MK_EINVAL, "mk_verify_attach was not called");
  if (k < 1 || k > VK) return set_err(m, MK_EINVAL, "k = %d outside 1..%d", k, VK);
  if (pos0 < 0 || (long long)pos0 + k > m->cfg.max_ctx || pos0 + k > V_MAXPOS)
    return set_err(m, MK_EINVAL, "positions %d..%d outside the cache or the verify window (%d)", pos0, pos0 + k - 1,
                   V_MAXPOS);
  VParams p = {};
  p.layers = m->dlayers;
  p.n_layers = m->cfg.n_layers;
  p.embed = m->embed;
  p.final_norm = m->final_norm;
  p.vocab = m->cfg.vocab;
  p.max_ctx = m->cfg.max_ctx;
  p.eps = m->cfg.rms_eps;
  p.vw = m->vw;
  p.vhead = m->vhead;
  p.layer_bf16 = m->vlayer_bf16;
  p.head_bf16 = m->vhead_bf16;
  p.kc = m->kc;
  p.vc = m->vc;
  p.rope_cos = m->rope_cos;
  p.rope_sin = m->rope_sin;
  p.tokens = tokens_dev;
  p.k = k;
  p.pos0 = pos0;
  p.next_out = next_dev;
  p.logits = logits_dev;
  m->vsteps += 1;
  const size_t w = v_x_words(m->cfg.n_layers);
  p.x = m->vx + (m->vsteps & 1u) * w;
  p.x_reset = m->vx + ((m->vsteps + 1u) & 1u) * w;
  p.sync = m->sync;
  p.timeout_ns = m->timeout_ns;
  if (launch_verify(p, m->stream)) return set_err(m, MK_ECUDA, "verify launch: %s", cudaGetErrorString(cudaGetLastError()));
  return MK_OK;
}

int mk_pack_fp8_row(const void* w, int rows, int cols, void* codes, float* scales, void* stream) {
  if (!w || !codes || !scales || rows < 1 || cols < 2 || cols % 2) return MK_EINVAL;
  return launch_pack_fp8(w, rows, cols, codes, scales, 0, stream) ? MK_ECUDA : MK_OK;
}

int mk_pack_fp8_row_bf16scale(const void* w, int rows, int cols, void* codes, float* scales, void* stream) {
  if (!w || !codes || !scales || rows < 1 || cols < 2 || cols % 2) return MK_EINVAL;
  return launch_pack_fp8(w, rows, cols, codes, scales, 1, stream) ? MK_ECUDA : MK_OK;
}

int mk_pack_nvfp4(const void* w, int rows, int cols, void* codes, void* bscales, float* tscale, void* stream) {
  if (!w || !codes || !bscales || !tscale || rows < 1 || cols < 16 || cols % 16) return MK_EINVAL;
  return launch_pack_nvfp4(w, rows, cols, codes, bscales, tscale, stream) ? MK_ECUDA : MK_OK;
}

int mk_pack_nvfp4_mse(const void* w, int rows, int cols, void* codes, void* bscales, float* tscale, void* stream) {
  if (!w || !codes || !bscales || !tscale || rows < 1 || cols < 16 || cols % 16) return MK_EINVAL;
  return launch_pack_nvfp4_mse(w, rows, cols, codes, bscales, tscale, stream) ? MK_ECUDA : MK_OK;
}

int mk_gemv(const mk_mat* w, int rows, int cols, const float* x, float* y, void* stream) {
  if (!w || !x || !y || rows < 1 || cols < 1024 || cols % 1024 || cols > XS_MAX) return MK_EINVAL;
  if (w->fmt < 0 || w->fmt > 2 || !w->data || !aligned16(w->data)) return MK_EINVAL;
  if (w->fmt != MK_BF16 && (!w->scale || !aligned16(w->scale))) return MK_EINVAL;
  int grid;
  if (device_grid(&grid)) return MK_ECUDA;
  return launch_gemv(to_dmat(*w), rows, cols, x, y, grid, stream) ? MK_ECUDA : MK_OK;
}

int mk_stream_read(const void* buf, size_t bytes, void* stream) {
  int grid;
  if (device_grid(&grid)) return MK_ECUDA;
  const size_t unit = (size_t)16384 * grid;
  if (!buf || !aligned16(buf) || bytes == 0 || bytes % unit) return MK_EINVAL;
  return launch_stream_read(buf, bytes, grid, stream) ? MK_ECUDA : MK_OK;
}

int mk_probe_cvt(uint32_t* a, uint32_t* b, const float* in, int n, uint16_t* e4, uint8_t* e2, void* stream) {
  if (n < 0 || (in && n % 2)) return MK_EINVAL;
  return launch_probe_cvt(a, b, in, n, e4, e2, stream) ? MK_ECUDA : MK_OK;
}

}  // extern "C"
