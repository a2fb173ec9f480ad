// mk_decode_step_static: one decode step that allocates nothing.
//
// Some callers cannot allocate device memory at the moment they decode: a host framework that owns
// every device allocation and hands its plug-ins only fixed buffers, a process that must not grow
// its device footprint after start-up (a memory budget fixed when it was admitted to a shared GPU),
// or a latency-critical loop where cudaMalloc's implicit device-wide synchronisation is not
// acceptable. They still own the weights and the KV cache, but cannot provide the decode kernel's
// scratch (sync words, the tagged activation buffers, attention partials, the layer table and the
// RoPE table). This file keeps that scratch in one file-scope __device__ array of fixed size, so the
// step needs no workspace and no model object.
//
// Limits and sharing: every GPU that loads the library holds the array until the process exits.
// All calls on a device share it and it keeps the previous call's contents, so two calls that run
// at the same time on one GPU (different streams, or different host threads without ordering)
// race on it and give wrong results. The kernel resets the sync words it uses at the end of every
// step; after a failed step they are cleared here. The first call on a device looks the array's
// device address up with that device current (cudaGetSymbolAddress); make that first call before
// any stream capture begins. Every call synchronises the caller's stream before it returns.
#include <cuda_runtime.h>

#include <mutex>

#include "mk_host.h"

using namespace mk;

namespace {

constexpr int STATIC_MAX_LAYERS = MAX_LAYERS;
constexpr int STATIC_MAX_CTX = MK_STATIC_MAX_CTX;

struct __align__(256) StaticScratch {
  SyncBlock sync;
  DLayer layers[STATIC_MAX_LAYERS];
  llword h_mlp[HID];
  llword h_attn[HID];
  llword qkv[QKV_ROWS];
  llword att[QROWS];
  llword act[FFN];
  float attp[NKVH * MAXC * 2 * PART_STRIDE];
  float rope_cos[STATIC_MAX_CTX * (HD / 2)];
  float rope_sin[STATIC_MAX_CTX * (HD / 2)];
};

// The scratch itself (zero-initialised when the module loads).
__device__ __align__(256) StaticScratch g_static_scratch;

// Per-device state of the host side.
struct DevState {
  bool ready = false;
  StaticScratch* ptr = nullptr;  // device address of g_static_scratch on this device
  float rope_theta = 0.f;        // theta the RoPE table was built for (0 = not built)
  uint32_t steps = 0;
  int grid = 0;
};
constexpr int MAX_DEVICES = 64;
DevState g_dev[MAX_DEVICES];
std::mutex g_mu;
int fail(int code, const char* msg) {
  set_global_error(msg);
  return code;
}

}  // namespace

extern "C" {

int mk_decode_step_static(const mk_config* c, const mk_weights* w, void* kv_k_dev, void* kv_v_dev, int32_t token,
                          int32_t pos, int32_t* next_token_host, float* logits_dev, void* stream) {
  if (!c || !w || !kv_k_dev || !kv_v_dev || !next_token_host) return fail(MK_EINVAL, "NULL argument");
  int rc;
  if ((rc = check_config(c, STATIC_MAX_LAYERS)) != MK_OK) return rc;
  if (c->max_ctx > STATIC_MAX_CTX)
    return fail(MK_EINVAL, "max_ctx must be at most MK_STATIC_MAX_CTX for the static entry point");
  if (token < 0 || token >= c->vocab || pos < 0 || pos >= c->max_ctx) return fail(MK_EINVAL, "token or pos out of range");
  if (((uintptr_t)kv_k_dev & 15u) || ((uintptr_t)kv_v_dev & 15u)) return fail(MK_EINVAL, "KV cache not 16-byte aligned");
  // the layer table of this call, checked like mk_create's (pageable source: the copy below
  // completes before this call returns)
  DLayer dl[STATIC_MAX_LAYERS];
  if ((rc = check_weights(c, w, dl)) != MK_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return fail(MK_ECUDA, "no current device");
  cudaStream_t st = (cudaStream_t)stream;

  std::lock_guard<std::mutex> lock(g_mu);
  DevState& D = g_dev[dev];
  if (!D.ready) {  // set-up, once per device, with that device current
    int grid = 0, mu = 0;
    if ((rc = check_device(c, &grid, &mu)) != MK_OK) return rc;
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return fail(MK_ECUDA, cudaGetErrorString(e));
    D.ptr = static_cast<StaticScratch*>(p);
    D.grid = grid;
    D.ready = true;
  }
  const int max_units = (D.grid / NKVH) > MAXC ? MAXC : (D.grid / NKVH);
  if (c->max_ctx > max_units * UNIT_POS) return fail(MK_EINVAL, "max_ctx exceeds this device's attention window");
  StaticScratch* S = D.ptr;
  cudaError_t e = cudaSuccess;
  if (D.rope_theta != c->rope_theta) {  // (re)build the RoPE table for this theta
    if (launch_rope_table(S->rope_cos, S->rope_sin, STATIC_MAX_CTX, c->rope_theta, st)) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(MK_ECUDA, cudaGetErrorString(e));
    D.rope_theta = c->rope_theta;
  }
  e = cudaMemcpyAsync(S->layers, dl, sizeof(DLayer) * c->n_layers, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return fail(MK_ECUDA, cudaGetErrorString(e));

  KParams p = {};
  p.layers = S->layers;
  p.n_layers = c->n_layers;
  p.embed.data = (const uint8_t*)w->embed.data;
  p.embed.scale = (const uint8_t*)w->embed.scale;
  p.embed.tscale = w->embed.tensor_scale;
  p.embed.fmt = w->embed.fmt;
  p.final_norm = (const uint16_t*)w->final_norm;
  p.vocab = c->vocab;
  p.max_ctx = c->max_ctx;
  p.eps = c->rms_eps;
  p.kc = (uint16_t*)kv_k_dev;
  p.vc = (uint16_t*)kv_v_dev;
  p.rope_cos = S->rope_cos;
  p.rope_sin = S->rope_sin;
  p.h_mlp = S->h_mlp;
  p.h_attn = S->h_attn;
  p.qkv = S->qkv;
  p.att = S->att;
  p.act = S->act;
  p.attp = S->attp;
  p.sync = &S->sync;
  p.hidden_dbg = nullptr;
  p.logits = logits_dev;
  p.trace = nullptr;
  p.token = token;
  p.token_ptr = nullptr;
  p.pos = pos;
  p.next_out = nullptr;
  p.units = (pos + 1 <= UNIT_POS) ? 1 : max_units;
  D.steps = (D.steps + 1) & 0x03FFFFFFu;
  if (D.steps == 0) D.steps = 1;
  p.tagbase = D.steps * 64u;
  p.timeout_ns = 500000000ull;
  p.fault_cta = -1;
  p.fault_phase = -1;
  if (launch_decode(p, D.grid, 0, st)) return fail(MK_ECUDA, cudaGetErrorString(cudaGetLastError()));
  // the step's status and token (SyncBlock::status then ::tok, 64 words)
  uint32_t hs[64];
  e = cudaMemcpyAsync(hs, S->sync.status, sizeof hs, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail(MK_ECUDA, cudaGetErrorString(e));
  if (hs[0] != 0) {  // a failed step leaves sync words behind: clear them for the next call
    cudaMemsetAsync(&S->sync, 0, sizeof(SyncBlock), st);
    cudaStreamSynchronize(st);
    return fail(hs[0] == 4 ? MK_EINVAL : MK_ETIMEOUT, "device step failed");
  }
  *next_token_host = (int32_t)hs[32];
  return MK_OK;
}

}  // extern "C"
