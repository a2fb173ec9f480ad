// Definitions shared by the kernels (mk_kernel.cu, mk_aux.cu) and the host ABI (mk_api.cu).
#pragma once
#include <cstddef>
#include <cstdint>

namespace mk {

// Qwen3-0.6B shape family (monolith page, "Upstream facts", model bullet).
constexpr int HID = 1024, NQH = 16, NKVH = 8, HD = 128, FFN = 3072;
constexpr int QROWS = NQH * HD;                 // 2048
constexpr int KVROWS = NKVH * HD;               // 1024
constexpr int QKV_ROWS = QROWS + 2 * KVROWS;    // 4096
constexpr int GQA = NQH / NKVH;                 // 2 query heads per KV head

// Persistent CTA shape: 8 consumer warps + 1 producer warp. Every GEMV phase of a CTA is small
// (tens of rows), so its time goes to per-warp bookkeeping as much as to math: fewer warps, each
// computing four rows at once, keep the SM's issue slots on the dot products. Nine warps leave
// 168 registers per thread (no spills: with shared memory taking most of the SM, spills miss L1).
constexpr int NCW = 8;
constexpr int NCT = NCW * 32;
constexpr int NTHREADS = NCT + 32;

// Shared-memory weight ring.
constexpr int SLOT = 16384;
constexpr int NSLOT = 12;
constexpr int MAX_LAYERS = 40;  // layer table held in each CTA's shared memory
constexpr int KVT = 32;                         // positions per KV tile (K 8 KB + V 8 KB)
constexpr int UNIT_TILES = 9;                   // KV tiles an attention unit holds at once
constexpr int UNIT_POS = KVT * UNIT_TILES;      // 288 positions per attention unit
constexpr int MAXC = 32;                        // attention units per KV head, upper bound
constexpr int XS_MAX = 4096;                    // floats of staged GEMV input
constexpr int PART_STRIDE = 132;                // floats per attention partial (m, l, pad, acc[128])

enum Phase { PH_QKV = 0, PH_ATTN = 1, PH_O = 2, PH_GATEUP = 3, PH_DOWN = 4, PH_HEAD = 5, PH_EMBED = 6,
             PH_WAIT = 7, PH_COUNT = 8 };
enum MatIdx { M_Q = 0, M_K, M_V, M_O, M_GATE, M_UP, M_DOWN };

struct DMat {
  const uint8_t* data;
  const uint8_t* scale;
  float tscale;
  int fmt;
};

struct DLayer {
  DMat m[7];
  const uint16_t* ln_in;
  const uint16_t* ln_post;
  const uint16_t* q_norm;
  const uint16_t* k_norm;
};

// Sync words, each on its own 128-byte line.
struct SyncBlock {
  uint32_t c[8][32];           // per-phase arrival counters (reset by the last CTA of a step)
  uint32_t grp[NKVH][32];      // attention units finished, per KV head
  unsigned long long key[16];  // packed (logit, index) argmax key
  uint32_t status[32];         // [0] status code, [1] detail word, [2] abort flag, [3] a CTA exited with
                               // bulk copies still in flight (its drain gave up)
  int32_t tok[32];             // [0] token produced by the last step
};

// X-ray record (24 bytes).
struct TraceRec {
  unsigned long long gtime;
  unsigned long long clk;
  uint32_t smid;
  uint16_t cta;
  uint8_t phase;
  uint8_t kind;  // 0 = phase begin, 1 = phase end, 2 = wait begin, 3 = wait end
};
constexpr int TRACE_PER_CTA = 2048;

// Activations cross SMs as 64-bit words {fp32 value (low), u32 tag (high)} stored with one
// single-copy-atomic 64-bit store: a consumer polls the words themselves until every one carries
// the tag of the (step, layer) it needs, so no fence, counter or second round trip is involved.
typedef unsigned long long llword;

struct KParams {
  const DLayer* layers;
  int n_layers;
  DMat embed;
  const uint16_t* final_norm;
  int vocab;
  int max_ctx;
  float eps;
  uint16_t* kc;          // bf16 [L][NKVH][max_ctx][HD]
  uint16_t* vc;
  const float* rope_cos; // [max_ctx][HD/2]
  const float* rope_sin;
  llword* h_mlp;         // residual after the MLP block (layer output) [HID]
  llword* h_attn;        // residual after the attention block [HID]
  llword* qkv;           // raw q|k|v [QKV_ROWS]
  llword* att;           // attention output [QROWS]
  llword* act;           // SwiGLU output [FFN]
  float* attp;           // attention partials [NKVH][MAXC][2][PART_STRIDE]
  SyncBlock* sync;
  float* hidden_dbg;     // nullable [(L+1)][HID]
  float* logits;         // nullable [vocab]
  TraceRec* trace;       // nullable [grid][TRACE_PER_CTA]
  int token;
  const int32_t* token_ptr;  // nullable: read the input token here instead
  int pos;
  int32_t* next_out;
  int units;             // attention units per KV head this step
  uint32_t tagbase;      // tag of layer l in this step = tagbase + l (unique per launch, never 0)
  unsigned long long timeout_ns;
  int fault_cta;         // test hook (-1 = off)
  int fault_phase;
  uint32_t stress_seed;  // test hook: nonzero = every CTA waits a seeded 0..20 us before each step
  // Folded O-projection (contexts of one attention unit, grid FOLD_GRID): every CTA b runs the
  // attention of q head b / FOLD_SLICES and multiplies its output by the 128 x 128 block of W_o
  // whose rows are [128 (b % FOLD_SLICES), +128) and whose columns are that head's; the partial
  // sums of the 16 heads meet in count words (see acc) that the gate/up step polls in place of
  // h_attn. 0: attention units and an o_proj GEMV step as above.
  int fold_o;
  const uint8_t* wo_rep;   // W_o repacked per (layer, head, slice) block, see wo_block_bytes()
  size_t wo_lbytes;        // bytes of one layer's blocks
  unsigned long long* acc;       // count words of this launch [n_layers][HID]
  unsigned long long* acc_zero;  // the other launch parity's count words, cleared by this launch
};

// Folded O-projection geometry: 16 q heads x 8 row slices of 128 rows = a grid of 128 CTAs.
constexpr int FOLD_SLICES = 8;
constexpr int FOLD_GRID = NQH * FOLD_SLICES;
constexpr int FOLD_ROWS = HID / FOLD_SLICES;  // 128 output rows per block
// Bytes of one repacked W_o block (FOLD_ROWS rows x HD columns): bf16 and FP8 codes row-major;
// NVFP4 codes row-major [128][64 B] followed by the E4M3 block scales [128][8 B].
__host__ __device__ inline int wo_block_bytes(int fmt) {
  return fmt == 0 ? FOLD_ROWS * HD * 2 : (fmt == 1 ? FOLD_ROWS * HD : FOLD_ROWS * (HD / 2 + HD / 16));
}
// Count words: a contribution v adds ((int64)round(v * 2^24) << 8) + 1 with one 64-bit integer
// atomic add, so the low byte counts the contributions and the rest holds their fixed-point sum
// (2^-24 resolution); integer addition makes the result independent of arrival order.
constexpr float COUNT_SCALE = 16777216.0f;

// CTAs of the persistent decode grid on a device with `sms` SMs (one CTA per SM): 128 where the
// device has them, so that every CTA's share of each exchanged vector (8 of the 1024 hidden rows,
// 24 of the 3072 FFN units, 32 q/k/v rows) is a whole number of 32-byte sectors; otherwise the
// largest multiple of 8 (one group per KV head).
inline int decode_grid_for(int sms) { return sms >= 128 ? 128 : (sms / NKVH) * NKVH; }

// Launchers (mk_kernel.cu / mk_aux.cu)
// xray: 0 = plain kernel, 1 = X-ray phase and wait stamps, 2 = stamps and sub-phase marks
int launch_decode(const KParams& p, int grid, int xray, void* stream);
int decode_smem_bytes();
int launch_gemv(const DMat& m, int rows, int cols, const float* x, float* y, int grid, void* stream);
int launch_stream_read(const void* buf, size_t bytes, int grid, void* stream);
int launch_rope_table(float* cosb, float* sinb, int max_ctx, float theta, void* stream);
int launch_pack_fp8(const void* w, int rows, int cols, void* codes, float* scales, int bf16_scale, void* stream);
int launch_pack_nvfp4(const void* w, int rows, int cols, void* codes, void* bscales, float* t, void* stream);
int launch_pack_nvfp4_mse(const void* w, int rows, int cols, void* codes, void* bscales, float* t, void* stream);
int launch_repack_o(const void* data, const void* scale, int fmt, void* dst, void* stream);
int launch_probe_cvt(uint32_t* a, uint32_t* b, const float* in, int n, uint16_t* e4, uint8_t* e2, void* stream);
int decode_occupancy(int* blocks_per_sm);
// Record an error text for mk_last_error(NULL) (mk_api.cu).
void set_global_error(const char* msg);

}  // namespace mk
