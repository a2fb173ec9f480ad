/* mk.h -- C ABI of libmk.so, a single-GPU batch-1 decode engine for Qwen3-0.6B-shaped
 * transformers on NVIDIA GB300 (sm_103a).
 *
 * One call of mk_decode_step runs ONE persistent kernel that executes every layer and the
 * LM-head argmax, so one launch produces one token (monolith page, "Why it's exciting", first
 * bullet: a single persistent launch per decode step, with the upstream LM-head kernels folded in;
 * "Design decisions", sync experiment 5).
 *
 * Conventions for every entry point below:
 *  - Pointers named *_dev are device pointers; the caller allocates and owns them and keeps them
 *    alive for as long as the library may read or write them. Pointers named *_host are host
 *    pointers. `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *  - Calls return MK_OK (0) or a negative MK_E* code; they never abort the process.
 *  - No entry point allocates device memory except where stated; the model's workspace is a
 *    caller-owned device buffer of mk_workspace_bytes() bytes.
 *  - All weight matrices are row-major with rows = output features, cols = input features
 *    ("canonical packed form"); see mk_mat.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status codes */
#define MK_OK 0
#define MK_EINVAL (-1)       /* bad shape, format, alignment, token or position */
#define MK_ECUDA (-2)        /* a CUDA runtime call failed (text in mk_last_error) */
#define MK_ETIMEOUT (-3)     /* a device-side wait exceeded its deadline; the step was abandoned */
#define MK_ENORESIDENT (-4)  /* the persistent grid cannot be made co-resident on this GPU */
#define MK_ENOTRACE (-5)     /* X-ray requested but the model was created without it */
#define MK_EBOUNDS (-6)      /* bounds-checking build only: a device access out of range was skipped */

/* ---------------------------------------------------------------- weight formats
 * MK_BF16:    data = bf16 [rows][cols]; scale = NULL.
 * MK_FP8_ROW: data = OCP FP8 E4M3 bytes [rows][cols]; scale = fp32 [rows], one per output row;
 *             w = e4m3(code) * scale[row]  ("FP8 format", monolith page, "Design decisions").
 * MK_NVFP4:   data = E2M1 codes [rows][cols/2], element 2j in the low nibble of byte j;
 *             scale = E4M3 bytes [rows][cols/16], one per 16 consecutive inputs of a row;
 *             tensor_scale = fp32; w = e2m1(code) * e4m3(block scale) * tensor_scale
 *             ("NVFP4 format", monolith page, "Design decisions"; E2M1 grid: TSCT super-kernel
 *             page, section 3b).
 * Every data/scale pointer must be 16-byte aligned. */
enum mk_fmt { MK_BF16 = 0, MK_FP8_ROW = 1, MK_NVFP4 = 2 };

typedef struct {
  const void* data;   /* device */
  const void* scale;  /* device or NULL (bf16) */
  float tensor_scale; /* NVFP4 only */
  int fmt;            /* enum mk_fmt */
} mk_mat;

/* Model shape. This build supports the Qwen3-0.6B shape family: hidden 1024, 16 query heads,
 * 8 KV heads of width 128, FFN 3072 (model bullet, monolith page, "Upstream facts"); any
 * 1 <= n_layers <= 40, 1 <= vocab < 2^24, 1 <= max_ctx <= mk_max_context(). */
typedef struct {
  int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab, max_ctx;
  float rope_theta; /* 1e6 for Qwen3 */
  float rms_eps;    /* 1e-6 for Qwen3 */
} mk_config;

/* One decoder layer. q/k/v must share one format, and gate/up must share one format.
 * Norm weights are bf16 device vectors: ln_in/ln_post [hidden], q_norm/k_norm [head_dim]. */
typedef struct {
  mk_mat q, k, v, o, gate, up, down;
  const void *ln_in, *ln_post, *q_norm, *k_norm;
} mk_layer;

/* The tied embedding / LM-head matrix [vocab][hidden] is MK_BF16 or MK_FP8_ROW (the NVFP4 variant
 * keeps its LM head in FP8: monolith page, "Design decisions", NVFP4 format). */
typedef struct {
  const mk_layer* layers; /* host array of n_layers entries (copied by mk_create) */
  mk_mat embed;
  const void* final_norm; /* bf16 [hidden], device */
} mk_weights;

typedef struct mk_model mk_model; /* opaque; library-owned host object */

/* mk_create flags */
#define MK_FLAG_XRAY 1u /* keep per-CTA per-phase timestamps of the last step (mk_trace_dump) */
/* MK_FLAG_XRAY plus sub-phase marks inside each phase (kind 4 records, SM clock only): a finer
 * split of a phase at a higher cost (the marks slow a token by several per cent). */
#define MK_FLAG_XRAY_MARKS 4u
/* Keep the o_proj GEMV step at every context length. By default, on a decode grid of 128 CTAs
 * and where every layer's W_o has one format, steps whose context fits one attention unit
 * (pos < 288) fold the O-projection into attention: every CTA attends for one q head and
 * multiplies the output by its 128 x 128 block of W_o (repacked into the workspace by mk_create),
 * and the 16 heads' partial sums meet in order-independent integer accumulators, which removes
 * one step and one exchange a layer. The results equal the unfolded step's within fp32 rounding
 * and are deterministic. */
#define MK_FLAG_NO_FOLD 8u

/* ---------------------------------------------------------------- model lifetime */

/* Largest max_ctx this build accepts on the current device (attention splits the context into
 * at most one unit per SM, each holding up to 288 positions in shared memory). */
int mk_max_context(void);

/* CTAs of the persistent decode grid on the current device (one per SM, at most 128), or 0 when
 * the device cannot be queried. mk_gemv and mk_stream_read use the same grid. */
int mk_decode_grid(void);

/* Bytes of device workspace a model needs: bf16 KV cache [n_layers][n_kv][max_ctx][head_dim] for
 * keys and for values, a RoPE cos/sin table, activations, sync counters, an optional per-layer
 * hidden-state buffer and, with MK_FLAG_XRAY, the trace buffer. Returns 0 on a bad config.
 * An addition of this library (the pages have no counterpart): it lets the caller own every
 * device allocation. */
size_t mk_workspace_bytes(const mk_config* cfg, unsigned flags);

/* Validate the config and weights, lay out the caller's zeroed-or-not workspace (it is cleared
 * here), upload the layer table and build the RoPE table, all on `stream`. The weights and the
 * workspace must outlive the model. On success *out receives the handle. */
int mk_create(const mk_config* cfg, const mk_weights* w, void* workspace_dev, size_t workspace_bytes,
              void* stream, unsigned flags, mk_model** out);

void mk_destroy(mk_model* m);

/* Text of the last error on this model (or of the last mk_create failure when m == NULL). */
const char* mk_last_error(const mk_model* m);

/* ---------------------------------------------------------------- decoding */

/* One decode step: embed `token`, write its K/V at position `pos`, attend over 0..pos in every
 * layer, and return the argmax of the logits (lowest index among equal maxima) in
 * *next_token_host. If logits_dev != NULL, the fp32 logits [vocab] are written there.
 * Positions < pos must already be filled (by earlier steps or through mk_kv_cache).
 * Synchronises `stream` once at the end. Deterministic for identical inputs. */
int mk_decode_step(mk_model* m, int32_t token, int32_t pos, int32_t* next_token_host, float* logits_dev);

/* n greedy steps without host round trips: step i (0-based) runs at position pos0 + i on the
 * token produced by step i-1 (step 0 on first_token); every launch reads its input token from
 * device memory. tokens_dev (device int32 [n]) receives the produced tokens. Does not
 * synchronise; errors of the device steps are reported by the next mk_sync. */
int mk_decode_greedy(mk_model* m, int32_t first_token, int32_t pos0, int32_t n, int32_t* tokens_dev);

/* One decode launch without a host round trip: the input token is read from token_dev (device
 * int32), the produced token is written to next_dev (device int32), optional logits to
 * logits_dev. Does not synchronise; device-side errors are reported by the next mk_sync. */
int mk_decode_next(mk_model* m, const int32_t* token_dev, int32_t pos, int32_t* next_dev, float* logits_dev);

/* Wait for the model's stream and report any device-side status (e.g. MK_ETIMEOUT). */
int mk_sync(mk_model* m);

/* Device pointers to layer `layer`'s bf16 K and V caches, each [n_kv_heads][max_ctx][head_dim],
 * for prefilling or inspecting the cache. An addition of this library (the pages have no
 * counterpart); the cache itself is kept in bf16 as the monolith page's "Design decisions" (KV
 * cache) fix it. Returns MK_EINVAL for a NULL model or a layer out of range. */
int mk_kv_cache(mk_model* m, int layer, void** k_dev, void** v_dev);

/* Copy the residual stream of the last step into out_dev (device fp32 [(n_layers+1)][hidden]):
 * row 0 = embedding output, row l+1 = residual after layer l. An addition of this library for
 * per-layer parity checks (the pages have no counterpart). Synchronises the model's stream;
 * MK_EINVAL for NULL arguments, MK_ECUDA if the copy fails. */
int mk_debug_hidden(mk_model* m, float* out_dev);

/* X-ray: copy the last step's trace into host_buf (the in-kernel timing of the monolith page,
 * "Design decisions", "Timing": %globaltimer, clock64 and %smid stamped per block per phase; and
 * its "M2: X-ray" milestone). Records are 24 bytes: u64 globaltimer, u64 clock64, u32 smid,
 * u16 cta, u8 phase, u8 kind (0 phase begin, 1 phase end, 2 wait begin, 3 wait end, 4 sub-phase
 * mark carrying only clock64); one row of 2048 records per CTA, ended by a record of kind 255
 * where it is not full. host_buf must hold grid * 2048 * 24 bytes (MK_EINVAL otherwise);
 * *written receives the bytes copied. Synchronises the model's stream. Returns MK_ENOTRACE if the
 * model was created without MK_FLAG_XRAY. */
int mk_trace_dump(mk_model* m, void* host_buf, size_t cap, size_t* written);

/* Test hook: make CTA `cta` skip its signal after phase `phase` of layer 0 in the next steps, so
 * that every wait on it runs out; with timeout_ms the device deadline of every wait. Pass
 * cta = -1 to disable. The failed step returns MK_ETIMEOUT and the model stays usable. */
int mk_debug_fault(mk_model* m, int cta, int phase, int timeout_ms);

/* Race-detection aid (an addition of this library; the pages have no counterpart): with seed != 0,
 * every CTA of the following steps waits a pseudo-random 0 .. 20 us (a hash of the seed, the CTA,
 * the layer and the step, timed with %globaltimer) before each step, so the CTAs reach every
 * exchange in a different order; a correct step gives bit-identical results. seed = 0 turns it
 * off. */
int mk_debug_stress(mk_model* m, uint32_t seed);

/* ---------------------------------------------------------------- building blocks */

/* Quantise a bf16 matrix [rows][cols] into MK_FP8_ROW on the device: scale[r] = fp32(absmax/448),
 * code = E4M3 round-to-nearest-even, saturating, of fp32(w / scale[r]); an all-zero row gives
 * scale 0 and zero codes. codes_dev: [rows][cols] bytes; scales_dev: fp32 [rows]. */
int mk_pack_fp8_row(const void* w_bf16_dev, int rows, int cols, void* codes_dev, float* scales_dev, void* stream);

/* MK_FP8_ROW with bf16 row scales (the monolith page, "Design decisions", FP8 format, allows an
 * fp32 or a bf16 scale): scale[r] = bf16_RNE(fp32(absmax/448)), stored widened in the same fp32
 * array (its low 16 bits are zero), code = E4M3 round-to-nearest-even, saturating, of
 * fp32(w / scale[r]); a row whose scale rounded down may saturate its maximum at 448. Same
 * arguments, layouts and errors as mk_pack_fp8_row. */
int mk_pack_fp8_row_bf16scale(const void* w_bf16_dev, int rows, int cols, void* codes_dev, float* scales_dev,
                              void* stream);

/* Quantise a bf16 matrix into MK_NVFP4 on the device (cols a multiple of 16):
 * t = fp32(amax/2688); block scale b = E4M3_RNE(fp32(amax_block / fp32(6 t))); code =
 * E2M1_RNE_satfinite(fp32(w / fp32(e4m3(b) * t))). tscale_dev (device fp32) receives t; it is
 * also used as the amax accumulator while the call runs. */
int mk_pack_nvfp4(const void* w_bf16_dev, int rows, int cols, void* codes_dev, void* bscales_dev,
                  float* tscale_dev, void* stream);

/* MK_NVFP4 with a per-block scale search (the monolith page, "Design decisions", NVFP4 format:
 * round to nearest plus a block-scale choice that minimises the squared error). t as in
 * mk_pack_nvfp4. Every E4M3 code b in 0 .. 0x7E is tried for each block: its codes are formed
 * with the mk_pack_nvfp4 quotient rule (all zero when fp32(e4m3(b) * t) is 0) and its error is
 * sum_j (w_j - e2m1(code_j) * e4m3(b) * t)^2 in double, in element order, without fused
 * multiply-add; the least error wins, ties to the smaller b (an all-zero block keeps b = 0).
 * Same arguments, layouts and errors as mk_pack_nvfp4 (MK_EINVAL for NULL pointers or cols not
 * a positive multiple of 16). */
int mk_pack_nvfp4_mse(const void* w_bf16_dev, int rows, int cols, void* codes_dev, void* bscales_dev,
                      float* tscale_dev, void* stream);

/* y = W x with the same streaming dequant-GEMV the megakernel uses, as one persistent launch.
 * x_dev: fp32 [cols]; y_dev: fp32 [rows]; cols a multiple of 1024 and at most 4096. */
int mk_gemv(const mk_mat* w, int rows, int cols, const float* x_dev, float* y_dev, void* stream);

/* Streaming-read probe: read `bytes` (multiple of 16 * 1024 * mk_decode_grid()) from buf_dev once
 * with bulk copies into shared memory, on `stream`. Used to measure achievable HBM bandwidth. */
int mk_stream_read(const void* buf_dev, size_t bytes, void* stream);

/* Run the hardware conversions on every input, for checking them against a CPU table:
 * f16_from_e4m3 [65536] = cvt.rn.f16x2.e4m3x2 of every 16-bit pair; f16_from_e2m1 [256] =
 * cvt.rn.f16x2.e2m1x2 of every byte; e4m3_from_f32 [n/2] and e2m1_from_f32 [n/2] = the
 * saturating encoders applied to pairs (in[2i], in[2i+1]) of in_dev [n]. All device buffers;
 * any output may be NULL. */
int mk_probe_cvt(uint32_t* f16_from_e4m3_dev, uint32_t* f16_from_e2m1_dev, const float* in_dev, int n,
                 uint16_t* e4m3_from_f32_dev, uint8_t* e2m1_from_f32_dev, void* stream);

/* ---------------------------------------------------------------- batched verify
 * The batched speculative-verify step (monolith page, "Upstream facts", tensor cores and ISA, and
 * the throughput bullets: batch-1 decode does not use tensor cores, a batched verify would): k given
 * tokens at positions pos0 .. pos0 + k - 1 run through every layer and the LM head in ONE persistent
 * launch that reads each weight byte once for all k, with the GEMMs on the tcgen05 tensor cores
 * (bf16 layers as bf16; FP8 and NVFP4 layers as their exact f16 values; every activation split into
 * a 16-bit high and low part, fp32 accumulation), causal attention over the k new positions, and
 * one argmax per position. The result is what k teacher-forced mk_decode_step calls give, within
 * the parity tolerances; the keys and values of the k positions are written to the model's cache. */

/* Most tokens one verify launch takes. */
#define MK_VERIFY_MAX 8

/* Bytes of device workspace mk_verify_attach needs for model m (a 16-bit repacked copy of every
 * weight matrix laid out for the tensor cores, about 2 bytes per weight, plus exchange buffers). */
size_t mk_verify_workspace_bytes(const mk_model* m);

/* Prepare m for mk_verify_step: repack its weights into workspace_dev (caller-owned, at least
 * mk_verify_workspace_bytes(m) bytes, 16-byte aligned; it must outlive m). Needs the decode grid of
 * 128 CTAs (MK_ENORESIDENT otherwise) and layers that are all bf16 or all quantised (MK_EINVAL).
 * Synchronises the model's stream. */
int mk_verify_attach(mk_model* m, void* workspace_dev, size_t workspace_bytes);

/* One verify launch: tokens_dev (device int32 [k], 1 <= k <= MK_VERIFY_MAX) are the inputs at
 * positions pos0 .. pos0 + k - 1 (pos0 + k <= max_ctx and <= 1024; positions < pos0 must be in the
 * cache); next_dev (device int32 [k]) receives the argmax after each position (lowest index among
 * equal maxima) and logits_dev, if not NULL, the fp32 logits [k][vocab]. Does not synchronise;
 * device-side errors are reported by the next mk_sync. MK_EINVAL for bad arguments or a model
 * without mk_verify_attach. */
int mk_verify_step(mk_model* m, const int32_t* tokens_dev, int32_t k, int32_t pos0, int32_t* next_dev,
                   float* logits_dev);

/* ---------------------------------------------------------------- allocation-free step */

/* Largest max_ctx mk_decode_step_static accepts. */
#define MK_STATIC_MAX_CTX 4352

/* One decode step that allocates nothing. The pages have no counterpart: it is mk_decode_step
 * without a model object or workspace, for callers that cannot allocate device memory at the
 * moment they decode: a host framework that owns every device allocation and hands its plug-ins
 * only fixed buffers, a process whose device footprint is fixed when it starts (a memory budget on
 * a shared GPU), or a latency-critical loop that cannot afford cudaMalloc's implicit device-wide
 * synchronisation. The caller passes the weights (as for mk_create, checked the same way), the
 * bf16 KV cache as two device buffers k_dev, v_dev, each holding at least
 * n_layers * n_kv_heads * cfg->max_ctx * head_dim elements laid out
 * [n_layers][n_kv_heads][cfg->max_ctx][head_dim] (the library cannot check their size: a smaller
 * buffer is read and written out of bounds), the token and position, and receives the next token
 * in *next_token_host (and the fp32 logits in logits_dev if not NULL).
 * The kernel's scratch (sync words, activation exchange buffers, attention partials, layer table
 * and RoPE table, about 2.6 MB) lives in one fixed device array that every GPU loading the library
 * holds until the process exits; cfg->max_ctx <= MK_STATIC_MAX_CTX and n_layers <= 40, larger
 * values are rejected with MK_EINVAL. The first call on a device does a one-time set-up: it looks
 * the array's device address up on that device (the device must be current) and checks the
 * device as mk_create does; make that first call before any stream capture begins. A call with a
 * new rope_theta rebuilds the RoPE table. Calls share the array, which keeps the last call's
 * contents (the kernel clears the sync words it uses at the end of every step): two calls that
 * overlap on one GPU race and give wrong results. Synchronises `stream` before it returns.
 * Errors: MK_EINVAL, MK_ECUDA, MK_ETIMEOUT, MK_ENORESIDENT, with text in mk_last_error(NULL). */
int mk_decode_step_static(const mk_config* cfg, const mk_weights* w, void* k_dev, void* v_dev, int32_t token,
                          int32_t pos, int32_t* next_token_host, float* logits_dev, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
