// The batched verify step: k <= VK given tokens at consecutive positions run through every layer
// and the LM head in one persistent launch, each weight byte read once for all k tokens, the
// GEMMs on the fifth-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
// Shared by the kernel (mk_verify.cu) and the host entry points (mk_api.cu).
#pragma once
#include <cstddef>
#include <cstdint>

#include "mk_internal.h"

namespace mk {

// The empty value of a sentinel exchange word: a NaN bit pattern that fp32 arithmetic never
// produces (computed NaNs are the canonical 0x7FFFFFFF), so no real value can be mistaken for it.
constexpr uint32_t X_EMPTY = 0xFFFFFFFFu;

constexpr int VK = 8;        // tokens per verify launch, at most
constexpr int VN = 16;       // B rows a segment: 0..7 the tokens' high parts, 8..15 the low parts
constexpr int V_NSLOT = 6;   // weight ring slots (SLOT bytes each)
constexpr int V_GRID = 128;  // the verify grid (one CTA per SM)
constexpr int V_HEAD_CHUNK = 128;  // LM-head rows per MMA (M = 128)
constexpr int V_MAXPOS = 1024;     // positions a verify step attends over, at most (pos0 + k)

// The GEMM steps of a layer and their per-CTA operand blocks. A CTA owns R whole rows of a step
// (all K inputs of each), split into S segments of KS = K / S inputs; its block is stored as
// 128-row tiles ("boxes") of 64 input columns, 16-bit values, 128-byte swizzled, where tile row
// L = seg * R + r holds row r's inputs seg * KS + 64 b .. + 63 (box b of KS / 64). S * R = 128, so
// every row of every MMA is a real weight row; the B operand holds, for segment seg, the k token
// vectors' inputs of that segment (rows 16 seg + t: high parts, 16 seg + 8 + t: low parts), so the
// diagonal blocks D[seg * R + r][16 seg + ...] of the product are row r's partial sums, which the
// epilogue adds in segment order. One box fills one ring slot (16 KB).
enum VStep { VS_QKV = 0, VS_O = 1, VS_GU = 2, VS_DOWN = 3, VS_COUNT = 4 };
constexpr int V_GU_CTAS = 96;  // gate/up: CTAs 0..95 own 32 FFN units (32 gate + 32 up rows) each
struct VStepGeom {
  int R, S, KS, KB, N;  // rows, segments, inputs a segment, boxes (KS / 64), MMA N (16 S)
};
__host__ __device__ inline VStepGeom v_step_geom(int step) {
  switch (step) {
    case VS_QKV: return {32, 4, 256, 4, 64};
    case VS_O: return {8, 16, 128, 2, 256};
    case VS_GU: return {64, 2, 512, 8, 32};
    default: return {8, 16, 192, 3, 256};
  }
}
__host__ __device__ inline int v_cols(int step) { return step == VS_O ? QROWS : (step == VS_DOWN ? FFN : HID); }
// Boxes of CTA c's block of a step (gate/up: none for CTAs V_GU_CTAS..).
__host__ __device__ inline int v_nbox(int step, int c) {
  return (step == VS_GU && c >= V_GU_CTAS) ? 0 : v_step_geom(step).KB;
}
constexpr size_t V_BOX = 16384;  // 128 rows x 64 columns x 2 bytes
// Bytes of one layer's blocks (all steps, all CTAs); steps are stored one after another, each as
// its CTAs' blocks in CTA order.
__host__ __device__ inline size_t v_step_bytes(int step) {
  const int ctas = step == VS_GU ? V_GU_CTAS : V_GRID;
  return (size_t)ctas * v_step_geom(step).KB * V_BOX;
}
__host__ __device__ inline size_t v_layer_bytes() {
  return v_step_bytes(VS_QKV) + v_step_bytes(VS_O) + v_step_bytes(VS_GU) + v_step_bytes(VS_DOWN);
}
// Offset of CTA c's block of step s within a layer.
__host__ __device__ inline size_t v_block_offset(int s, int c) {
  size_t o = 0;
  for (int i = 0; i < s; ++i) o += v_step_bytes(i);
  return o + (size_t)c * v_step_geom(s).KB * V_BOX;
}
// LM head: CTA c's rows split_range(vocab, V_GRID, c) in chunks of V_HEAD_CHUNK rows; every chunk
// gets a full V_HEAD_CHUNK x HID block (the last one zero-padded).
__host__ __device__ inline int v_head_chunks(int vocab) { return (vocab / V_GRID + 1 + V_HEAD_CHUNK - 1) / V_HEAD_CHUNK; }
__host__ __device__ inline size_t v_head_cta_bytes(int vocab) {
  return (size_t)v_head_chunks(vocab) * V_HEAD_CHUNK * HID * 2;
}

// Parameters of one verify launch.
struct VParams {
  const DLayer* layers;  // the model's layer table (canonical weights: scales, norms)
  int n_layers;
  DMat embed;
  const uint16_t* final_norm;
  int vocab, max_ctx;
  float eps;
  const uint8_t* vw;     // repacked layer blocks, n_layers * v_layer_bytes()
  const uint8_t* vhead;  // repacked LM-head blocks, V_GRID * v_head_cta_bytes(vocab)
  int layer_bf16, head_bf16;  // operand type of the layer steps / the LM head: 1 bf16, 0 f16
  uint16_t* kc;          // the model's bf16 KV cache [L][NKVH][max_ctx][HD]
  uint16_t* vc;
  const float* rope_cos;
  const float* rope_sin;
  const int32_t* tokens; // device int32[k]: the input token of each position
  int k, pos0;
  int32_t* next_out;     // device int32[k]: the argmax after each position
  float* logits;         // nullable device fp32 [k][vocab]
  uint32_t* x;           // this launch's sentinel exchange set, v_x_words(n_layers) words
  uint32_t* x_reset;     // the other set, refilled with X_EMPTY by this launch
  SyncBlock* sync;
  unsigned long long timeout_ns;
};

// Sentinel exchange words of one verify launch: per layer and token, q|k|v, attention output,
// h_attn, SwiGLU output and the layer output.
constexpr int V_XL = QKV_ROWS + QROWS + HID + FFN + HID;  // words per layer and token
__host__ __device__ inline size_t v_x_words(int n_layers) { return (size_t)n_layers * VK * V_XL; }

int launch_verify(const VParams& p, void* stream);
int verify_smem_bytes();
// Repack one layer's or the LM head's weights into the verify blocks (see above).
int launch_verify_repack_layer(const DLayer& L, int to_bf16, uint8_t* dst, void* stream);
int launch_verify_repack_head(const DMat& e, int vocab, int to_bf16, uint8_t* dst, void* stream);

}  // namespace mk
