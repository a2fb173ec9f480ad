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
constexpr int VN = 16;       // MMA N: B rows 0..7 hold the tokens' high parts, rows 8..15 the low parts
constexpr int V_NSLOT = 6;   // weight ring slots (SLOT bytes each)
constexpr int V_GRID = 128;  // the verify grid (one CTA per SM)
constexpr int V_HEAD_CHUNK = 128;  // LM-head rows per MMA (M = 128)
constexpr int V_MAXPOS = 1024;     // positions a verify step attends over, at most (pos0 + k)

// The GEMM steps of a layer and their per-CTA operand blocks. Each CTA's rows of a step are stored
// as 16-bit values in "boxes" of 64 input columns: box j holds R8 rows (the CTA's rows rounded up to
// a multiple of 8, zero-padded) x 128 bytes, 128-byte swizzled, so one bulk copy puts a run of boxes
// into shared memory in the layout the MMA reads. Boxes of a block are contiguous.
enum VStep { VS_QKV = 0, VS_O = 1, VS_GU = 2, VS_DOWN = 3, VS_COUNT = 4 };
__host__ __device__ inline int v_rows8(int step) { return step == VS_QKV ? 32 : (step == VS_GU ? 48 : 8); }
__host__ __device__ inline int v_cols(int step) { return step == VS_O ? QROWS : (step == VS_DOWN ? FFN : HID); }
__host__ __device__ inline size_t v_block_bytes(int step) { return (size_t)v_rows8(step) * v_cols(step) * 2; }
// Bytes of one layer's blocks (all steps, all CTAs) and the offset of step s's blocks in a layer.
__host__ __device__ inline size_t v_layer_bytes() {
  return (size_t)V_GRID * (v_block_bytes(0) + v_block_bytes(1) + v_block_bytes(2) + v_block_bytes(3));
}
__host__ __device__ inline size_t v_step_offset(int s) {
  size_t o = 0;
  for (int i = 0; i < s; ++i) o += (size_t)V_GRID * v_block_bytes(i);
  return o;
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
