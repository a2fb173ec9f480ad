// Host-side checks shared by the C entry points (defined in mk_api.cu), so that mk_create and
// mk_decode_step_static reject the same inputs with the same codes and texts (mk_last_error(NULL)).
#pragma once
#include "../../include/mk.h"
#include "mk_internal.h"

namespace mk {

// Shape family, 1 <= n_layers <= max_layers, vocab, max_ctx, eps and theta.
int check_config(const mk_config* c, int max_layers);
// The current device: at least 64 SMs, cooperative launch, one resident decode CTA per SM, and
// max_ctx within its attention window. On success *grid / *max_units receive the decode grid and
// the attention units per KV head.
int check_device(const mk_config* c, int* grid, int* max_units);
// Every matrix (format, 16-byte alignment, scales, shape), the per-layer format rules, the norm
// weights, the tied embedding and the final norm; fills dl[0 .. n_layers) on success.
int check_weights(const mk_config* c, const mk_weights* w, DLayer* dl);

}  // namespace mk
