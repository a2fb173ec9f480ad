"""GPU: the allocation-free entry point (mk_decode_step_static) against the regular one.

mk_decode_step_static is for callers that cannot allocate device memory when they decode (for
example code running while a stream is captured, or a host framework that hands out only fixed
buffers): its scratch lives in a fixed device array inside the library. It must give the same
tokens and logits as mk_decode_step on the same weights, over consecutive calls that share that
array. This file is collected last so that, if it fails, every other test has already run.
"""
import numpy as np
import pytest
import torch

from quantized_gemv_gb300 import mk
from quantized_gemv_gb300 import synthetic as S
from tests.gpu_util import LOGIT_ATOL

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant", ["fp8", "bf16"])
def test_static_step_matches_regular_step(variant):
    cfg = S.ModelConfig(n_layers=2, vocab=4099, max_ctx=256)
    packed = mk.pack_model(S.master_weights(cfg, seed=91), S.format_map(variant))
    model = mk.Model(cfg, packed)
    n = cfg.n_layers * cfg.n_kv_heads * cfg.max_ctx * cfg.head_dim
    k_cache = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    v_cache = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    tok = 17
    for pos in range(4):  # consecutive calls: the shared scratch carries over between them
        la = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
        lb = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
        na = model.decode_step(tok, pos, la)
        nb = mk.decode_step_static(cfg, packed, k_cache, v_cache, tok, pos, lb)
        assert na == nb
        assert float(np.max(np.abs(la.cpu().numpy() - lb.cpu().numpy()))) <= LOGIT_ATOL
        tok = na
    # the caller's cache holds what the model's own cache holds
    for l in range(cfg.n_layers):
        kt, vt = model.kv_cache(l)
        ks = k_cache.view(cfg.n_layers, cfg.n_kv_heads, cfg.max_ctx, cfg.head_dim)[l]
        vs = v_cache.view(cfg.n_layers, cfg.n_kv_heads, cfg.max_ctx, cfg.head_dim)[l]
        assert torch.equal(kt[:, :4], ks[:, :4]) and torch.equal(vt[:, :4], vs[:, :4])
    model.close()


def test_static_step_rejects_oversized_context():
    cfg = S.ModelConfig(n_layers=1, vocab=64, max_ctx=mk.MK_STATIC_MAX_CTX + 64)
    packed = mk.pack_model(S.master_weights(cfg, seed=92), S.format_map("bf16"))
    n = cfg.n_layers * cfg.n_kv_heads * cfg.max_ctx * cfg.head_dim
    kc = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mk.MkError) as ei:
        mk.decode_step_static(cfg, packed, kc, kc, 1, 0)
    assert ei.value.code == mk.MK_EINVAL
