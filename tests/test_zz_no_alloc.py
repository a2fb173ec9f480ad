"""GPU: the allocation-free entry point (mk_decode_step_static) against the regular one.

mk_decode_step_static serves callers that cannot allocate device memory at the moment they
decode: a host framework that owns every device allocation and hands out only fixed buffers, a
process whose device footprint is fixed at start-up, or a loop that cannot afford cudaMalloc's
implicit synchronisation. Its scratch lives in a fixed device array inside the library and keeps
the previous call's contents. It runs the same kernel as mk_decode_step on the same inputs, so its
tokens, logits and KV cache must be bit-identical to the regular step's, over consecutive calls
that share that array, and across a change of rope_theta (which rebuilds the RoPE table). This
file is collected last so that, if it fails, every other test has already run.
"""
import dataclasses

import pytest
import torch

from quantized_gemv_gb300 import mk
from quantized_gemv_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


def _caches(cfg):
    n = cfg.n_layers * cfg.n_kv_heads * cfg.max_ctx * cfg.head_dim
    return (torch.zeros(n, dtype=torch.bfloat16, device="cuda"), torch.zeros(n, dtype=torch.bfloat16, device="cuda"))


def _run_pair(cfg, packed, k_cache, v_cache, tokens):
    """Steps at positions 0.. on both entry points (teacher-forced on `tokens`); asserts bit-equal
    tokens and logits at every step. The allocation-free step keeps the o_proj GEMV step (its
    fixed array holds no repacked W_o), so it is compared with a model that keeps it too."""
    model = mk.Model(cfg, packed, flags=mk.MK_FLAG_NO_FOLD)
    for pos, tok in enumerate(tokens):
        la = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
        lb = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
        na = model.decode_step(tok, pos, la)
        nb = mk.decode_step_static(cfg, packed, k_cache, v_cache, tok, pos, lb)
        assert na == nb, (pos, na, nb)
        assert torch.equal(la.view(torch.int32), lb.view(torch.int32)), pos
    n = len(tokens)
    for l in range(cfg.n_layers):
        kt, vt = model.kv_cache(l)
        ks = k_cache.view(cfg.n_layers, cfg.n_kv_heads, cfg.max_ctx, cfg.head_dim)[l]
        vs = v_cache.view(cfg.n_layers, cfg.n_kv_heads, cfg.max_ctx, cfg.head_dim)[l]
        assert torch.equal(kt[:, :n].view(torch.int16), ks[:, :n].view(torch.int16))
        assert torch.equal(vt[:, :n].view(torch.int16), vs[:, :n].view(torch.int16))
    model.close()


@pytest.mark.parametrize("variant", ["fp8", "bf16"])
def test_static_step_matches_regular_step(variant):
    cfg = S.ModelConfig(n_layers=2, vocab=4099, max_ctx=256)
    packed = mk.pack_model(S.master_weights(cfg, seed=91), S.format_map(variant))
    k_cache, v_cache = _caches(cfg)
    # two calls in a row on one array, then more: the scratch carries over between them
    _run_pair(cfg, packed, k_cache, v_cache, [17, 4000, 3, 1234])


def test_static_step_follows_rope_theta():
    """A second theta rebuilds the static RoPE table, and going back to the first rebuilds it again."""
    cfg_a = S.ModelConfig(n_layers=1, vocab=1031, max_ctx=128)
    cfg_b = dataclasses.replace(cfg_a, rope_theta=1e4)
    packed = mk.pack_model(S.master_weights(cfg_a, seed=93), S.format_map("fp8"))
    for cfg in (cfg_a, cfg_b, cfg_a):
        k_cache, v_cache = _caches(cfg)
        _run_pair(cfg, packed, k_cache, v_cache, [5, 77, 901])


def test_static_step_rejects_oversized_context():
    cfg = S.ModelConfig(n_layers=1, vocab=64, max_ctx=mk.MK_STATIC_MAX_CTX + 64)
    packed = mk.pack_model(S.master_weights(cfg, seed=92), S.format_map("bf16"))
    kc, vc = _caches(cfg)
    with pytest.raises(mk.MkError) as ei:
        mk.decode_step_static(cfg, packed, kc, vc, 1, 0)
    assert ei.value.code == mk.MK_EINVAL
    assert "MK_STATIC_MAX_CTX" in str(ei.value)


def test_static_step_rejects_small_cache():
    cfg = S.ModelConfig(n_layers=1, vocab=64, max_ctx=64)
    packed = mk.pack_model(S.master_weights(cfg, seed=94), S.format_map("bf16"))
    kc, vc = _caches(cfg)
    with pytest.raises(ValueError):
        mk.decode_step_static(cfg, packed, kc[:-1], vc, 1, 0)
    with pytest.raises(ValueError):
        mk.decode_step_static(cfg, packed, kc, vc.float(), 1, 0)
