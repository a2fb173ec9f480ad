"""GPU: the batched verify step (mk_verify_step, tensor cores) against the oracle.

One launch runs k given tokens at positions pos0 .. pos0 + k - 1 through every layer; its k argmaxes
and logits must be those of k teacher-forced oracle steps (the parity tolerances of the decode
step: logits max abs <= 2e-2, tokens exact unless the oracle's top-2 gap is below 1e-3), and the
keys and values it writes to the cache those of the oracle's bf16 cache.
"""
import numpy as np
import pytest
import torch

from quantized_gemv_gb300 import mk
from quantized_gemv_gb300 import synthetic as S
from tests.gpu_util import LOGIT_ATOL, TIE_GAP, make_pair

pytestmark = pytest.mark.gpu


def _prefix(model, om, toks, n):
    """Positions 0 .. n-1 through the decode step on the GPU and the oracle (fills both caches)."""
    for pos in range(n):
        model.decode_step(int(toks[pos]), pos)
        om.step(int(toks[pos]), pos, want_logits=False)


def _verify_against_oracle(model, om, toks, pos0, k):
    cfg = model.cfg
    tdev = torch.tensor(toks[pos0: pos0 + k], dtype=torch.int32, device="cuda")
    nxt = torch.zeros(k, dtype=torch.int32, device="cuda")
    logits = torch.empty((k, cfg.vocab), dtype=torch.float32, device="cuda")
    model.verify_step(tdev, pos0, nxt, logits)
    model.sync()
    nxt, lg = nxt.cpu().numpy(), logits.cpu().numpy().astype(np.float64)
    worst, matches = 0.0, 0
    for i in range(k):
        o_next, o_logits, _, top2 = om.step(int(toks[pos0 + i]), pos0 + i)
        err = float(np.max(np.abs(lg[i] - o_logits)))
        worst = max(worst, err)
        assert err <= LOGIT_ATOL, (i, err)
        if nxt[i] != o_next:
            assert top2[0] - top2[1] < TIE_GAP, (i, nxt[i], o_next)
        matches += int(nxt[i] == o_next)
    return worst, matches


@pytest.mark.parametrize("variant", ["bf16", "fp8", "nvfp4"])
@pytest.mark.parametrize("k", [1, 2, 3, 4, 8])
def test_verify_small_model(variant, k):
    cfg = S.ModelConfig(n_layers=2, vocab=4099, max_ctx=256)
    _, model, om = make_pair(cfg, variant, seed=101 + k)
    model.verify_attach()
    toks = S.prompt_ids(cfg, 40, seed=11 + k)
    _prefix(model, om, toks, 20)
    _, matches = _verify_against_oracle(model, om, toks, 20, k)
    assert matches >= k - 1
    # the keys and values the launch wrote are the oracle's (bf16; a rounding step apart at most)
    ko, vo = om.get_kv(20 + k)
    for l in range(cfg.n_layers):
        kt, vt = model.kv_cache(l)
        for got, want in ((kt, ko[l]), (vt, vo[l])):
            g = got[:, 20: 20 + k].float().cpu().numpy()
            w = torch.from_numpy(want[:, 20: 20 + k].astype(np.int32) << 16).view(torch.float32).numpy()
            assert np.max(np.abs(g - w)) <= 2 ** -7 * np.max(np.abs(w)) + 1e-6
    model.close()


def test_verify_then_decode_continues():
    """Decoding after a verify launch reads the cache rows the launch wrote."""
    cfg = S.ModelConfig(n_layers=2, vocab=4099, max_ctx=256)
    _, model, om = make_pair(cfg, "fp8", seed=131)
    model.verify_attach()
    toks = S.prompt_ids(cfg, 40, seed=31)
    _prefix(model, om, toks, 10)
    _verify_against_oracle(model, om, toks, 10, 8)
    lg = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
    for pos in range(18, 22):
        model.decode_step(int(toks[pos]), pos, lg)
        _, o_logits, _, _ = om.step(int(toks[pos]), pos)
        assert float(np.max(np.abs(lg.cpu().numpy() - o_logits))) <= LOGIT_ATOL
    model.close()


def test_verify_position_zero_and_rejects_bad_arguments():
    cfg = S.ModelConfig(n_layers=1, vocab=1031, max_ctx=64)
    _, model, om = make_pair(cfg, "bf16", seed=141)
    model.verify_attach()
    toks = S.prompt_ids(cfg, 8, seed=41)
    _verify_against_oracle(model, om, toks, 0, 8)   # nothing cached: attention over the new positions only
    nxt = torch.zeros(9, dtype=torch.int32, device="cuda")
    with pytest.raises(mk.MkError):
        model.verify_step(torch.zeros(9, dtype=torch.int32, device="cuda"), 0, nxt)  # k > MK_VERIFY_MAX
    with pytest.raises(mk.MkError):
        model.verify_step(torch.zeros(4, dtype=torch.int32, device="cuda"), 62, nxt)  # past max_ctx
    model.close()


@pytest.mark.parametrize("k", [2, 4, 8])
def test_verify_full_bf16_model(k):
    """The 28-layer bf16 model with its 151,936-row tied head, after the 32-token prompt."""
    wl = S.WORKLOADS["qwen3_0.6b_bf16"]
    cfg = wl.config()
    _, model, om = make_pair(cfg, "bf16", seed=0)
    model.verify_attach()
    prompt = S.prompt_ids(cfg, wl.prompt_len)
    toks = np.concatenate([prompt, S.prompt_ids(cfg, 8, seed=9)])
    _prefix(model, om, toks, wl.prompt_len)
    _, matches = _verify_against_oracle(model, om, toks, wl.prompt_len, k)
    assert matches >= k - 1
    model.close()


@pytest.mark.parametrize("variant", ["fp8", "nvfp4"])
def test_verify_full_quantised_model(variant):
    """The 28-layer FP8 and NVFP4 models (their tiles held as f16, the codes exact) after the 32-token
    prompt, k = 8: the tokens and logits of eight teacher-forced oracle steps."""
    wl = S.WORKLOADS["qwen3_0.6b_" + variant]
    cfg = wl.config()
    _, model, om = make_pair(cfg, variant, seed=0)
    model.verify_attach()
    prompt = S.prompt_ids(cfg, wl.prompt_len)
    toks = np.concatenate([prompt, S.prompt_ids(cfg, 8, seed=19)])
    _prefix(model, om, toks, wl.prompt_len)
    _, matches = _verify_against_oracle(model, om, toks, wl.prompt_len, 8)
    assert matches >= 7
    model.close()


def test_verify_at_the_position_limit():
    """pos0 = 1016, k = 8: the last token attends over all 1,024 positions the verify step allows
    (1,016 of them prefilled in both caches), so every score slot is used; one position further is
    rejected."""
    cfg = S.ModelConfig(n_layers=2, vocab=4099, max_ctx=1100)
    _, model, om = make_pair(cfg, "bf16", seed=151, prefill=1016)
    model.verify_attach()
    toks = S.prompt_ids(cfg, 1024, seed=51)
    _, matches = _verify_against_oracle(model, om, toks, 1016, 8)
    assert matches >= 7
    nxt = torch.zeros(8, dtype=torch.int32, device="cuda")
    with pytest.raises(mk.MkError):
        model.verify_step(torch.zeros(8, dtype=torch.int32, device="cuda"), 1017, nxt)
    model.close()
