"""The synthetic inputs (the stand-ins for the trained checkpoint, the prompt set and the KV cache):
distributions, draw order, seeds, bf16 rounding and determinism, as the recipe states them."""
import numpy as np
import torch

from quantized_gemv_gb300 import synthetic as S

TINY = S.ModelConfig(n_layers=2, vocab=700, max_ctx=64)


def _f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_same_seed_same_bits_other_seed_other_bits():
    a, b, c = S.master_weights(TINY, seed=3), S.master_weights(TINY, seed=3), S.master_weights(TINY, seed=4)
    assert np.array_equal(a["embed"], b["embed"]) and not np.array_equal(a["embed"], c["embed"])
    for la, lb in zip(a["layers"], b["layers"]):
        for k in la:
            assert np.array_equal(la[k], lb[k])


def test_draw_order_and_bf16_rounding():
    """Embedding first, then per layer q, k, v, o, gate, up, down, ln_in, ln_post, q_norm, k_norm,
    then the final norm, from one generator; every value is torch's RNE bf16 rounding."""
    m = S.master_weights(TINY, seed=5)
    g = torch.Generator(device="cpu")
    g.manual_seed(5)
    bits = lambda t: t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    assert np.array_equal(m["embed"], bits(torch.randn(TINY.vocab, TINY.hidden, generator=g) * 0.02))
    sh = TINY.shapes()
    for L in m["layers"]:
        for n in S.LINEARS:
            assert np.array_equal(L[n], bits(torch.randn(*sh[n], generator=g) * 0.02)), n
        for n, size in (("ln_in", TINY.hidden), ("ln_post", TINY.hidden), ("q_norm", TINY.head_dim),
                        ("k_norm", TINY.head_dim)):
            assert np.array_equal(L[n], bits(1.0 + 0.1 * torch.randn(size, generator=g))), n
    assert np.array_equal(m["final_norm"], bits(1.0 + 0.1 * torch.randn(TINY.hidden, generator=g)))


def test_distributions():
    m = S.master_weights(S.ModelConfig(n_layers=1, vocab=4096), seed=0)
    w = _f32(m["embed"]).astype(np.float64)
    assert abs(w.mean()) < 2e-4 and abs(w.std() - 0.02) < 2e-4  # 4.2M draws of N(0, 0.02^2)
    gate = _f32(m["layers"][0]["gate"]).astype(np.float64)
    assert abs(gate.std() - 0.02) < 2e-4
    norms = np.concatenate([_f32(m["layers"][0][k]) for k in ("ln_in", "ln_post")]).astype(np.float64)
    assert abs(norms.mean() - 1.0) < 0.02 and abs(norms.std() - 0.1) < 0.01


def test_prompt_ids_uniform_in_vocab_and_seeded():
    ids = S.prompt_ids(S.QWEN3_06B, 32)
    g = torch.Generator(device="cpu")
    g.manual_seed(1)
    assert ids.dtype == np.int32
    assert np.array_equal(ids, torch.randint(0, 151936, (32,), generator=g).numpy())
    many = S.prompt_ids(TINY, 20000, seed=9)
    assert many.min() >= 0 and many.max() < TINY.vocab
    counts = np.bincount(many, minlength=TINY.vocab)
    assert counts.min() > 0  # every id drawn at least once out of 20000 over 700 ids


def test_prefilled_kv_layout_and_distribution():
    k, v = S.prefill_kv(TINY, 40, seed=2)
    assert k.shape == v.shape == (TINY.n_layers, TINY.n_kv_heads, 40, TINY.head_dim)
    assert k.dtype == np.uint16
    kf, vf = _f32(k).astype(np.float64), _f32(v).astype(np.float64)
    assert abs(kf.std() - 1.0) < 0.05 and abs(vf.std() - 1.0) < 0.05
    assert not np.array_equal(k, v)  # keys are drawn first, then values, from one generator
    g = torch.Generator(device="cpu")
    g.manual_seed(2)
    first = torch.randn(TINY.n_layers, TINY.n_kv_heads, 40, TINY.head_dim, generator=g)
    assert np.array_equal(k, first.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def test_workloads_fit_their_contexts():
    for wl in S.WORKLOADS.values():
        cfg = wl.config()
        start = wl.prefill + wl.prompt_len
        assert start + wl.steps <= cfg.max_ctx, wl.name
        assert cfg.n_layers == wl.n_layers
