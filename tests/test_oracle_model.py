"""Pins for the oracle's full decode step (CPU only).

The pages print no worked example for the model, so the whole step is pinned by (a) a
float64 composition of PyTorch library routines (rms_norm, scaled_dot_product_attention with
GQA, silu, matmul, complex rotation) over weights dequantised without the oracle (torch's
float8 view and the printed E2M1 grid), and (b) invariants: determinism, thread-count
independence, and KV-cache round trips.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle as O
from quantized_gemv_gb300 import synthetic as S
from tests._helpers import golden_e2m1_grid, oracle_pack_model

TINY = S.ModelConfig(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16, ffn=128,
                     vocab=500, max_ctx=64)


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(torch.float64)


def _torch_dequant(pm):
    if pm.fmt == O.FMT_BF16:
        return _bf16(pm.data)
    if pm.fmt == O.FMT_FP8_ROW:
        q = torch.from_numpy(pm.data).view(torch.float8_e4m3fn).to(torch.float64)
        return q * torch.from_numpy(pm.scale).to(torch.float64)[:, None]
    grid = torch.tensor(golden_e2m1_grid(), dtype=torch.float64)
    table = torch.cat([grid, -grid])
    lo = torch.from_numpy((pm.data & 0xF).astype(np.int64))
    hi = torch.from_numpy((pm.data >> 4).astype(np.int64))
    codes = torch.stack([lo, hi], dim=-1).reshape(pm.rows, pm.cols)
    bs = torch.from_numpy(pm.scale).view(torch.float8_e4m3fn).to(torch.float64)
    return table[codes] * bs.repeat_interleave(16, dim=1) * pm.tensor_scale


def _torch_rope(x, pos, theta):
    d = x.shape[-1]
    inv = theta ** (-torch.arange(0, d, 2, dtype=torch.float64) / d)
    rot = torch.polar(torch.ones_like(inv), pos * inv)
    z = torch.complex(x[..., : d // 2], x[..., d // 2:]) * rot
    return torch.cat([z.real, z.imag], dim=-1)


class TorchRef:
    """Float64 decode step assembled from PyTorch library routines."""

    def __init__(self, cfg, packed):
        self.cfg = cfg
        self.E = _torch_dequant(packed["embed"])
        self.fn = _bf16(packed["final_norm"])
        self.L = []
        for Lp in packed["layers"]:
            d = {n: _torch_dequant(Lp[n]) for n in O.LINEARS}
            for n in ("ln_in", "ln_post", "q_norm", "k_norm"):
                d[n] = _bf16(Lp[n])
            self.L.append(d)
        shape = (cfg.n_layers, cfg.n_kv_heads, cfg.max_ctx, cfg.head_dim)
        self.K = torch.zeros(shape, dtype=torch.float64)
        self.V = torch.zeros(shape, dtype=torch.float64)

    def step(self, token, pos):
        c = self.cfg
        eps = c.rms_eps
        h = self.E[token].clone()
        for l, W in enumerate(self.L):
            xn = F.rms_norm(h, (c.hidden,), weight=W["ln_in"], eps=eps)
            q = (W["q"] @ xn).view(c.n_q_heads, c.head_dim)
            k = (W["k"] @ xn).view(c.n_kv_heads, c.head_dim)
            v = (W["v"] @ xn).view(c.n_kv_heads, c.head_dim)
            q = _torch_rope(F.rms_norm(q, (c.head_dim,), weight=W["q_norm"], eps=eps), pos, c.rope_theta)
            k = _torch_rope(F.rms_norm(k, (c.head_dim,), weight=W["k_norm"], eps=eps), pos, c.rope_theta)
            self.K[l, :, pos] = k.to(torch.bfloat16).to(torch.float64)
            self.V[l, :, pos] = v.to(torch.bfloat16).to(torch.float64)
            att = F.scaled_dot_product_attention(q[None, :, None, :], self.K[l, :, : pos + 1][None],
                                                 self.V[l, :, : pos + 1][None], enable_gqa=True)
            h = h + W["o"] @ att.reshape(-1)
            xn = F.rms_norm(h, (c.hidden,), weight=W["ln_post"], eps=eps)
            h = h + W["down"] @ (F.silu(W["gate"] @ xn) * (W["up"] @ xn))
        logits = self.E @ F.rms_norm(h, (c.hidden,), weight=self.fn, eps=eps)
        return int(torch.argmax(logits)), logits.numpy()


@pytest.mark.parametrize("variant", ["bf16", "fp8", "nvfp4", "fp8_bf16head", "nvfp4_mse", "nvfp4_all", "fp8_bf16scale"])
def test_oracle_matches_torch_composition(variant):
    master = S.master_weights(TINY, seed=11)
    packed = oracle_pack_model(master, S.format_map(variant))
    om = O.OracleModel(TINY, packed, n_threads=2)
    ref = TorchRef(TINY, packed)
    kp, vp = S.prefill_kv(TINY, 5, seed=12)
    om.set_kv(kp, vp)
    ref.K[:, :, :5] = _bf16(kp)
    ref.V[:, :, :5] = _bf16(vp)
    tok = 7
    for pos in range(5, 12):
        nxt, logits, _, top2 = om.step(tok, pos)
        rn, rl = ref.step(tok, pos)
        assert np.allclose(logits, rl, rtol=0, atol=1e-9)
        assert nxt == rn or abs(top2[0] - top2[1]) < 1e-9
        tok = nxt


def test_oracle_deterministic_and_thread_independent():
    master = S.master_weights(TINY, seed=13)
    packed = oracle_pack_model(master, S.format_map("fp8"))
    outs = []
    for nt in (1, 3, 1):
        om = O.OracleModel(TINY, packed, n_threads=nt)
        seq, tok = [], 3
        for pos in range(6):
            tok, logits, hidden, _ = om.step(tok, pos, want_hidden=True)
            seq.append((tok, logits.copy(), hidden.copy()))
        outs.append(seq)
    for seq in outs[1:]:
        for a, b in zip(outs[0], seq):
            assert a[0] == b[0] and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])


def test_oracle_kv_roundtrip_and_hidden_layout():
    master = S.master_weights(TINY, seed=14)
    packed = oracle_pack_model(master, S.format_map("bf16"))
    om = O.OracleModel(TINY, packed, n_threads=1)
    kp, vp = S.prefill_kv(TINY, 4, seed=15)
    om.set_kv(kp, vp)
    k2, v2 = om.get_kv(4)
    assert np.array_equal(k2, kp) and np.array_equal(v2, vp)
    _, _, hidden, _ = om.step(9, 4, want_hidden=True)
    # hidden[0] is the embedding row of the token
    assert np.array_equal(hidden[0], _bf16(master["embed"][9]).numpy())
    with pytest.raises(ValueError):
        om.step(9, TINY.max_ctx)
    with pytest.raises(ValueError):
        om.step(TINY.vocab, 0)
