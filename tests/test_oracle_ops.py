"""Pins for the oracle's GEMV, RMSNorm, RoPE, attention, SiLU and argmax (CPU only)."""
import math

import numpy as np
import torch
import torch.nn.functional as F

from oracle import oracle as O
from quantized_gemv_gb300 import synthetic as S


def _bf16_bits_of(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_gemv_exact_on_integer_inputs():
    """Small-integer weights and inputs: every product and partial sum is exact, so the result
    must equal the integer dot product computed with Python ints."""
    rng = np.random.default_rng(0)
    for rows, cols in ((7, 48), (33, 160)):
        wi = rng.integers(-8, 9, size=(rows, cols))
        xi = rng.integers(-16, 17, size=cols)
        exact = [int(sum(int(a) * int(b) for a, b in zip(wi[r], xi))) for r in range(rows)]
        # bf16 holds small integers exactly
        m = O.PackedMat(O.FMT_BF16, rows, cols, _bf16_bits_of(wi))
        assert list(O.gemv(m, xi.astype(np.float64))) == exact
        # FP8: integers |v| <= 8 are E4M3 values; scale 1
        codes = np.array([[O.e4m3_encode(float(v)) for v in row] for row in wi], dtype=np.uint8)
        m = O.PackedMat(O.FMT_FP8_ROW, rows, cols, codes, np.ones(rows, np.float32))
        assert list(O.gemv(m, xi.astype(np.float64))) == exact
    # NVFP4: values on the E2M1 grid times block scale 2 and tensor scale 0.5
    rows, cols = 5, 64
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    idx = rng.integers(0, 16, size=(rows, cols))
    vals = np.where(idx >= 8, -grid[idx % 8], grid[idx % 8])
    packed = (idx[:, 0::2] | (idx[:, 1::2] << 4)).astype(np.uint8)
    bs = np.full((rows, cols // 16), O.e4m3_encode(2.0), np.uint8)
    m = O.PackedMat(O.FMT_NVFP4, rows, cols, packed, bs, 0.5)
    x = rng.integers(-16, 17, size=cols).astype(np.float64)
    assert np.array_equal(O.gemv(m, x), vals @ x)


def test_gemv_independent_of_thread_count():
    w = S.random_matrix(3000, 1024, seed=3)
    x = S.random_vector(1024, seed=4).astype(np.float64)
    m = O.PackedMat(O.FMT_BF16, 3000, 1024, w)
    assert np.array_equal(O.gemv(m, x, 1), O.gemv(m, x, 4))


def test_rmsnorm_hand_cases():
    eps = 1e-6
    one = _bf16_bits_of([1.0] * 8)
    c = 3.0
    out = O.rmsnorm(np.full(8, c), one, eps)
    assert np.allclose(out, c / math.sqrt(c * c + eps), rtol=0, atol=1e-15)
    out = O.rmsnorm(np.array([3.0, 4.0]), _bf16_bits_of([1.0, 1.0]), eps)
    assert np.allclose(out, np.array([3.0, 4.0]) / math.sqrt(12.5 + eps), rtol=0, atol=1e-15)
    w = _bf16_bits_of([2.0, 0.5])
    out = O.rmsnorm(np.array([3.0, 4.0]), w, eps)
    assert np.allclose(out, np.array([6.0, 2.0]) / math.sqrt(12.5 + eps), rtol=0, atol=1e-15)
    # library routine: torch's rms_norm in float64
    x = np.random.default_rng(1).normal(size=128)
    wn = _bf16_bits_of(np.random.default_rng(2).normal(1, 0.1, 128))
    wt = torch.from_numpy(wn.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    ref = F.rms_norm(torch.from_numpy(x), (128,), weight=wt, eps=eps).numpy()
    assert np.allclose(O.rmsnorm(x, wn, eps), ref, rtol=1e-13, atol=0)


def test_rope_properties():
    rng = np.random.default_rng(3)
    theta = 1e6
    x = rng.normal(size=128)
    assert np.array_equal(O.rope(x, 0, theta), x)                           # position 0: identity
    for pos in (1, 17, 4159):
        assert abs(np.linalg.norm(O.rope(x, pos, theta)) - np.linalg.norm(x)) < 1e-12
    q, k = rng.normal(size=128), rng.normal(size=128)
    d1 = O.rope(q, 40, theta) @ O.rope(k, 30, theta)                        # depends on m - n only
    d2 = O.rope(q, 1010, theta) @ O.rope(k, 1000, theta)
    assert abs(d1 - d2) < 1e-9
    # head_dim 2: a plain 2-D rotation by pos radians
    assert np.allclose(O.rope(np.array([1.0, 0.0]), 1, theta), [math.cos(1), math.sin(1)], atol=1e-15)
    # half-split pairing: element i pairs with i + d/2 (the pair with frequency index 1 for d=4)
    y = O.rope(np.array([0.0, 1.0, 0.0, 0.0]), 2, 100.0)
    ang = 2 * 100.0 ** (-2 * 1 / 4)
    assert np.allclose(y, [0.0, math.cos(ang), 0.0, math.sin(ang)], atol=1e-15)


def test_attention_pins():
    rng = np.random.default_rng(4)
    d = 128
    K = _bf16_bits_of(rng.normal(size=(1, d)))
    V = _bf16_bits_of(rng.normal(size=(1, d)))
    vf = torch.from_numpy(V.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.attend(rng.normal(size=d), K, V), vf[0])        # one position: V[0]
    n = 7
    Keq = np.repeat(K, n, axis=0)
    Vn = _bf16_bits_of(rng.normal(size=(n, d)))
    vnf = torch.from_numpy(Vn.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.allclose(O.attend(rng.normal(size=d), Keq, Vn), vnf.mean(axis=0), atol=1e-14)  # equal keys
    # library routine: scaled_dot_product_attention in float64
    n = 50
    Kr = _bf16_bits_of(rng.normal(size=(n, d)))
    Vr = _bf16_bits_of(rng.normal(size=(n, d)))
    q = rng.normal(size=d) * 3
    kt = torch.from_numpy(Kr.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    vt = torch.from_numpy(Vr.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    ref = F.scaled_dot_product_attention(torch.from_numpy(q)[None, None, None], kt[None, None], vt[None, None])
    assert np.allclose(O.attend(q, Kr, Vr), ref[0, 0, 0].numpy(), rtol=1e-12, atol=1e-13)


def test_silu():
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(40.0) - 40.0) < 1e-12
    assert abs(O.silu(-40.0)) < 1e-12
    z = np.linspace(-9, 9, 37)
    ref = F.silu(torch.from_numpy(z)).numpy()
    assert np.allclose([O.silu(v) for v in z], ref, rtol=1e-14, atol=1e-15)


def test_argmax_lowest_index_on_ties():
    x = np.array([0.5, 2.0, -1.0, 2.0, 2.0])
    assert O.argmax(x) == 1
    x = np.zeros(1000)
    x[[700, 13, 999]] = 1.0
    assert O.argmax(x) == 13
    assert O.argmax(np.array([-3.0])) == 0
