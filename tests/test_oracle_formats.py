"""Pins for the oracle's number formats and quantisers (CPU only).

Each pin compares the oracle with something other than itself: the E2M1 grid printed on the
TSCT super-kernel page (section 3b), PyTorch's float8_e4m3fn / bfloat16 casts (library
routines), brute-force nearest-value search, and closed-form error bounds.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantized_gemv_gb300 import synthetic as S
from tests._helpers import golden_e2m1_grid


def test_e2m1_codes_span_printed_grid():
    grid = golden_e2m1_grid()
    pos = [O.e2m1_value(c) for c in range(8)]
    neg = [O.e2m1_value(c) for c in range(8, 16)]
    assert pos == grid                      # codes 0..7 are the printed magnitudes, ascending
    assert neg == [-v for v in grid]        # codes 8..15 carry the sign bit
    assert math.copysign(1.0, O.e2m1_value(8)) == -1.0


def _nearest_even(v, table):
    """Brute force: nearest entry of `table` (code -> value); ties to the even code."""
    best = None
    for c, x in table.items():
        d = abs(x - v)
        if best is None or d < best[0] - 1e-300 or (abs(d - best[0]) <= 1e-300 and c % 2 == 0 and best[1] % 2 == 1):
            best = (d, c)
    return best[1]


def test_e2m1_encode_bruteforce():
    grid = golden_e2m1_grid()
    table = {c: grid[c] for c in range(8)}
    rng = np.random.default_rng(0)
    vals = list(rng.uniform(0, 6, 4000)) + [m for m in np.arange(0, 6.0001, 0.25)]
    vals += [(a + b) / 2 for a, b in zip(grid[:-1], grid[1:])]  # every midpoint
    for v in vals:
        c = O.e2m1_encode(v)
        assert c == _nearest_even(v, table), v
        assert O.e2m1_encode(-v) == (c | 8)
    for v in (6.0, 6.1, 7.0, 1e9):
        assert O.e2m1_encode(v) == 7 and O.e2m1_encode(-v) == 15
    # midpoints resolve to the even mantissa (printed grid, ties to even)
    assert [O.e2m1_value(O.e2m1_encode(m)) for m in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)] == \
        [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = O.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v) and c in (0x7F, 0xFF)
        else:
            assert v == ref[c] and math.copysign(1, v) == math.copysign(1, ref[c]), c


def test_e4m3_encode_roundtrip_and_saturation():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert O.e4m3_encode(O.e4m3_value(c)) == c
    for v in (448.0, 449.0, 464.0, 500.0, 1e30):
        assert O.e4m3_encode(v) == 0x7E and O.e4m3_encode(-v) == 0xFE
    assert O.e4m3_encode(-1e-30) == 0x80   # sign kept when the magnitude rounds to zero


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(1)
    mids = []
    vals = sorted({O.e4m3_value(c) for c in range(0x7F)})
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1e-2, 5000),
                        np.array(mids), -np.array(mids)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([O.e4m3_encode(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_bf16_encode_matches_torch_cast():
    rng = np.random.default_rng(2)
    base = rng.normal(0, 1, 20000).astype(np.float32)
    # values exactly halfway between bf16 neighbours (ties) and one float32 ulp either side
    u = base.view(np.uint32) & np.uint32(0xFFFF0000)
    ties = (u | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([base, ties, np.nextafter(ties, np.float32(np.inf)), np.nextafter(ties, np.float32(-np.inf))])
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([O.bf16_encode(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)
    for b in (0x0000, 0x3F80, 0xBF80, 0x0001, 0x7F7F):
        assert O.bf16_encode(O.bf16_value(b)) == b


def _torch_fp8_row_codes(w_bits):
    w = torch.from_numpy(w_bits.view(np.int16)).view(torch.bfloat16).to(torch.float32)
    amax = w.abs().amax(dim=1)
    s = amax / torch.tensor(448.0, dtype=torch.float32)
    q = w / s[:, None]
    return q.to(torch.float8_e4m3fn).view(torch.uint8).numpy(), s.numpy()


def test_quant_fp8_matches_torch_cast():
    w = S.random_matrix(67, 320, seed=5)
    codes, scales = O.quant_fp8_row(w)
    ref_codes, ref_s = _torch_fp8_row_codes(w)
    assert np.array_equal(scales, ref_s)
    assert np.array_equal(codes, ref_codes)


def test_quant_fp8_error_bound_and_zero_row():
    w = S.random_matrix(40, 256, seed=6)
    w[3, :] = 0
    codes, scales = O.quant_fp8_row(w)
    assert scales[3] == 0 and not codes[3].any()
    deq = O.dequant(O.PackedMat(O.FMT_FP8_ROW, 40, 256, codes, scales))
    wf = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    # half an E4M3 ulp: 2^-4 relative for normals, 2^-10 absolute (times s) for subnormals,
    # plus the fp32 rounding of w/s
    s = scales.astype(np.float64)[:, None]
    bound = np.maximum(np.abs(wf) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 2.0 ** -20)
    assert np.all(np.abs(deq - wf) <= bound)
    assert np.all(np.abs(deq).max(axis=1)[np.arange(40) != 3] <= scales[np.arange(40) != 3] * 448 * (1 + 1e-6))


def test_quant_nvfp4_bruteforce():
    grid = golden_e2m1_grid()
    table = {c: grid[c] for c in range(8)}
    w = S.random_matrix(9, 96, seed=7)
    w[2, 16:32] = 0                          # one all-zero block
    codes, bscales, t = O.quant_nvfp4(w)
    wf32 = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).to(torch.float32)
    amax_t = wf32.abs().max()
    t_ref = amax_t / torch.tensor(2688.0)
    assert t == float(t_ref)
    t6 = torch.tensor(6.0) * t_ref
    blocks = wf32.view(9, 6, 16)
    ratio = blocks.abs().amax(dim=2) / t6
    b_ref = ratio.to(torch.float8_e4m3fn)
    assert np.array_equal(bscales, b_ref.view(torch.uint8).numpy())
    denom = (b_ref.to(torch.float32) * t_ref)[:, :, None]
    q = (blocks / denom).numpy()
    for r in range(9):
        for k in range(96):
            b, j = divmod(k, 16)
            nib = (codes[r, k // 2] >> (4 * (k % 2))) & 0xF
            if float(denom[r, b, 0]) == 0.0:
                assert nib == 0
                continue
            v = float(q[r, b, j])
            want = _nearest_even(abs(v), table) if abs(v) < 6 else 7
            if math.copysign(1, v) < 0:
                want |= 8
            assert nib == want, (r, k, v)
    deq = O.dequant(O.PackedMat(O.FMT_NVFP4, 9, 96, codes, bscales, t))
    assert not deq[2, 16:32].any()
