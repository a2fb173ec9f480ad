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



def test_quant_fp8_bf16_scale_matches_torch_cast():
    """bf16 row scales: torch's fp32 division, its bfloat16 cast of the scale, then its float8 cast
    of w / scale clamped to the finite range (saturation), as library routines."""
    w = S.random_matrix(67, 320, seed=8)
    w[4, :] = 0
    codes, scales = O.quant_fp8_row(w, bf16_scale=True)
    wf = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).to(torch.float32)
    s = (wf.abs().amax(dim=1) / torch.tensor(448.0)).to(torch.bfloat16).to(torch.float32)
    q = torch.where(s[:, None] > 0, wf / s[:, None], torch.zeros_like(wf)).clamp(-448.0, 448.0)
    assert np.array_equal(scales, s.numpy())
    assert np.array_equal(codes, q.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    # the scales are bf16 numbers; rows whose scale rounded down saturate their maximum at 448
    assert np.array_equal(scales.view(np.uint32) & 0xFFFF, np.zeros(67, np.uint32))
    fp32_s = (wf.abs().amax(dim=1) / torch.tensor(448.0)).numpy()
    down = np.nonzero(scales < fp32_s)[0]
    assert len(down) > 5 and all((codes[r] & 0x7F).max() == 0x7E for r in down)

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



def _e2m1_round(q, grid):
    """Vectorised brute force: nearest printed E2M1 magnitude (ties to the even code, saturating
    at 6); returns the codes with the sign bit of q."""
    g = np.asarray(grid)
    a = np.abs(q)
    d = np.abs(a[..., None] - g)
    hit = d == d.min(-1, keepdims=True)
    even = np.where(hit & (np.arange(8) % 2 == 0), np.arange(8), 99).min(-1)
    k = np.where(even < 99, even, np.where(hit, np.arange(8), 99).min(-1))
    k = np.where(a >= 6, 7, k)
    return k | np.where(np.signbit(q), 8, 0)


def test_quant_nvfp4_scale_search_bruteforce():
    """Every block scale tried by brute force (torch float8 decode, fp32 torch division, the
    printed grid): the oracle's choice has the least squared error, no smaller code reaches it,
    and its E2M1 codes are the round-to-nearest ones for that scale."""
    grid = golden_e2m1_grid()
    rows, cols = 24, 160
    w = S.random_matrix(rows, cols, seed=17)
    w[5, 32:48] = 0                                                  # an all-zero block
    w[6, 0:16] = S.random_matrix(1, 16, seed=18, std=1e-5)[0]        # a block far below the tensor amax
    codes, bscales, t = O.quant_nvfp4(w, scale_search=True)
    wf32 = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).to(torch.float32)
    assert t == float(wf32.abs().max() / torch.tensor(2688.0))
    blocks = wf32.view(rows, cols // 16, 16)
    e4 = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32)
    denom = e4 * torch.tensor(t, dtype=torch.float32)                        # fp32, one per code
    q = (blocks[:, :, None, :] / denom[None, None, :, None]).numpy()        # [r][b][code][j]
    nib = _e2m1_round(np.nan_to_num(q, nan=0.0, posinf=0.0, neginf=0.0), grid)
    nib[:, :, denom.numpy() == 0, :] = 0
    val = np.asarray(grid)[nib & 7] * np.where(nib & 8, -1.0, 1.0)
    rec = val * e4.double().numpy()[None, None, :, None] * float(t)
    err = ((blocks.double().numpy()[:, :, None, :] - rec) ** 2).sum(-1)    # [r][b][code]
    for r in range(rows):
        for b in range(cols // 16):
            c = int(bscales[r, b])
            e = err[r, b]
            assert e[c] <= e.min() * (1 + 1e-12), (r, b, c, int(e.argmin()))
            assert np.all(e[:c] > e[c] * (1 + 1e-12)), (r, b, c)
            got = [(codes[r, (16 * b + j) // 2] >> (4 * (j % 2))) & 0xF for j in range(16)]
            assert got == list(nib[r, b, c]), (r, b)
    assert not bscales[5, 2] and not codes[5, 16:24].any()
    # never worse than the amax block scale, block by block, and better overall
    ca, ba, ta = O.quant_nvfp4(w)
    sse_s = err[np.arange(rows)[:, None], np.arange(cols // 16)[None, :], bscales]
    deq_a = O.dequant(O.PackedMat(O.FMT_NVFP4, rows, cols, ca, ba, ta)).reshape(rows, cols // 16, 16)
    sse_a = ((deq_a - blocks.double().numpy()) ** 2).sum(-1)
    assert np.all(sse_s <= sse_a * (1 + 1e-12))
    assert sse_s.sum() < 0.9 * sse_a.sum()


def test_quant_nvfp4_scale_search_worked_ties():
    """Hand-worked blocks at tensor scale t = 1 (tensor amax 2688 = 6 * 448):
    - {2688}: code 0x7E (448) puts it exactly on 6; no other scale is exact, since 2688/4 > 448.
    - {-10, -12}: scale 3 (code 68) gives -9, -12 and scale 6 (code 76) gives -9, -12 as well;
      both have squared error 1, the least of all scales; the tie goes to the smaller code, 68.
    - {-1, 5}: scale 0.8125 (code 53) gives -0.8125 and 4.875 (5/0.8125 saturates at 6), scale
      1.625 (code 61) gives -0.8125 and 4.875 (5/1.625 rounds to 3); error 0.05078125 each; 53.
    - all zero: code 0."""
    def bits(x):
        return int(torch.tensor(x, dtype=torch.bfloat16).view(torch.int16)) & 0xFFFF
    w = np.zeros((4, 16), np.uint16)
    w[0, 0] = bits(2688.0)
    w[1, 3], w[1, 9] = bits(-10.0), bits(-12.0)
    w[2, 7], w[2, 3] = bits(-1.0), bits(5.0)
    codes, bscales, t = O.quant_nvfp4(w, scale_search=True)
    assert t == 1.0
    assert list(bscales[:, 0]) == [0x7E, 68, 53, 0]
    deq = O.dequant(O.PackedMat(O.FMT_NVFP4, 4, 16, codes, bscales, t))
    assert deq[0, 0] == 2688.0 and deq[1, 3] == -9.0 and deq[1, 9] == -12.0
    assert deq[2, 7] == -0.8125 and deq[2, 3] == 4.875
    assert not deq[3].any() and np.count_nonzero(deq) == 5

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
