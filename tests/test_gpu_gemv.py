"""GPU: the streaming dequant-GEMV (mk_gemv) against the oracle's double-precision GEMV."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantized_gemv_gb300 import mk
from quantized_gemv_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


def _oracle_mat(dm: mk.PackedMat) -> O.PackedMat:
    scale = None if dm.scale is None else dm.scale.cpu().numpy()
    data = dm.data.cpu()
    data = data.view(torch.int16).numpy().view(np.uint16) if dm.fmt == 0 else data.numpy()
    return O.PackedMat(dm.fmt, dm.rows, dm.cols, data, scale, dm.tensor_scale)


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("rows,cols", [(1, 1024), (7, 2048), (331, 1024), (1000, 3072), (4099, 1024), (64, 4096)])
def test_gemv_matches_oracle(fmt, rows, cols):
    w = S.random_matrix(rows, cols, seed=rows + cols + fmt)
    dm = mk.pack(mk.upload_bf16(w), fmt)
    x = S.random_vector(cols, seed=7)
    y = mk.gemv(dm, torch.from_numpy(x).cuda()).cpu().numpy().astype(np.float64)
    om = _oracle_mat(dm)
    yo = O.gemv(om, x.astype(np.float64))
    # fp32 accumulation: bound the error by a small multiple of eps * sum|w x|
    absw = np.abs(O.dequant(om))
    bound = 4 * 2.0 ** -24 * cols ** 0.5 * (absw @ np.abs(x.astype(np.float64))) + 1e-30
    assert np.all(np.abs(y - yo) <= bound * 8), np.max(np.abs(y - yo) / bound)


def _e4m3_codes(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)


E2M1_CODE = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("rows,cols", [(1, 1024), (7, 2048), (331, 3072), (4099, 1024), (64, 4096)])
def test_gemv_integer_inputs_exact(fmt, rows, cols):
    """Weights and inputs on small integer (or half-integer) grids, so every product and partial
    sum is exact in fp32: the GPU must equal the exact dot products bit for bit, whatever its
    summation order. A dropped, doubled or misplaced chunk shows up as an exact mismatch."""
    g = np.random.default_rng(rows * 7 + cols + fmt)
    x = g.integers(-4, 5, size=cols).astype(np.float32)
    if fmt == 0:      # bf16 integers in [-8, 8]
        wv = g.integers(-8, 9, size=(rows, cols)).astype(np.float32)
        dm = mk.PackedMat(0, rows, cols, torch.from_numpy(wv).to(torch.bfloat16).cuda())
        exact = wv.astype(np.float64) @ x.astype(np.float64)
    elif fmt == 1:    # E4M3 integers in [-8, 8], row scales powers of two
        wv = g.integers(-8, 9, size=(rows, cols)).astype(np.float32)
        sc = (2.0 ** g.integers(-3, 4, size=rows)).astype(np.float32)
        codes = _e4m3_codes(wv.reshape(-1)).reshape(rows, cols)
        dm = mk.PackedMat(1, rows, cols, codes.cuda(), torch.from_numpy(sc).cuda())
        exact = (wv.astype(np.float64) @ x.astype(np.float64)) * sc
    else:             # E2M1 grid values, E4M3 block scales and tensor scale powers of two
        mag = np.array(sorted(E2M1_CODE), dtype=np.float32)
        wv = mag[g.integers(0, 8, size=(rows, cols))] * np.where(g.random((rows, cols)) < 0.5, -1.0, 1.0)
        wv = wv.astype(np.float32)
        nib = np.vectorize(lambda v: E2M1_CODE[abs(float(v))] | (8 if v < 0 else 0))(wv).astype(np.uint8)
        packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
        bsv = (2.0 ** g.integers(-2, 3, size=(rows, cols // 16))).astype(np.float32)
        bcodes = _e4m3_codes(bsv.reshape(-1)).reshape(rows, cols // 16)
        t = 0.5
        dm = mk.PackedMat(2, rows, cols, torch.from_numpy(packed).cuda(), bcodes.cuda(), t)
        exact = (wv.astype(np.float64) * np.repeat(bsv, 16, axis=1)) @ x.astype(np.float64) * t
    y = mk.gemv(dm, torch.from_numpy(x).cuda()).cpu().numpy()
    assert np.abs(exact).max() < 2 ** 22
    assert np.array_equal(y.astype(np.float64), exact), np.flatnonzero(y != exact)[:8]
