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
