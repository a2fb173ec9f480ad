"""GPU: the LM-head argmax's tie rule across CTAs, warps and lanes.

Two rows of the tied embedding / LM-head matrix are made bit-identical and far larger than every
other logit, so they tie for the maximum; the step must return the lower index (the lowest index
among equal maxima, as the oracle's argmax does). The rows are chosen so that the tie is resolved
across CTAs (rows owned by different CTAs of the decode grid), across warps of one CTA, and
between lanes of one warp's row group.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantized_gemv_gb300 import mk
from quantized_gemv_gb300 import synthetic as S
from tests._helpers import oracle_pack_model

pytestmark = pytest.mark.gpu

CFG = S.ModelConfig(n_layers=2, vocab=4099, max_ctx=64)


def _owner(row, vocab, grid):
    """CTA of the decode grid whose LM-head rows include `row` (even split of the vocabulary)."""
    return next(c for c in range(grid) if vocab * c // grid <= row < vocab * (c + 1) // grid)


@pytest.mark.parametrize("variant", ["bf16", "fp8"])
@pytest.mark.parametrize("a,b", [(200, 3000), (200, 212), (201, 202)])
def test_equal_maxima_give_lowest_index(variant, a, b):
    token, pos = 11, 0
    master = S.master_weights(CFG, seed=5)
    fmap = S.format_map(variant)
    # the final normalised hidden state of this step does not depend on rows a and b (the input
    # token is another row), so it is taken from the unmodified model
    om0 = O.OracleModel(CFG, oracle_pack_model(master, fmap))
    _, _, hid, _ = om0.step(token, pos, want_logits=False, want_hidden=True)
    h = hid[-1]
    w = master["final_norm"].astype(np.uint32) << 16
    xhat = h / np.sqrt(np.mean(h * h) + CFG.rms_eps) * w.view(np.float32)
    row = torch.from_numpy(np.where(xhat >= 0, 0.05, -0.05).astype(np.float32)).to(torch.bfloat16)
    bits = row.view(torch.int16).numpy().view(np.uint16)
    master["embed"] = master["embed"].copy()
    master["embed"][a] = bits
    master["embed"][b] = bits
    model = mk.Model(CFG, mk.pack_model(master, fmap))
    om = O.OracleModel(CFG, oracle_pack_model(master, fmap))
    logits = torch.empty(CFG.vocab, dtype=torch.float32, device="cuda")
    nxt = model.decode_step(token, pos, logits)
    o_next, o_logits, _, top2 = om.step(token, pos)
    lg = logits.cpu().numpy()
    assert o_next == a and top2[0] == top2[1]
    assert lg.view(np.uint32)[a] == lg.view(np.uint32)[b]
    assert lg[a] > np.max(np.delete(lg, [a, b])) + 1.0
    assert nxt == a, (nxt, a, b)
    # the same step without the logits output (the argmax alone)
    nxt2 = model.decode_step(token, pos)
    assert nxt2 == a
    grid = mk.decode_grid()
    if (a, b) == (200, 3000):
        assert _owner(a, CFG.vocab, grid) != _owner(b, CFG.vocab, grid)
    model.close()
