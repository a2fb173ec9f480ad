"""Shared test helpers: turn seeded bf16 masters into oracle-packed models, golden files."""
import os

import numpy as np

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_e2m1_grid():
    vals = []
    with open(os.path.join(GOLDEN, "e2m1_grid.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(float(line))
    return vals


def oracle_pack_model(master, fmap, nthreads=None):
    """Quantise every matrix of a master-weight dict with the oracle's own quantiser."""
    def pk(w, fmt):
        if fmt == O.FMT_BF16:
            return O.PackedMat(fmt, w.shape[0], w.shape[1], w)
        if fmt == O.FMT_FP8_ROW:
            c, s = O.quant_fp8_row(w, nthreads)
            return O.PackedMat(fmt, w.shape[0], w.shape[1], c, s)
        c, b, t = O.quant_nvfp4(w, nthreads)
        return O.PackedMat(fmt, w.shape[0], w.shape[1], c, b, t)

    out = {"embed": pk(master["embed"], fmap["embed"]), "final_norm": master["final_norm"], "layers": []}
    for L in master["layers"]:
        d = {n: pk(L[n], fmap[n]) for n in O.LINEARS}
        for n in ("ln_in", "ln_post", "q_norm", "k_norm"):
            d[n] = L[n]
        out["layers"].append(d)
    return out
