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
    return O.pack_model(master, fmap, nthreads)
