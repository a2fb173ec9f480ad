"""GPU: the bounds-checking debug build (libmk_debug.so, MK_DEBUG_BOUNDS) runs the decode and
verify paths clean and in parity with the oracle.

In that build every checked device access (ring rows and block scales, KV-cache rows and tiles,
exchange-word and logit indices, count-word accumulators, the verify operand and MMA windows) is
tested first; an out-of-range one is skipped and the step fails with MK_EBOUNDS instead of
touching memory. The library is chosen when a process first loads it, so the run happens in a
fresh interpreter with MK_LIBRARY=debug.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import os, sys
sys.path.insert(0, %(root)r)
import numpy as np, torch
from quantized_gemv_gb300 import mk
from quantized_gemv_gb300 import synthetic as S
from tests.gpu_util import compare_step, make_pair
assert os.path.basename(mk.lib()._name) == "libmk_debug.so", mk.lib()._name
for variant in ("bf16", "nvfp4"):
    cfg = S.ModelConfig(n_layers=2, vocab=4099, max_ctx=512)
    _, model, om = make_pair(cfg, variant, seed=151)
    toks = S.prompt_ids(cfg, 300, seed=13)
    for pos in range(296):  # across the single-unit attention window (288 positions)
        compare_step(model, om, int(toks[pos]), pos, check_hidden=pos in (5, 287, 295))
    model.verify_attach()
    t = torch.tensor(toks[296:300], dtype=torch.int32, device="cuda")
    nxt = torch.zeros(4, dtype=torch.int32, device="cuda")
    model.verify_step(t, 296, nxt)
    model.sync()
    model.close()
print("debug build clean")
"""


def test_debug_bounds_build_runs_clean_and_matches_the_oracle():
    env = dict(os.environ, MK_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", SCRIPT % {"root": ROOT}], env=env, capture_output=True, text=True,
                       timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "debug build clean" in r.stdout
