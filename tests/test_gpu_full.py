"""GPU: the full 28-layer Qwen3-0.6B-shaped models (151,936-token tied head) against the oracle,
teacher-forced, in the launch configuration the benchmark times."""
import pytest

from quantized_gemv_gb300 import synthetic as S
from tests.gpu_util import compare_step, make_pair

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["qwen3_0.6b_bf16", "qwen3_0.6b_fp8", "qwen3_0.6b_nvfp4", "qwen3_0.6b_fp8_bf16head"])
def test_full_model_prompt_then_greedy(name):
    wl = S.WORKLOADS[name]
    cfg = wl.config()
    _, model, om = make_pair(cfg, wl.variant, seed=0)
    prompt = S.prompt_ids(cfg, wl.prompt_len)
    tok = int(prompt[0])
    n = wl.prompt_len + 8
    matches = 0
    for pos in range(n):
        o_next, st = compare_step(model, om, tok, pos, check_hidden=(pos % 8 == 7))
        matches += st["match"]
        tok = int(prompt[pos + 1]) if pos + 1 < wl.prompt_len else o_next
    assert matches >= n - 1


def test_full_model_long_context():
    wl = S.WORKLOADS["qwen3_0.6b_fp8_ctx4096"]
    cfg = wl.config()
    _, model, om = make_pair(cfg, wl.variant, seed=0, prefill=wl.prefill)
    tok = int(S.prompt_ids(cfg, 1)[0])
    for pos in range(wl.prefill, wl.prefill + 4):
        tok, _ = compare_step(model, om, tok, pos, check_hidden=(pos == wl.prefill))
