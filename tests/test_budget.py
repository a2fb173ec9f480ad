"""The model shape and the bytes a decode step streams, against the figures the monolith page prints
("Upstream facts": weights read per step, derived weight counts; the byte-budget table that follows
it). The roofline in bench.py divides by these bytes, so they are pinned here."""
import pytest

import bench
from quantized_gemv_gb300 import synthetic as S

CFG = S.QWEN3_06B
MB = 1e6


def test_weight_counts_match_the_page():
    sh = CFG.shapes()
    attn = sum(r * c for n, (r, c) in sh.items() if n in ("q", "k", "v", "o"))
    mlp = sum(r * c for n, (r, c) in sh.items() if n in ("gate", "up", "down"))
    assert attn == 6_291_456 and round(attn / 1e6, 2) == 6.29   # "about 6.29M"
    assert mlp == 9_437_184 and round(mlp / 1e6, 2) == 9.44     # "about 9.44M"
    assert round((attn + mlp) / 1e6, 1) == 15.7                  # "about 15.7M per layer"
    embed = CFG.vocab * CFG.hidden
    assert round(embed / 1e6, 1) == 155.6                        # "about 155.6M"
    assert round((CFG.n_layers * (attn + mlp) + embed) / 1e6) == 596  # "about 596M"


def test_bf16_bytes_per_step_match_the_page():
    total = bench.weight_bytes(CFG, "bf16")
    head = 2 * CFG.vocab * CFG.hidden
    layers = total - head - 2 * CFG.hidden  # minus the final norm
    assert total == 1_192_099_840
    assert round(layers / MB, 1) == 880.9   # "880.9 MB for the 28 layers"
    assert round(head / MB, 1) == 311.2     # "311.2 MB for the LM head"
    assert round(total / MB, 1) == 1192.1   # "1,192.1 MB"


@pytest.mark.parametrize("variant,exact,approx_gb", [
    ("fp8", 598_099_456, 0.60),          # per-output-channel scales, LM head FP8
    ("nvfp4_all", 404_048_144, 0.40),    # every linear NVFP4 (4.5 bits a weight), LM head FP8
    ("nvfp4", 442_697_888, None),        # down_proj kept FP8 as well: the workload configuration
])
def test_quantised_bytes_per_step(variant, exact, approx_gb):
    b = bench.weight_bytes(CFG, variant)
    assert b == exact
    if approx_gb is not None:
        assert round(b / 1e9, 2) == approx_gb


def test_nvfp4_is_four_and_a_half_bits_a_weight():
    # codes (4 bits) + one E4M3 scale per 16 (0.5 bit) per weight, plus a 4-byte tensor scale
    r, c = CFG.shapes()["gate"]
    per = {S.FMT_NVFP4: r * c // 2 + r * c // 16 + 4}
    assert per[S.FMT_NVFP4] * 8 / (r * c) == pytest.approx(4.5, abs=1e-4)


def test_kv_bytes_per_position():
    # K and V, bf16, 8 KV heads of 128, 28 layers: read for every cached position, written for pos
    assert bench.kv_bytes(CFG, 0) == 28 * 8 * 128 * 2 * 2 == 114_688
    assert bench.kv_bytes(CFG, 4095) == 114_688 * 4096
