"""GPU: the decode megakernel against the oracle (teacher-forced), at small vocab and real width."""
import numpy as np
import pytest
import torch

from quantized_gemv_gb300 import mk
from quantized_gemv_gb300 import synthetic as S
from tests.gpu_util import compare_step, make_pair

pytestmark = pytest.mark.gpu

SMALL = S.ModelConfig(n_layers=2, vocab=4099, max_ctx=1024)


@pytest.mark.parametrize("variant", ["bf16", "fp8", "nvfp4", "fp8_bf16head", "nvfp4_mse", "nvfp4_all", "fp8_bf16scale"])
def test_small_model_prompt_and_greedy(variant):
    master, model, om = make_pair(SMALL, variant, seed=31)
    prompt = S.prompt_ids(SMALL, 8)
    tok = int(prompt[0])
    stats = []
    for pos in range(24):
        o_next, st = compare_step(model, om, tok, pos)
        stats.append(st)
        tok = int(prompt[pos + 1]) if pos + 1 < len(prompt) else o_next
    assert sum(s["match"] for s in stats) >= len(stats) - 1


def test_layer1_bf16_full_vocab_prefill16():
    """One bf16 layer + tied 151,936-row head, KV prefilled with 16 positions, one step at pos 16."""
    cfg = S.WORKLOADS["layer1_bf16"].config()
    _, model, om = make_pair(cfg, "bf16", seed=0, prefill=16)
    tok = int(S.prompt_ids(cfg, 1)[0])
    _, st = compare_step(model, om, tok, 16)
    assert st["match"] or st["gap"] < 1e-3


@pytest.mark.parametrize("prefill", [100, 700])
def test_attention_split_over_units(prefill):
    """Contexts long enough for several attention units per KV head and several KV tiles each."""
    cfg = S.ModelConfig(n_layers=1, vocab=1000, max_ctx=1024)
    _, model, om = make_pair(cfg, "fp8", seed=41, prefill=prefill)
    tok = 5
    for pos in range(prefill, prefill + 3):
        tok, _ = compare_step(model, om, tok, pos)


def test_long_context_4096():
    cfg = S.ModelConfig(n_layers=1, vocab=2000, max_ctx=4224)
    _, model, om = make_pair(cfg, "fp8", seed=42, prefill=4096)
    tok = 17
    for pos in range(4096, 4099):
        tok, _ = compare_step(model, om, tok, pos)


def test_deterministic_three_runs():
    cfg = SMALL
    master, model, _ = make_pair(cfg, "fp8", seed=51)
    runs = []
    for _ in range(3):
        outs = []
        for pos, tok in enumerate([3, 99, 1024, 7]):
            lg = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
            nxt = model.decode_step(tok, pos, lg)
            outs.append((nxt, lg.cpu().numpy().copy(), model.hidden().cpu().numpy().copy()))
        runs.append(outs)
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert a[0] == b[0]
            assert np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))
            assert np.array_equal(a[2].view(np.uint32), b[2].view(np.uint32))


def test_greedy_on_device_matches_stepwise():
    cfg = SMALL
    _, model, _ = make_pair(cfg, "nvfp4", seed=61)
    seq, tok = [], 11
    for pos in range(10):
        tok = model.decode_step(tok, pos)
        seq.append(tok)
    toks = model.decode_greedy(11, 0, 10)
    model.sync()
    assert toks.cpu().tolist() == seq


def test_timeout_is_reported_and_model_recovers():
    cfg = SMALL
    _, model, _ = make_pair(cfg, "fp8", seed=71)
    ref = model.decode_step(5, 0)
    model.debug_fault(cta=3, phase=0, timeout_ms=50)   # CTA 3 never signals its q/k/v rows
    with pytest.raises(mk.MkError) as ei:
        model.decode_step(5, 0)
    assert ei.value.code == mk.MK_ETIMEOUT
    model.debug_fault(cta=-1, phase=-1, timeout_ms=500)
    assert model.decode_step(5, 0) == ref


def test_invalid_arguments_are_rejected():
    cfg = SMALL
    _, model, _ = make_pair(cfg, "bf16", seed=81)
    for tok, pos in ((-1, 0), (cfg.vocab, 0), (0, -1), (0, cfg.max_ctx)):
        with pytest.raises(mk.MkError) as ei:
            model.decode_step(tok, pos)
        assert ei.value.code == mk.MK_EINVAL


def test_models_after_set_device_round_trip():
    """Function attributes (the 232 KB shared-memory opt-in) are applied per device: models made
    after switching the current device away and back, and on every visible device, still launch."""
    cfg = S.ModelConfig(n_layers=1, vocab=1031, max_ctx=64)
    master = S.master_weights(cfg, seed=83)
    ref = None
    for dev in list(range(torch.cuda.device_count())) + [0]:
        torch.cuda.set_device(dev)
        model = mk.Model(cfg, mk.pack_model(master, S.format_map("fp8"), device=f"cuda:{dev}"))
        tok = model.decode_step(9, 0)
        ref = tok if ref is None else ref
        assert tok == ref
        model.close()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("variant", ["bf16", "fp8", "nvfp4"])
def test_folded_o_projection_matches_unfolded(variant):
    """The folded O-projection (attention on every CTA, W_o blocks, count-word accumulators) and
    the o_proj GEMV step compute the same step up to fp32 rounding; both follow the oracle."""
    cfg = S.ModelConfig(n_layers=2, vocab=4099, max_ctx=512)
    master = S.master_weights(cfg, seed=77)
    packed = mk.pack_model(master, S.format_map(variant))
    fold = mk.Model(cfg, packed)
    plain = mk.Model(cfg, packed, flags=mk.MK_FLAG_NO_FOLD)
    toks = S.prompt_ids(cfg, 300, seed=8)
    worst = 0.0
    for pos in range(300):
        la = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
        lb = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
        fold.decode_step(int(toks[pos]), pos, la)
        plain.decode_step(int(toks[pos]), pos, lb)
        worst = max(worst, float((la - lb).abs().max()))
    # positions 288 and later take the unfolded path in both models
    assert worst <= 1e-3, worst
    fold.close()
    plain.close()


@pytest.mark.parametrize("variant", ["bf16", "nvfp4"])
def test_stress_delays_change_nothing(variant):
    """Seeded per-CTA waits before every step reorder the CTAs' arrivals at every exchange (and at
    the folded O-projection's accumulators); tokens, logits and hidden states stay bit-identical,
    at short contexts and at one past the single-unit attention window."""
    cfg = S.ModelConfig(n_layers=2, vocab=4099, max_ctx=512)
    _, model, _ = make_pair(cfg, variant, seed=87)
    toks = S.prompt_ids(cfg, 300, seed=12)
    checked = (3, 40, 288, 290)

    def run(seed):
        model.debug_stress(seed)
        out = []
        for pos in range(max(checked) + 1):
            lg = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
            nxt = model.decode_step(int(toks[pos]), pos, lg)
            if pos in checked:
                out.append((nxt, lg.cpu().numpy().copy(), model.hidden().cpu().numpy().copy()))
        return out

    ref = run(0)
    for seed in (1, 2):
        for a, b in zip(ref, run(seed)):
            assert a[0] == b[0]
            assert np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))
            assert np.array_equal(a[2].view(np.uint32), b[2].view(np.uint32))
    model.debug_stress(0)
    model.close()
