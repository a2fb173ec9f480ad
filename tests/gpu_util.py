"""Helpers for the GPU parity tests: build a device model and an oracle model from the same
seeded bf16 masters, and compare their outputs."""
import numpy as np
import torch

from oracle import oracle as O
from quantized_gemv_gb300 import mk
from quantized_gemv_gb300 import synthetic as S
from tests._helpers import oracle_pack_model


def make_pair(cfg, variant, seed=0, prefill=0, kv_seed=2, flags=0, oracle_threads=None):
    master = S.master_weights(cfg, seed=seed)
    fmap = S.format_map(variant)
    dev_packed = mk.pack_model(master, fmap)
    model = mk.Model(cfg, dev_packed, flags=flags)
    om = O.OracleModel(cfg, oracle_pack_model(master, fmap, oracle_threads), n_threads=oracle_threads)
    if prefill:
        k, v = S.prefill_kv(cfg, prefill, seed=kv_seed)
        om.set_kv(k, v)
        for l in range(cfg.n_layers):
            kt, vt = model.kv_cache(l)
            kt[:, :prefill].copy_(mk.upload_bf16(k[l]))
            vt[:, :prefill].copy_(mk.upload_bf16(v[l]))
        torch.cuda.synchronize()
    return master, model, om


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


# tolerances stated by the parity target: per-layer hidden states rel L2 <= 1e-2, logits max abs
# <= 2e-2, greedy tokens exact unless the oracle's top-2 gap is below 1e-3
HIDDEN_RTOL = 1e-2
LOGIT_ATOL = 2e-2
TIE_GAP = 1e-3


def compare_step(model, om, token, pos, check_hidden=True):
    """Run one step on both sides (teacher-forced input `token`); assert parity; return the
    oracle's token and diagnostics."""
    logits = torch.empty(model.cfg.vocab, dtype=torch.float32, device="cuda")
    nxt = model.decode_step(token, pos, logits)
    o_next, o_logits, o_hidden, top2 = om.step(token, pos, want_logits=True, want_hidden=check_hidden)
    lg = logits.cpu().numpy().astype(np.float64)
    max_abs = float(np.max(np.abs(lg - o_logits)))
    assert max_abs <= LOGIT_ATOL, (pos, max_abs)
    worst_h = 0.0
    if check_hidden:
        hid = model.hidden().cpu().numpy()
        for l in range(hid.shape[0]):
            e = rel_l2(hid[l], o_hidden[l])
            worst_h = max(worst_h, e)
            assert e <= HIDDEN_RTOL, (pos, l, e)
    gap = float(top2[0] - top2[1])
    if nxt != o_next:
        assert gap < TIE_GAP, (pos, nxt, o_next, gap)
    return o_next, {"max_abs_logit": max_abs, "worst_hidden_rel": worst_h, "gap": gap, "match": nxt == o_next}
