"""X-ray: the analyser on a hand-built trace (CPU), and the instrumented build on the GPU (same
tokens and logits as the plain build, well-formed per-CTA records)."""
import numpy as np
import pytest
import torch

from quantized_gemv_gb300 import xray

TRACE_DTYPE = np.dtype([("gtime", "<u8"), ("clk", "<u8"), ("smid", "<u4"), ("cta", "<u2"),
                        ("phase", "u1"), ("kind", "u1")])
B, E, WB, WE, MARK, STOP = 0, 1, 2, 3, 4, 255
QKV, ATT, O, GU, DOWN, HEAD, EMBED = 0, 1, 2, 3, 4, 5, 6


def _trace(rows_per_cta, width=64, clock_only_begins=False):
    """Records {t, clk = 7 t + 1}; with clock_only_begins, only the embedding's stamps, the start of
    each wait on the down phase and the LM head's end keep the global time (the others gtime 0), as
    the kernel writes them."""
    tr = np.zeros((len(rows_per_cta), width), dtype=TRACE_DTYPE)
    for c, rows in enumerate(rows_per_cta):
        for i, (t, ph, kind) in enumerate(rows + [(0, 0, STOP)]):
            anchor = ph == EMBED or (ph == HEAD and kind == E) or (ph == DOWN and kind == WB)
            g = 0 if (clock_only_begins and kind != MARK and not anchor) else t
            tr[c][i] = (g, 7 * t + 1, 3, c, ph, kind)
    return tr


def _one_layer(t0, wait_before_o):
    """Records of one CTA for one layer (ns from t0) with a sub-phase mark that carries no time."""
    return [(t0, QKV, B), (0, 40, MARK), (t0 + 100, QKV, E),
            (t0 + 100, ATT, WB), (t0 + 100 + wait_before_o, ATT, WE), (t0 + 110 + wait_before_o, O, B),
            (t0 + 160 + wait_before_o, O, E), (t0 + 160 + wait_before_o, O, WB), (t0 + 170 + wait_before_o, O, WE),
            (t0 + 170 + wait_before_o, GU, B), (t0 + 250 + wait_before_o, GU, E),
            (t0 + 250 + wait_before_o, GU, WB), (t0 + 260 + wait_before_o, GU, WE),
            (t0 + 260 + wait_before_o, DOWN, B), (t0 + 300 + wait_before_o, DOWN, E)]


def test_analyze_hand_trace():
    a = [(1000, EMBED, B), (1010, EMBED, E)] + _one_layer(1010, 40) + [(1350, DOWN, WB), (1360, DOWN, WE),
                                                                       (1360, HEAD, B), (1500, HEAD, E)]
    b = [(1005, EMBED, B), (1012, EMBED, E)] + _one_layer(1012, 20) + [(1332, DOWN, WB), (1340, DOWN, WE),
                                                                       (1340, HEAD, B), (1480, HEAD, E)]
    tr = _trace([a, b])
    # marks (kind 4, gtime 0) are not phase records
    assert all(k != MARK for _, recs in xray.records(tr) for _, _, k in recs)
    r = xray.analyze(tr)
    assert r["ctas"] == 2
    assert r["token_ns"] == 1500 - 1000
    # waits: CTA a 40 + 10 + 10 + 10 = 70, CTA b 20 + 10 + 10 + 8 = 48
    assert r["barrier_wait_ns"] == pytest.approx((70 + 48) / 2)
    # GEMV phases: qkv 100 + o 50 + gu 80 + down 40 = 270 for both
    assert r["weight_read_ns"] == pytest.approx(270)
    assert r["lm_head_ns"] == pytest.approx((140 + 140) / 2)
    # idle: a ends last (1500); b ends at 1480
    assert r["idle_ns"] == pytest.approx(10)
    assert xray.layer_timeline(tr) == []  # one layer: no layer-to-layer interval


def test_clock_only_begin_stamps_are_placed_by_interpolation():
    a = [(1000, EMBED, B), (1010, EMBED, E)] + _one_layer(1010, 40) + [(1350, DOWN, WB), (1360, DOWN, WE),
                                                                       (1360, HEAD, B), (1500, HEAD, E)]
    b = [(1005, EMBED, B), (1012, EMBED, E)] + _one_layer(1012, 20) + [(1332, DOWN, WB), (1340, DOWN, WE),
                                                                       (1340, HEAD, B), (1480, HEAD, E)]
    full, sparse = _trace([a, b]), _trace([a, b], clock_only_begins=True)
    assert (sparse["gtime"] == 0).sum() > (full["gtime"] == 0).sum()
    assert dict(xray.records(full)) == dict(xray.records(sparse))
    assert xray.analyze(full) == xray.analyze(sparse)


@pytest.mark.gpu
def test_instrumented_build_matches_plain_build():
    from quantized_gemv_gb300 import mk
    from quantized_gemv_gb300 import synthetic as S

    cfg = S.ModelConfig(n_layers=2, vocab=4099, max_ctx=256)
    master = S.master_weights(cfg, seed=61)
    packed = mk.pack_model(master, S.format_map("fp8"))
    plain = mk.Model(cfg, packed)
    xr = mk.Model(cfg, packed, flags=mk.MK_FLAG_XRAY | mk.MK_FLAG_XRAY_MARKS)
    tok = 3
    for pos in range(6):  # teacher-forced on the plain build's tokens
        lp = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
        lx = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
        nxt = plain.decode_step(tok, pos, lp)
        nxt_x = xr.decode_step(tok, pos, lx)
        # the same arithmetic in both builds (a different compilation may contract differently)
        assert torch.allclose(lp, lx, rtol=0, atol=1e-4)
        top2 = torch.topk(lp, 2).values
        assert nxt_x == nxt or float(top2[0] - top2[1]) < 1e-3
        tok = nxt
    tr = xr.trace()
    grid = mk.decode_grid()
    assert tr.shape == (grid, mk.TRACE_PER_CTA)
    written = []
    for c in range(grid):
        stop = np.flatnonzero(tr[c]["kind"] == STOP)
        assert len(stop) > 0, c  # every CTA ended its row (the rest of the buffer is not this step's)
        written.append(tr[c][: stop[0]])
    written = np.concatenate(written)
    assert set(np.unique(written["kind"]).tolist()) <= {B, E, WB, WE, MARK}
    marks = written[written["kind"] == MARK]
    assert len(marks) > 0 and np.all(marks["gtime"] == 0) and np.all(marks["clk"] > 0)
    for cta, recs in xray.records(tr):
        begins = [ph for _, ph, k in recs if k == B]
        # every CTA runs the four GEMV phases of each layer, then the LM head
        for ph in (QKV, O, GU, DOWN):
            assert begins.count(ph) == cfg.n_layers, (cta, ph)
        assert begins.count(HEAD) == 1
        ts = [t for t, _, _ in recs]
        assert ts == sorted(ts)
    r = xray.analyze(tr)
    assert r["ctas"] == grid
    for k in ("weight_read_ns", "barrier_wait_ns", "lm_head_ns"):
        assert 0 <= r[k] <= r["token_ns"]
    plain.close()
    xr.close()


@pytest.mark.parametrize("suffix", [".json", ".json.gz"])
def test_export_round_trip(tmp_path, suffix):
    a = [(1000, EMBED, B), (1010, EMBED, E)] + _one_layer(1010, 40)
    b = [(1005, EMBED, B), (1012, EMBED, E)] + _one_layer(1012, 20)
    tr = _trace([a, b])
    path = str(tmp_path / ("trace" + suffix))
    xray.export_json(tr, path, meta={"workload": "hand-built"})
    doc = xray.load_json(path)
    assert doc["meta"] == {"workload": "hand-built"}
    assert sorted(doc["ctas"]) == ["0", "1"]
    # times are relative to the first record of the token; marks are not exported
    assert doc["ctas"]["0"][0] == [0, EMBED, B]
    assert doc["ctas"]["1"][0] == [5, EMBED, B]
    assert len(doc["ctas"]["0"]) == len(a) - 1
    assert all(k != MARK for recs in doc["ctas"].values() for _, _, k in recs)


def test_layer_timeline_two_layers():
    # two layers: the interval between the last CTA's ends of down_proj
    a = _one_layer(100, 40) + _one_layer(500, 40)
    b = _one_layer(110, 20) + _one_layer(480, 20)
    tr = _trace([a, b])
    # CTA a ends down_proj at 440 and 840, CTA b at 430 and 800 (an all-zero record ends a row, so
    # no record sits at time 0)
    assert xray.layer_timeline(tr) == [840 - 440]


def test_critical_path_three_layers():
    # three identical layers per CTA, 400 ns apart; CTA b is 10 ns behind CTA a everywhere
    a = [(1000, EMBED, B), (1010, EMBED, E)]
    b = [(1000, EMBED, B), (1012, EMBED, E)]
    for l in range(3):
        t0 = 1100 + 400 * l
        a += ([(t0 - 20, DOWN, WB), (t0 - 5, DOWN, WE)] if l else []) + _one_layer(t0, 40)
        b += ([(t0 - 15, DOWN, WB), (t0 + 5, DOWN, WE)] if l else []) + _one_layer(t0 + 10, 40)
    tr = _trace([a, b], width=128)
    cp = xray.critical_path(tr)
    assert cp["layers"] == 3
    # layer 1 (t0 = 1500): o_proj's wait ends at t0 + 140 (a) and t0 + 150 (b); its phase ends at
    # t0 + 200 / t0 + 210; QKV ends at t0 + 100 / t0 + 110
    assert cp["phase_o_proj"] == 210 - 150
    assert cp["exchange_o_proj_first"] == 140 - 110
    assert cp["exchange_o_proj_last"] == 150 - 110
    # QKV of layer 1 waits for layer 0's down_proj (ends 1100 + 340 and 1110 + 340)
    assert cp["exchange_qkv_last"] == (1500 + 5) - (1110 + 340)
    assert cp["phase_qkv"] == (1510 + 100) - (1500 + 5)
    assert cp["layer"] == 400


@pytest.mark.gpu
def test_stamps_only_build_has_no_marks_and_spans_the_launch():
    """MK_FLAG_XRAY alone records phase and wait stamps only (no sub-phase marks), and on a
    28-layer model the span from the first to the last stamp of a step is within 5 % of that
    launch's CUDA-event time inside a back-to-back run (the X-ray milestone's check that the
    phases account for the token)."""
    from quantized_gemv_gb300 import mk
    from quantized_gemv_gb300 import synthetic as S

    cfg = S.ModelConfig(n_layers=28, vocab=4099, max_ctx=256)
    packed = mk.pack_model(S.master_weights(cfg, seed=62), S.format_map("bf16"))
    xr = mk.Model(cfg, packed, flags=mk.MK_FLAG_XRAY)
    n = 8
    toks = torch.zeros(n + 1, dtype=torch.int32, device="cuda")
    toks[0] = 5
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    torch.cuda.synchronize()
    with torch.cuda.stream(xr.stream):
        for i in range(n):
            ev[i].record(xr.stream)
            xr.decode_next(toks[i: i + 1], i, toks[i + 1: i + 2])
        ev[n].record(xr.stream)
    xr.sync()
    launch_ns = ev[n - 1].elapsed_time(ev[n]) * 1e6
    tr = xr.trace()
    kinds = set()
    for c in range(tr.shape[0]):
        stop = np.flatnonzero(tr[c]["kind"] == STOP)
        kinds |= set(np.unique(tr[c][: stop[0]]["kind"]).tolist())
    assert kinds <= {B, E, WB, WE}  # no sub-phase marks
    for cta, recs in xray.records(tr):  # every CTA's stamps reached the trace, in order
        begins = [ph for _, ph, k in recs if k == B]
        for ph in (QKV, GU, DOWN):
            assert begins.count(ph) == cfg.n_layers, (cta, ph)
        assert begins.count(HEAD) == 1
        ts = [t for t, _, _ in recs]
        assert ts == sorted(ts)
    span = xray.analyze(tr)["token_ns"]
    assert 0.95 * launch_ns <= span <= launch_ns, (span, launch_ns)
    xr.close()

