"""Benchmark: batch-1 greedy decode of a Qwen3-0.6B-shaped model, one megakernel launch per token.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A "step" is one decode step: one launch of the decode kernel producing one token (embedding,
28 layers, final norm, LM head and argmax). The timed region holds exactly K steps (positions
P..P+K-1 after the workload's 32-token prompt or prefilled KV), launched back to back with the
input token of each launch read from device memory; it is bracketed by a barrier and
torch.cuda.synchronize() and timed with CUDA events on the launching stream. Warm-up runs the
same positions W times first. Every step streams >= 0.4 GB of weights, more than the L2 holds,
so no L2 flush is needed between steps.

Extra keys beyond the base contract: `roofline` (the decode kernel against the measured HBM copy
bandwidth), `runs` (five more timed regions of the same K steps: median, min and max, the pages'
benchmark protocol), `cpu_baseline` (the CPU oracle on this host's cores in a fresh process, a
bounded sample, with a one-thread figure), `e2e` (the same metric through mk_decode_step, which
returns each token to the host), `clocks` (NVML samples during the timed region),
`stream_read_gbs` (the library's bulk-copy streaming-read probe, same run), `variants` (the FP8,
NVFP4 (amax and searched block scales; all-NVFP4), bf16-head FP8, bf16-scale FP8 and long-context
FP8 workloads, each timed the same way), `xray` (the instrumented build's split of a token, its
overhead against the plain build over the same positions and its span against the launch time,
for the headline and the long-context workload),
`layer1_bf16` (one layer + the LM head, timed cold after an L2 scrub and warm) and `sweep`
(throughput and energy against context length, FP8).

--impl reference times the CPU oracle (the only reference implementation of this method) on the
same workload and positions and prints its line with "impl": "reference". Under torchrun, rank 0
alone runs it. Multi-GPU: each rank decodes its own independent replica (the path has no
data-parallel exchange); value = tokens of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_gemv_gb300 import synthetic as S  # noqa: E402

HEADLINE = "qwen3_0.6b_bf16"
UPSTREAM_BF16_TOKS = 1033.0  # RTX 5090 upstream kernel, bf16 (monolith page, "Upstream facts")
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (about 8 TB/s); the roofline divides by the measured copy


# ------------------------------------------------------------------ byte accounting
def weight_bytes(cfg: S.ModelConfig, variant: str) -> int:
    """Bytes of every weight and scale one decode step reads (embedding row excluded)."""
    fmap = S.format_map(variant)
    per = {S.FMT_BF16: lambda r, c: 2 * r * c, S.FMT_FP8_ROW: lambda r, c: r * c + 4 * r,
           S.FMT_NVFP4: lambda r, c: r * c // 2 + r * c // 16 + 4}
    total = 0
    for name, (r, c) in cfg.shapes().items():
        total += per[fmap[name]](r, c)
    total += 2 * (2 * cfg.hidden + 2 * cfg.head_dim)  # norm weights
    total *= cfg.n_layers
    total += per[fmap["embed"]](cfg.vocab, cfg.hidden) + 2 * cfg.hidden  # LM head + final norm
    return total


def kv_bytes(cfg: S.ModelConfig, pos: int) -> int:
    """KV-cache bytes one step at `pos` reads (positions 0..pos-1) and writes (position pos)."""
    per_pos = cfg.n_layers * cfg.n_kv_heads * cfg.head_dim * 2 * 2
    return per_pos * (pos + 1)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_gemv_gb300", "csrc")
    for n in sorted(os.listdir(csrc)):
        if n.startswith("mk_kernel") or n.endswith((".cuh", ".h")):
            with open(os.path.join(csrc, n), "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks (read-only NVML)
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (read-only queries) in a thread."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake",
               0x100: "display_clocks"}

    def __init__(self, index: int):
        self.ok = False
        self.samples = []
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            p = torch.cuda.get_device_properties(index)
            bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0".encode()
            if self.nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(self.h)) != 0:
                return
            self.read()
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def read(self):
        clk, mx, rs, mw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk))       # NVML_CLOCK_SM
        self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
        self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs))
        if self.nv.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(mw)) != 0:  # board power, mW
            mw.value = 0
        return clk.value, mx.value, rs.value, mw.value

    def __enter__(self):
        self._stop = False
        if self.ok:
            self.samples.append(self.read())

            def loop():
                while not self._stop:
                    self.samples.append(self.read())
                    time.sleep(0.002)
            self.t = threading.Thread(target=loop, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        self._stop = True
        if self.ok:
            self.t.join()
            self.samples.append(self.read())

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        reasons = set()
        for _, _, r, _ in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit and name != "gpu_idle":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": max(s[1] for s in self.samples), "samples": len(self.samples),
                "reasons": sorted(reasons)}

    def watts(self):
        """Median board power over the samples (W), or None."""
        p = [s[3] for s in self.samples if s[3] > 0]
        return statistics.median(p) / 1e3 if p else None


# ------------------------------------------------------------------ GPU arm
def setup_model(wl: S.Workload, mk, flags: int = 0, master=None):
    cfg = wl.config()
    if master is None:
        master = S.master_weights(cfg, seed=0)
    packed = mk.pack_model(master, S.format_map(wl.variant))
    model = mk.Model(cfg, packed, flags=flags)
    start_pos = 0
    if wl.prefill:
        k, v = S.prefill_kv(cfg, wl.prefill, seed=2)
        for l in range(cfg.n_layers):
            kt, vt = model.kv_cache(l)
            kt[:, : wl.prefill].copy_(mk.upload_bf16(k[l]))
            vt[:, : wl.prefill].copy_(mk.upload_bf16(v[l]))
        start_pos = wl.prefill
        first = int(S.prompt_ids(cfg, 1)[0])
    else:
        prompt = S.prompt_ids(cfg, wl.prompt_len)
        tok = int(prompt[0])
        for pos in range(wl.prompt_len):  # prompt fed token by token, untimed
            nxt = model.decode_step(tok, pos)
            tok = int(prompt[pos + 1]) if pos + 1 < wl.prompt_len else nxt
        start_pos = wl.prompt_len
        first = tok
    torch.cuda.synchronize()
    return cfg, master, model, start_pos, first


def time_steps(model, first: int, pos0: int, k: int, warmup: int, dist=None):
    """Time exactly k launches; returns (total_ms, per-launch ms list, tokens)."""
    dev = torch.device("cuda")
    toks = torch.zeros(k + 1, dtype=torch.int32, device=dev)
    stream = model.stream

    def run(n):
        toks[0] = first
        for i in range(n):
            model.decode_next(toks[i: i + 1], pos0 + i, toks[i + 1: i + 2])

    for _ in range(max(warmup, 0)):
        run(min(k, 8))
    model.sync()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(k + 1)]
    toks[0] = first
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(k):
            ev[i].record(stream)
            model.decode_next(toks[i: i + 1], pos0 + i, toks[i + 1: i + 2])
        ev[k].record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    model.sync()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(k)]
    total = ev[0].elapsed_time(ev[k])
    return total, per, toks[1:].cpu().numpy()


def time_e2e(model, first: int, pos0: int, k: int):
    """Per-token host loop through mk_decode_step: the token goes in with the launch and comes back
    to the host before the next step is issued."""
    tok = first
    model.decode_step(tok, pos0)  # warm
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(k):
        tok = model.decode_step(tok, pos0 + i)
    return (time.perf_counter() - t0) * 1e3


def stream_read_gbs(mk):
    unit = 16384 * mk.decode_grid()
    n = (2 << 30) // unit * unit
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        mk.stream_read(buf)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = 1e9
    for _ in range(5):
        e0.record()
        mk.stream_read(buf)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    del buf
    return n / (best * 1e-3) / 1e9


def oracle_sample(wl: S.Workload, master, seconds: float = 12.0, steps: int | None = None, warmup: int = 0,
                  budget_s: float = 150.0, threads: int | None = None):
    """The CPU oracle decoding the same workload on this host's cores, at the positions the GPU arm
    times: the prompt (or the prefilled KV cache) first, untimed, then `warmup` untimed greedy
    steps from the first timed position, then timed greedy steps from that same position again
    (they rewrite the same cache rows with the same values): `steps` of them, or as many as fit in
    `seconds` when steps is None, and never more than fit in `budget_s` (the sample says how many
    were timed). `threads`: oracle threads (default: every core this process may use)."""
    from oracle import oracle as O
    cfg = wl.config()
    cores = len(os.sched_getaffinity(0)) if threads is None else int(threads)
    packed = O.pack_model(master, S.format_map(wl.variant), len(os.sched_getaffinity(0)))
    om = O.OracleModel(cfg, packed, n_threads=cores)
    if wl.prefill:
        k, v = S.prefill_kv(cfg, wl.prefill, seed=2)
        om.set_kv(k, v)
        pos0, tok0 = wl.prefill, int(S.prompt_ids(cfg, 1)[0])
    else:
        prompt = S.prompt_ids(cfg, wl.prompt_len)
        tok = int(prompt[0])
        for pos in range(wl.prompt_len):
            nxt, _, _, _ = om.step(tok, pos, want_logits=False)
            tok = int(prompt[pos + 1]) if pos + 1 < wl.prompt_len else nxt
        pos0, tok0 = wl.prompt_len, tok
    tok, pos = tok0, pos0
    for _ in range(max(warmup, 0)):
        tok, _, _, _ = om.step(tok, pos, want_logits=False)
        pos += 1
    tok, pos, n, t0 = tok0, pos0, 0, time.perf_counter()
    while True:
        tok, _, _, _ = om.step(tok, pos, want_logits=False)
        pos += 1
        n += 1
        el = time.perf_counter() - t0
        if steps is not None and n >= steps:
            break
        if steps is None and el >= seconds and n >= 2:
            break
        if el >= budget_s and n >= 2:
            break
    return {"value": n / el, "unit": "tok/s", "cores": cores, "kind": "oracle", "steps": n,
            "positions": f"{pos0}..{pos - 1}",
            "sample": f"{n} timed greedy steps of {wl.name} at positions {pos0}..{pos - 1} after "
                      f"{'the prefilled KV' if wl.prefill else 'the prompt'} and {max(warmup, 0)} untimed steps at "
                      f"the same positions ({el:.1f} s, double precision, {cores} threads)"}


def cpu_leg_subprocess(wl: S.Workload, seconds: float, one_thread_seconds: float):
    """The oracle timed in a fresh process (no CUDA context or torch thread pool competing with its
    threads): all cores, then one thread. Returns the all-core sample with the one-thread figure."""
    import subprocess
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-leg", "--workload", wl.name,
           "--cpu-seconds", str(seconds), "--cpu-seconds-1t", str(one_thread_seconds)]
    env = dict(os.environ, OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        return {"value": None, "unit": "tok/s", "kind": "oracle", "error": r.stderr[-400:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_cpu_leg(wl: S.Workload, seconds: float, one_thread_seconds: float):
    master = S.master_weights(wl.config(), seed=0)
    allc = oracle_sample(wl, master, seconds=seconds)
    one = oracle_sample(wl, master, seconds=one_thread_seconds, threads=1)
    allc["one_thread"] = {"value": one["value"], "steps": one["steps"], "sample": one["sample"]}
    allc["process"] = "a fresh process (no CUDA context), OMP_NUM_THREADS=1 for torch"
    print(json.dumps(allc))


def xray_summary(wl: S.Workload, mk, master, steps: int = 64, runs: int = 3):
    """The workload through the instrumented build (MK_FLAG_XRAY): the last step's split of a token
    into weight-read, wait, attention and LM-head time, the critical path per layer, and the X-ray
    milestone's two checks: instrumented throughput against the plain build's over the same
    positions (plain and instrumented regions alternate, `runs` each; medians) and the first-to-last
    stamp span of the last step against that launch's CUDA-event time."""
    from quantized_gemv_gb300 import xray
    cfg, master, plain, pos0, first = setup_model(wl, mk, master=master)
    _, _, inst, _, _ = setup_model(wl, mk, flags=mk.MK_FLAG_XRAY, master=master)
    k = min(steps, cfg.max_ctx - pos0)

    def rate(model):
        t_ms, per, _ = time_steps(model, first, pos0, k, 3)
        return k / (t_ms * 1e-3), per

    rp, ri = [], []
    for _ in range(runs):
        rp.append(rate(plain)[0])
        r, per = rate(inst)
        ri.append(r)
    tr = inst.trace()  # the last instrumented step
    a = xray.analyze(tr)
    cp = xray.critical_path(tr)
    plain.close()
    inst.close()
    t = a["token_ns"]
    p_med, i_med = float(np.median(rp)), float(np.median(ri))
    return {"token_us": round(t / 1e3, 1), "ctas": a["ctas"],
            "weight_read_share": round(a["weight_read_ns"] / t, 3), "barrier_wait_share": round(a["barrier_wait_share"], 3),
            "attention_share": round(a["attention_ns"] / t, 3), "lm_head_share": round(a["lm_head_ns"] / t, 3),
            "plain_tok_s": round(p_med, 1), "instrumented_tok_s": round(i_med, 1),
            "overhead_vs_plain": round(p_med / i_med - 1.0, 4),
            "last_launch_us": round(per[-1] * 1e3, 1),
            "span_over_launch": round(t / 1e3 / (per[-1] * 1e3), 4),
            "critical_path_us": {kk: round(v / 1e3, 3) for kk, v in cp.items() if kk != "layers"},
            "note": f"{runs} alternating regions of {k} steps from position {pos0} per build (medians); the split "
                    "is the last instrumented step's, shares of the token's wall time averaged over CTAs; "
                    "span_over_launch = first-to-last stamp / CUDA-event launch time"}


SWEEP_POSITIONS = (16, 128, 512, 1024, 2048)


def run_sweep(mk, steps: int = 32, warmup: int = 3):
    """Decode throughput and energy against context length: the FP8 model with the KV cache prefilled
    (seeded N(0,1) bf16) to each position, then `steps` greedy steps from there."""
    import dataclasses
    base = S.WORKLOADS["qwen3_0.6b_fp8"]
    cfg = dataclasses.replace(base.config(), max_ctx=max(SWEEP_POSITIONS) + steps + 8)
    master = S.master_weights(cfg, seed=0)
    packed = mk.pack_model(master, S.format_map(base.variant))
    model = mk.Model(cfg, packed)
    k_all, v_all = S.prefill_kv(cfg, max(SWEEP_POSITIONS), seed=2)
    for l in range(cfg.n_layers):
        kt, vt = model.kv_cache(l)
        kt[:, : max(SWEEP_POSITIONS)].copy_(mk.upload_bf16(k_all[l]))
        vt[:, : max(SWEEP_POSITIONS)].copy_(mk.upload_bf16(v_all[l]))
    first = int(S.prompt_ids(cfg, 1)[0])
    wbytes = weight_bytes(cfg, base.variant)
    rows = []
    for p0 in SWEEP_POSITIONS:
        sampler = ClockSampler(torch.cuda.current_device())
        with sampler:
            total_ms, per, _ = time_steps(model, first, p0, steps, warmup)
        tok_s = steps / (total_ms * 1e-3)
        w = sampler.watts()
        kv = kv_bytes(cfg, p0 + (steps - 1) // 2)
        rows.append({"pos": f"{p0}..{p0 + steps - 1}", "tok_s": round(tok_s, 1), "ms_per_step": round(total_ms / steps, 4),
                     "gbs_weights_kv": round((wbytes + kv) / (float(np.mean(per)) * 1e-3) / 1e9, 1),
                     "watts": round(w, 1) if w else None, "tok_per_joule": round(tok_s / w, 2) if w else None,
                     "clocks": sampler.summary()})
    model.close()
    return {"metric": "batch-1 decode tok/s and tokens per joule against context length (Qwen3-0.6B shape, FP8)",
            "unit": "tok/s", "higher_is_better": True, "steps_per_point": steps, "warmup": warmup,
            "data": "synthetic (seeded N(0,0.02) weights; KV cache prefilled N(0,1) bf16)", "sweep": rows}


def run_verify(mk, name: str = HEADLINE, ks=(1, 2, 4, 8), launches: int = 16, warmup: int = 3):
    """The batched verify step (tensor cores): verified tokens per second for k tokens a launch, on
    the workload's model after its prompt; launch i verifies k seeded uniform-random tokens at
    positions P + i k .. P + i k + k - 1. Each launch reads every weight once (the 16-bit copy the
    verify step streams), so its weight stream is reported against the measured copy bandwidth."""
    wl = S.WORKLOADS[name]
    cfg, _, model, pos0, _ = setup_model(wl, mk)
    model.verify_attach()
    stream = model.stream
    toks = torch.tensor(S.prompt_ids(cfg, 8 * (launches + warmup), seed=5), dtype=torch.int32, device="cuda")
    nxt = torch.zeros(8, dtype=torch.int32, device="cuda")
    vbytes = 2 * sum(r * c for r, c in cfg.shapes().values()) * cfg.n_layers + 2 * cfg.vocab * cfg.hidden
    peak, _ = measured_peaks()
    rows = []
    for k in ks:
        if pos0 + k * (launches + warmup) > min(cfg.max_ctx, 1024):
            continue
        for i in range(warmup):
            model.verify_step(toks[k * i: k * i + k], pos0 + k * i, nxt[:k])
        model.sync()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(launches + 1)]
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for i in range(launches):
                ev[i].record(stream)
                model.verify_step(toks[k * i: k * i + k], pos0 + k * i, nxt[:k])
            ev[launches].record(stream)
        model.sync()
        per = [ev[i].elapsed_time(ev[i + 1]) for i in range(launches)]
        ms = ev[0].elapsed_time(ev[launches]) / launches
        gbs = vbytes / (float(np.mean(per)) * 1e-3) / 1e9
        rows.append({"k": k, "verified_tok_s": round(k / (ms * 1e-3), 1), "ms_per_launch": round(ms, 4),
                     "weight_gbs": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak, 4),
                     "positions": f"{pos0}..{pos0 + k * launches - 1}"})
    model.close()
    return {"workload": name, "launches": launches, "warmup": warmup, "weight_bytes_per_launch": vbytes,
            "note": "one launch per k tokens (tcgen05 GEMMs, fp32 accumulation); tokens seeded uniform, "
                    "so this measures verify throughput, not an acceptance rate", "rows": rows}


def run_workload(wl: S.Workload, steps: int, warmup: int, mk, dist=None, e2e_steps: int | None = None,
                 runs: int = 5):
    """The contract's timed region of `steps` launches, then `runs` more regions of the same
    positions for the median / min / max the pages' benchmark protocol reports."""
    cfg, master, model, pos0, first = setup_model(wl, mk)
    k = steps
    if pos0 + k > cfg.max_ctx:
        raise SystemExit(f"{wl.name}: {k} steps from position {pos0} exceed max_ctx {cfg.max_ctx}")
    sampler = ClockSampler(torch.cuda.current_device())
    with sampler:
        total_ms, per, toks = time_steps(model, first, pos0, k, warmup, dist)
        rates = []
        for _ in range(runs):
            t_ms, _, _ = time_steps(model, first, pos0, k, 0)
            rates.append(k / (t_ms * 1e-3))
    e2e_ms = time_e2e(model, first, pos0, e2e_steps or k)
    wbytes = weight_bytes(cfg, wl.variant)
    mean_pos = pos0 + (k - 1) / 2
    launch_ms = float(np.mean(per))
    res = {"tok_s": k / (total_ms * 1e-3), "ms_per_step": total_ms / k, "launch_ms": launch_ms,
           "weight_bytes": wbytes, "kv_bytes": kv_bytes(cfg, int(round(mean_pos))),
           "e2e_tok_s": (e2e_steps or k) / (e2e_ms * 1e-3), "clocks": sampler.summary(),
           "watts": sampler.watts(), "first_tokens": toks[:4].tolist(),
           "runs": {"n": runs, "steps_each": k, "median_tok_s": round(statistics.median(rates), 1),
                    "min_tok_s": round(min(rates), 1), "max_tok_s": round(max(rates), 1)} if runs else None}
    res["weight_gbs"] = wbytes / (launch_ms * 1e-3) / 1e9
    res["total_gbs"] = (wbytes + res["kv_bytes"]) / (launch_ms * 1e-3) / 1e9
    model.close()
    return res, master


def run_layer1(mk, repeats: int = 21):
    """One bf16 decoder layer + the tied 151,936-row LM head, KV prefilled with 16 positions, one step
    at position 16: its 342.7 MB fit the 126 MB L2 only in part, so it is timed both after a 512 MB
    scrub of L2 before every repeat (cold) and back to back (warm). Each repeat is one launch timed
    with CUDA events; median, min and max over the repeats."""
    wl = S.WORKLOADS["layer1_bf16"]
    cfg, _, model, pos0, first = setup_model(wl, mk)
    tok = torch.tensor([first], dtype=torch.int32, device="cuda")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    scrub = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = model.stream
    out = {}
    for mode in ("cold", "warm"):
        ms = []
        for i in range(repeats + 3):
            if mode == "cold":
                scrub.fill_(i & 0xFF)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                e0.record(stream)
                model.decode_next(tok, pos0, nxt)
                e1.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                ms.append(e0.elapsed_time(e1))
        model.sync()
        med = statistics.median(ms)
        b = weight_bytes(cfg, wl.variant) + kv_bytes(cfg, pos0)
        out[mode] = {"median_ms": round(med, 5), "min_ms": round(min(ms), 5), "max_ms": round(max(ms), 5),
                     "tok_s": round(1e3 / med, 1), "gbs": round(b / (med * 1e-3) / 1e9, 1)}
    del scrub
    model.close()
    out["bytes_per_step"] = weight_bytes(cfg, wl.variant) + kv_bytes(cfg, pos0)
    out["l2"] = "cold: a 512 MB buffer written before every repeat; warm: repeats back to back"
    return out


def whole_job_rate(local_total_ms: float, steps: int, world: int, dist=None):
    """Replicas: tokens of all ranks over the slowest rank's timed region -> (tok/s, that time in ms).

    Every rank calls this (the MAX all-reduce is collective); without a process group it is the
    single-GPU rate."""
    total_ms = float(local_total_ms)
    if dist is not None:
        t = torch.tensor([total_ms], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return world * steps / (total_ms * 1e-3), total_ms


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(S.WORKLOADS))
    ap.add_argument("--impl", default="engine", choices=["engine", "reference"])
    ap.add_argument("--no-variants", action="store_true", help="skip the FP8/NVFP4/long-context lines")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-xray", action="store_true", help="skip the instrumented-build summary")
    ap.add_argument("--sweep", action="store_true", help="print the context-length sweep (FP8) alone")
    ap.add_argument("--no-sweep", action="store_true", help="leave the context-length sweep out of the line")
    ap.add_argument("--no-layer1", action="store_true", help="leave the one-layer workload out of the line")
    ap.add_argument("--no-verify", action="store_true", help="leave the batched verify step out of the line")
    ap.add_argument("--cpu-leg", action="store_true", help=argparse.SUPPRESS)  # internal: the oracle leg
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-seconds-1t", type=float, default=10.0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.cpu_leg:  # runs in a fresh process started by the GPU arm
        run_cpu_leg(S.WORKLOADS[args.workload], args.cpu_seconds, args.cpu_seconds_1t)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("gloo")
        dist = tdist
    wl = S.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return
        master = S.master_weights(wl.config(), seed=0)
        # warm-up steps replay the first timed positions, so the timed positions are the GPU arm's
        cb = oracle_sample(wl, master, steps=args.steps, warmup=args.warmup)
        line = {"metric": "batch-1 decode tok/s (Qwen3-0.6B shape)", "value": cb["value"], "unit": "tok/s",
                "impl": "reference", "device": "host cpu", "n_gpus": args.gpus, "steps": cb["steps"],
                "warmup": args.warmup, "higher_is_better": True,
                "dtype": "f64", "data": "synthetic (seeded random weights, uniform prompt ids)",
                "config": {"workload": wl.name, "description": wl.description},
                "cpu_baseline": cb, "e2e": {"value": cb["value"], "unit": "tok/s", "h2d_bytes_per_step": 0,
                                            "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    torch.cuda.set_device(local)
    from quantized_gemv_gb300 import mk
    if args.sweep:
        if rank == 0:
            print(json.dumps(run_sweep(mk)))
        return
    stream_gbs = stream_read_gbs(mk) if rank == 0 else None
    res, master = run_workload(wl, args.steps, args.warmup, mk, dist)
    value, total_ms = whole_job_rate(res["ms_per_step"] * args.steps, args.steps, world, dist)
    peak, peak_kind = measured_peaks()
    achieved = (res["weight_bytes"] + res["kv_bytes"]) / (res["launch_ms"] * 1e-3) / 1e9
    variants = {}
    if not args.no_variants and rank == 0:
        for name in ("qwen3_0.6b_fp8", "qwen3_0.6b_nvfp4", "qwen3_0.6b_nvfp4_mse", "qwen3_0.6b_nvfp4_all",
                     "qwen3_0.6b_fp8_bf16head", "qwen3_0.6b_fp8_bf16scale", "qwen3_0.6b_fp8_ctx4096"):
            if name == wl.name:
                continue
            w2 = S.WORKLOADS[name]
            r2, _ = run_workload(w2, min(args.steps, w2.steps), args.warmup, mk, None, e2e_steps=16)
            variants[name] = {"tok_s": round(r2["tok_s"], 1), "ms_per_step": round(r2["ms_per_step"], 4),
                              "runs": r2["runs"],
                              "watts": round(r2["watts"], 1) if r2["watts"] else None,
                              "weight_gbs": round(r2["weight_gbs"], 1),
                              "roofline_frac_weights": round(r2["weight_gbs"] / peak, 4),
                              "roofline_frac_weights_kv": round(r2["total_gbs"] / peak, 4),
                              "frac_of_nominal_weights_kv": round(r2["total_gbs"] / NOMINAL_HBM_GBS, 4),
                              "e2e_tok_s": round(r2["e2e_tok_s"], 1), "clocks": r2["clocks"]}
    xr = None
    if rank == 0 and not args.no_xray:
        xr = xray_summary(wl, mk, master, steps=min(args.steps, wl.steps))
        if not args.no_variants and wl.name != "qwen3_0.6b_fp8_ctx4096":
            w4 = S.WORKLOADS["qwen3_0.6b_fp8_ctx4096"]
            xr_ctx = xray_summary(w4, mk, None, steps=min(args.steps, w4.steps))
            xr = {"headline": xr, "qwen3_0.6b_fp8_ctx4096": xr_ctx}
    layer1 = run_layer1(mk) if rank == 0 and not args.no_layer1 else None
    verify = (run_verify(mk, wl.name if wl.prefill + wl.prompt_len + 8 * 19 <= 1024 else HEADLINE)
              if rank == 0 and not args.no_verify else None)
    sweep = run_sweep(mk) if rank == 0 and not args.no_sweep else None
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        del master
        cpu = cpu_leg_subprocess(wl, 12.0, 10.0)
    if rank != 0:
        return
    line = {
        "metric": "batch-1 decode tok/s (Qwen3-0.6B shape)", "value": round(value, 2), "unit": "tok/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": round(value / world / UPSTREAM_BF16_TOKS, 3) if wl.name == HEADLINE else None,
        "dtype": "f32", "weights": wl.variant,
        "data": "synthetic (seeded N(0,0.02) bf16 weights, uniform prompt ids)",
        "config": {"workload": wl.name, "description": wl.description, "model": "Qwen3-0.6B shape, random init",
                   "global_batch": world, "positions": f"{S.WORKLOADS[wl.name].prompt_len + wl.prefill}.."
                   f"{S.WORKLOADS[wl.name].prompt_len + wl.prefill + args.steps - 1}",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "no flush: every step reads >= 0.4 GB of weights, more than the 126 MB L2"},
        "weight_stream_gbs": round(res["weight_gbs"], 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profiled_traffic(wl.name),
                     "kernel": "mk::k_decode", "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": res["weight_bytes"] + res["kv_bytes"],
                     "launch_ms": round(res["launch_ms"], 5),
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "nominal_peak": NOMINAL_HBM_GBS},
        "stream_read_gbs": round(stream_gbs, 1) if stream_gbs else None,
        "cpu_baseline": cpu,
        "e2e": {"value": round(res["e2e_tok_s"], 2), "unit": "tok/s", "h2d_bytes_per_step": 4,
                "d2h_bytes_per_step": 256, "api": "mk_decode_step (token in with the launch, status+token back)"},
        "gpu_launches": args.steps,
        "clocks": res["clocks"],
        "energy": {"watts": round(res["watts"], 1) if res["watts"] else None,
                   "tok_per_joule": round(value / world / res["watts"], 2) if res["watts"] else None,
                   "source": "NVML board power, median over the timed region"},
        "runs": res["runs"],
        "xray": xr,
        "variants": variants,
        "layer1_bf16": layer1,
        "verify": verify,
        "sweep": sweep["sweep"] if sweep else None,
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
