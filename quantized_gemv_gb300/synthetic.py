"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle harness.

This module only draws random numbers and names shapes; it holds none of the decode step's
arithmetic. Weights come from torch's CPU generator so every machine draws the same bits:

  * linear weights ~ N(0, 0.02), norm weights 1 + 0.1 N(0, 1), all rounded to bf16 (RNE by torch);
  * draw order: embedding, then per layer q, k, v, o, gate, up, down, ln_in, ln_post, q_norm,
    k_norm, then the final norm (one generator seeded with `seed`);
  * prompt ids: uniform in [0, vocab) from a generator seeded with 1;
  * prefilled KV: N(0, 1) rounded to bf16 from a generator seeded with 2, keys then values,
    layout [layer][kv_head][position][head_dim].
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np
import torch

FMT_BF16, FMT_FP8_ROW, FMT_NVFP4 = 0, 1, 2
LINEARS = ("q", "k", "v", "o", "gate", "up", "down")


@dataclass(frozen=True)
class ModelConfig:
    n_layers: int = 28
    hidden: int = 1024
    n_q_heads: int = 16
    n_kv_heads: int = 8
    head_dim: int = 128
    ffn: int = 3072
    vocab: int = 151936
    max_ctx: int = 4352
    rope_theta: float = 1e6
    rms_eps: float = 1e-6

    def shapes(self):
        """(rows, cols) = (out, in) of every linear layer."""
        H, D = self.hidden, self.head_dim
        return {"q": (self.n_q_heads * D, H), "k": (self.n_kv_heads * D, H),
                "v": (self.n_kv_heads * D, H), "o": (H, self.n_q_heads * D),
                "gate": (self.ffn, H), "up": (self.ffn, H), "down": (H, self.ffn)}


QWEN3_06B = ModelConfig()


def format_map(variant: str):
    """Per-matrix storage format of a model variant: {"embed": fmt, "q": fmt, ...}."""
    if variant == "bf16":
        m = {n: FMT_BF16 for n in LINEARS}
        m["embed"] = FMT_BF16
    elif variant == "fp8":
        m = {n: FMT_FP8_ROW for n in LINEARS}
        m["embed"] = FMT_FP8_ROW
    elif variant == "fp8_bf16scale":  # FP8 everywhere, row scales rounded to bf16
        m = {n: FMT_FP8_ROW for n in LINEARS}
        m["embed"] = FMT_FP8_ROW
        m["bf16_scale"] = True
    elif variant == "fp8_bf16head":  # FP8 layers, bf16 tied embedding / LM head
        m = {n: FMT_FP8_ROW for n in LINEARS}
        m["embed"] = FMT_BF16
    elif variant in ("nvfp4", "nvfp4_mse"):  # _mse: block scales chosen by least squared error
        m = {n: FMT_NVFP4 for n in ("q", "k", "v", "o", "gate", "up")}
        m["down"] = FMT_FP8_ROW
        m["embed"] = FMT_FP8_ROW
        if variant == "nvfp4_mse":
            m["scale_search"] = True
    elif variant == "nvfp4_all":  # every linear NVFP4 (searched block scales), FP8 tied embedding / head
        m = {n: FMT_NVFP4 for n in LINEARS}
        m["embed"] = FMT_FP8_ROW
        m["scale_search"] = True
    else:
        raise ValueError(variant)
    return m


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def master_weights(cfg: ModelConfig, seed: int = 0):
    """bf16 master weights as uint16 bit arrays: {"embed", "layers": [dict], "final_norm"}."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    sh = cfg.shapes()

    def lin(rows, cols):
        return _bf16_bits(torch.randn(rows, cols, generator=g, dtype=torch.float32) * 0.02)

    def norm(n):
        return _bf16_bits(1.0 + 0.1 * torch.randn(n, generator=g, dtype=torch.float32))

    out = {"embed": lin(cfg.vocab, cfg.hidden), "layers": []}
    for _ in range(cfg.n_layers):
        L = {n: lin(*sh[n]) for n in LINEARS}
        L["ln_in"] = norm(cfg.hidden)
        L["ln_post"] = norm(cfg.hidden)
        L["q_norm"] = norm(cfg.head_dim)
        L["k_norm"] = norm(cfg.head_dim)
        out["layers"].append(L)
    out["final_norm"] = norm(cfg.hidden)
    return out


def prompt_ids(cfg: ModelConfig, n: int = 32, seed: int = 1) -> np.ndarray:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randint(0, cfg.vocab, (n,), generator=g).numpy().astype(np.int32)


def prefill_kv(cfg: ModelConfig, n_pos: int, seed: int = 2):
    """Random bf16 keys and values for positions [0, n_pos): uint16 [L][n_kv][n_pos][head_dim]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (cfg.n_layers, cfg.n_kv_heads, n_pos, cfg.head_dim)
    k = _bf16_bits(torch.randn(*shape, generator=g, dtype=torch.float32))
    v = _bf16_bits(torch.randn(*shape, generator=g, dtype=torch.float32))
    return k, v


def random_matrix(rows: int, cols: int, seed: int, std: float = 0.02) -> np.ndarray:
    """A standalone bf16 matrix ~ N(0, std^2) (uint16 bits)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return _bf16_bits(torch.randn(rows, cols, generator=g, dtype=torch.float32) * std)


def random_vector(n: int, seed: int, std: float = 1.0) -> np.ndarray:
    """A float32 vector ~ N(0, std^2)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return (torch.randn(n, generator=g, dtype=torch.float32) * std).numpy()


@dataclass(frozen=True)
class Workload:
    """A decode workload: model variant, number of layers, prompt, prefilled KV and steps."""
    name: str
    variant: str
    n_layers: int
    prompt_len: int      # prompt tokens fed one by one before the measured steps
    prefill: int         # positions of random KV written before the first step
    steps: int           # greedy steps
    description: str

    def config(self, base: ModelConfig = QWEN3_06B) -> ModelConfig:
        start = self.prefill if self.prefill else 0
        need = start + self.prompt_len + self.steps
        max_ctx = max(base.max_ctx, ((need + 63) // 64) * 64)
        return replace(base, n_layers=self.n_layers, max_ctx=max_ctx)


WORKLOADS = {
    "layer1_bf16": Workload("layer1_bf16", "bf16", 1, 0, 16, 1,
                            "one bf16 decoder layer + tied LM head, KV prefilled with 16 positions, one step at pos 16"),
    "qwen3_0.6b_bf16": Workload("qwen3_0.6b_bf16", "bf16", 28, 32, 0, 128,
                                "28-layer bf16, 32-token uniform prompt, 128 greedy steps (pos 32..159)"),
    "qwen3_0.6b_fp8": Workload("qwen3_0.6b_fp8", "fp8", 28, 32, 0, 256,
                               "28-layer FP8-E4M3 per-row incl. LM head, 32-token prompt, 256 greedy steps"),
    "qwen3_0.6b_nvfp4": Workload("qwen3_0.6b_nvfp4", "nvfp4", 28, 32, 0, 256,
                                 "NVFP4 q/k/v/o/gate/up, FP8 down + LM head, 32-token prompt, 256 greedy steps"),
    "qwen3_0.6b_nvfp4_mse": Workload("qwen3_0.6b_nvfp4_mse", "nvfp4_mse", 28, 32, 0, 256,
                                     "NVFP4 as qwen3_0.6b_nvfp4 with least-squared-error block scales, "
                                     "32-token prompt, 256 greedy steps"),
    "qwen3_0.6b_nvfp4_all": Workload("qwen3_0.6b_nvfp4_all", "nvfp4_all", 28, 32, 0, 256,
                                     "every linear NVFP4 incl. down (least-squared-error block scales), FP8 LM "
                                     "head, 32-token prompt, 256 greedy steps"),
    "qwen3_0.6b_fp8_bf16scale": Workload("qwen3_0.6b_fp8_bf16scale", "fp8_bf16scale", 28, 32, 0, 256,
                                         "28-layer FP8-E4M3 incl. LM head, bf16 row scales, 32-token prompt, "
                                         "256 greedy steps"),
    "qwen3_0.6b_fp8_bf16head": Workload("qwen3_0.6b_fp8_bf16head", "fp8_bf16head", 28, 32, 0, 256,
                                        "28-layer FP8-E4M3 per-row, bf16 tied embedding and LM head, 32-token "
                                        "prompt, 256 greedy steps"),
    "qwen3_0.6b_fp8_ctx4096": Workload("qwen3_0.6b_fp8_ctx4096", "fp8", 28, 0, 4096, 64,
                                       "FP8, KV prefilled to 4096 positions, 64 greedy steps (pos 4096..4159)"),
}
