"""ctypes harness around liboracle.so -- test infrastructure only.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg use this module. It
marshals numpy arrays into the oracle's C entry points; all arithmetic lives in oracle.cpp.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

FMT_BF16, FMT_FP8_ROW, FMT_NVFP4 = 0, 1, 2

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        L.or_e4m3_value.restype = C.c_double
        L.or_e4m3_value.argtypes = [C.c_int]
        L.or_e4m3_encode.restype = C.c_int
        L.or_e4m3_encode.argtypes = [C.c_double]
        L.or_e2m1_value.restype = C.c_double
        L.or_e2m1_value.argtypes = [C.c_int]
        L.or_e2m1_encode.restype = C.c_int
        L.or_e2m1_encode.argtypes = [C.c_double]
        L.or_bf16_value.restype = C.c_double
        L.or_bf16_value.argtypes = [C.c_int]
        L.or_bf16_encode.restype = C.c_int
        L.or_bf16_encode.argtypes = [C.c_double]
        L.or_silu.restype = C.c_double
        L.or_silu.argtypes = [C.c_double]
        L.or_model_create.restype = C.c_void_p
        L.or_model_destroy.argtypes = [C.c_void_p]
        L.or_model_set_kv.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int]
        L.or_model_get_kv.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int]
        L.or_model_step.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p]
        L.or_model_step.restype = C.c_int
        L.or_rmsnorm.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_double, C.c_void_p]
        L.or_rope.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_double]
        L.or_argmax.argtypes = [C.c_void_p, C.c_int]
        L.or_argmax.restype = C.c_int
        _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(C.c_void_p) if a is not None else None


# ------------------------------------------------------------------ codecs
def e4m3_value(code: int) -> float:
    return lib().or_e4m3_value(int(code))


def e4m3_encode(v: float) -> int:
    return lib().or_e4m3_encode(float(v))


def e2m1_value(code: int) -> float:
    return lib().or_e2m1_value(int(code))


def e2m1_encode(v: float) -> int:
    return lib().or_e2m1_encode(float(v))


def bf16_value(bits: int) -> float:
    return lib().or_bf16_value(int(bits))


def bf16_encode(v: float) -> int:
    return lib().or_bf16_encode(float(v))


def silu(z: float) -> float:
    return lib().or_silu(float(z))


# ------------------------------------------------------------------ matrices
class OrMat(C.Structure):
    _fields_ = [("data", C.c_void_p), ("scale", C.c_void_p), ("tensor_scale", C.c_float),
                ("fmt", C.c_int)]


class PackedMat:
    """Canonical packed matrix held in host numpy arrays (keeps the arrays alive)."""

    def __init__(self, fmt, rows, cols, data, scale=None, tensor_scale=0.0):
        self.fmt, self.rows, self.cols = fmt, rows, cols
        self.data = np.ascontiguousarray(data)
        self.scale = None if scale is None else np.ascontiguousarray(scale)
        self.tensor_scale = float(tensor_scale)

    def c(self) -> OrMat:
        return OrMat(self.data.ctypes.data, None if self.scale is None else self.scale.ctypes.data,
                     self.tensor_scale, self.fmt)


def _nt(n):
    return len(os.sched_getaffinity(0)) if n is None else int(n)


def quant_fp8_row(w_bf16: np.ndarray, nthreads=None, bf16_scale=False):
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    rows, cols = w.shape
    codes = np.zeros((rows, cols), np.uint8)
    scales = np.zeros(rows, np.float32)
    fn = lib().or_quant_fp8_row_bf16scale if bf16_scale else lib().or_quant_fp8_row
    fn(_p(w), rows, cols, _p(codes), _p(scales), _nt(nthreads))
    return codes, scales


def quant_nvfp4(w_bf16: np.ndarray, nthreads=None, scale_search=False):
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    rows, cols = w.shape
    assert cols % 16 == 0
    codes = np.zeros((rows, cols // 2), np.uint8)
    bscales = np.zeros((rows, cols // 16), np.uint8)
    t = np.zeros(1, np.float32)
    fn = lib().or_quant_nvfp4_mse if scale_search else lib().or_quant_nvfp4
    fn(_p(w), rows, cols, _p(codes), _p(bscales), _p(t), _nt(nthreads))
    return codes, bscales, float(t[0])


def pack(w_bf16: np.ndarray, fmt: int) -> PackedMat:
    """Quantise a bf16 master matrix (uint16 bits) into the canonical packed form."""
    rows, cols = w_bf16.shape
    if fmt == FMT_BF16:
        return PackedMat(fmt, rows, cols, np.ascontiguousarray(w_bf16, dtype=np.uint16))
    if fmt == FMT_FP8_ROW:
        c, s = quant_fp8_row(w_bf16)
        return PackedMat(fmt, rows, cols, c, s)
    c, b, t = quant_nvfp4(w_bf16)
    return PackedMat(fmt, rows, cols, c, b, t)


def pack_model(master, fmap, nthreads=None):
    """Quantise every matrix of a bf16 master-weight dict with the oracle's own quantisers.
    master: {"embed", "layers": [{"q".."down", "ln_in", "ln_post", "q_norm", "k_norm"}], "final_norm"}
    fmap: {"embed": fmt, "q": fmt, ...}; fmap["scale_search"] (optional) selects the NVFP4
    block-scale search, fmap["bf16_scale"] (optional) bf16 FP8 row scales."""
    search = bool(fmap.get("scale_search", False))
    bf16s = bool(fmap.get("bf16_scale", False))

    def pk(w, fmt):
        if fmt == FMT_BF16:
            return PackedMat(fmt, w.shape[0], w.shape[1], w)
        if fmt == FMT_FP8_ROW:
            c, s = quant_fp8_row(w, nthreads, bf16s)
            return PackedMat(fmt, w.shape[0], w.shape[1], c, s)
        c, b, t = quant_nvfp4(w, nthreads, search)
        return PackedMat(fmt, w.shape[0], w.shape[1], c, b, t)

    out = {"embed": pk(master["embed"], fmap["embed"]), "final_norm": master["final_norm"], "layers": []}
    for L in master["layers"]:
        d = {n: pk(L[n], fmap[n]) for n in LINEARS}
        for n in ("ln_in", "ln_post", "q_norm", "k_norm"):
            d[n] = L[n]
        out["layers"].append(d)
    return out


def dequant(m: PackedMat) -> np.ndarray:
    out = np.zeros((m.rows, m.cols), np.float64)
    mc = m.c()
    lib().or_dequant(C.byref(mc), m.rows, m.cols, _p(out))
    return out


def gemv(m: PackedMat, x: np.ndarray, nthreads: int = 1) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    assert x.shape == (m.cols,)
    y = np.zeros(m.rows, np.float64)
    mc = m.c()
    lib().or_gemv(C.byref(mc), m.rows, m.cols, _p(x), _p(y), int(nthreads))
    return y


def rmsnorm(x: np.ndarray, w_bf16: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    out = np.zeros_like(x)
    lib().or_rmsnorm(_p(x), _p(w), x.size, float(eps), _p(out))
    return out


def attend(q: np.ndarray, K_bf16: np.ndarray, V_bf16: np.ndarray) -> np.ndarray:
    """Single-query attention over n bf16 rows; K, V: uint16 [n][d]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K_bf16, dtype=np.uint16)
    V = np.ascontiguousarray(V_bf16, dtype=np.uint16)
    n, d = K.shape
    out = np.zeros(d, np.float64)
    lib().or_attend(_p(q), _p(K), _p(V), n, d, _p(out))
    return out


def argmax(x: np.ndarray) -> int:
    x = np.ascontiguousarray(x, dtype=np.float64)
    return int(lib().or_argmax(_p(x), x.size))


def rope(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    y = np.array(x, dtype=np.float64, copy=True)
    lib().or_rope(_p(y), y.size, int(pos), float(theta))
    return y


# ------------------------------------------------------------------ the decoder
class OrLayer(C.Structure):
    _fields_ = [("q", OrMat), ("k", OrMat), ("v", OrMat), ("o", OrMat), ("gate", OrMat),
                ("up", OrMat), ("down", OrMat), ("ln_in", C.c_void_p), ("ln_post", C.c_void_p),
                ("q_norm", C.c_void_p), ("k_norm", C.c_void_p)]


class OrDesc(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("hidden", C.c_int), ("n_q_heads", C.c_int),
                ("n_kv_heads", C.c_int), ("head_dim", C.c_int), ("ffn", C.c_int),
                ("vocab", C.c_int), ("max_ctx", C.c_int), ("rope_theta", C.c_double),
                ("rms_eps", C.c_double), ("layers", C.c_void_p), ("embed", OrMat),
                ("final_norm", C.c_void_p), ("n_threads", C.c_int)]


LINEARS = ("q", "k", "v", "o", "gate", "up", "down")


class OracleModel:
    """The oracle decoder over canonical packed weights.

    `packed` is a dict: {"layers": [ {name: PackedMat for LINEARS, "ln_in", "ln_post", "q_norm",
    "k_norm": uint16 arrays}, ...], "embed": PackedMat, "final_norm": uint16 array}.
    """

    def __init__(self, cfg, packed, n_threads: int | None = None):
        self.cfg = cfg
        self.packed = packed  # keep arrays alive
        if n_threads is None:
            n_threads = len(os.sched_getaffinity(0))
        self.n_threads = n_threads
        layers = (OrLayer * cfg.n_layers)()
        self._norms = []
        for i, Lp in enumerate(packed["layers"]):
            kw = {name: Lp[name].c() for name in LINEARS}
            norms = [np.ascontiguousarray(Lp[n], dtype=np.uint16) for n in ("ln_in", "ln_post", "q_norm", "k_norm")]
            self._norms.append(norms)
            layers[i] = OrLayer(**kw, ln_in=norms[0].ctypes.data, ln_post=norms[1].ctypes.data,
                                q_norm=norms[2].ctypes.data, k_norm=norms[3].ctypes.data)
        self._layers = layers
        self._final = np.ascontiguousarray(packed["final_norm"], dtype=np.uint16)
        d = OrDesc(cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn,
                   cfg.vocab, cfg.max_ctx, cfg.rope_theta, cfg.rms_eps,
                   C.cast(layers, C.c_void_p), packed["embed"].c(), self._final.ctypes.data, n_threads)
        self._desc = d
        self.h = lib().or_model_create(C.byref(d))
        if not self.h:
            raise ValueError("oracle rejected the model description")

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            lib().or_model_destroy(h)
            self.h = None

    def set_kv(self, k_bf16: np.ndarray, v_bf16: np.ndarray):
        """k, v: uint16 [n_layers][n_kv_heads][n_pos][head_dim]."""
        k = np.ascontiguousarray(k_bf16, dtype=np.uint16)
        v = np.ascontiguousarray(v_bf16, dtype=np.uint16)
        n_pos = k.shape[2]
        if lib().or_model_set_kv(self.h, _p(k), _p(v), n_pos) != 0:
            raise ValueError("bad n_pos")

    def get_kv(self, n_pos: int):
        c = self.cfg
        shape = (c.n_layers, c.n_kv_heads, n_pos, c.head_dim)
        k = np.zeros(shape, np.uint16)
        v = np.zeros(shape, np.uint16)
        if lib().or_model_get_kv(self.h, _p(k), _p(v), n_pos) != 0:
            raise ValueError("bad n_pos")
        return k, v

    def step(self, token: int, pos: int, want_logits=True, want_hidden=False):
        c = self.cfg
        logits = np.zeros(c.vocab, np.float64) if want_logits else None
        hidden = np.zeros((c.n_layers + 1, c.hidden), np.float64) if want_hidden else None
        top2 = np.zeros(2, np.float64)
        nxt = lib().or_model_step(self.h, int(token), int(pos), _p(logits), _p(hidden), _p(top2))
        if nxt < 0:
            raise ValueError("oracle rejected token/pos")
        return nxt, logits, hidden, top2
