"""Python binding of libmk.so (include/mk.h): argument marshalling only.

Every step of the decode path runs in the library's CUDA kernels; PyTorch provides device
memory and the stream. Importing this module loads (building if needed) the CUDA library and
raises if it cannot: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

from . import build as _build
from .synthetic import FMT_BF16, FMT_FP8_ROW, FMT_NVFP4, LINEARS, ModelConfig

MK_OK, MK_EINVAL, MK_ECUDA, MK_ETIMEOUT, MK_ENORESIDENT, MK_ENOTRACE, MK_EBOUNDS = 0, -1, -2, -3, -4, -5, -6
MK_FLAG_XRAY = 1
MK_FLAG_XRAY_MARKS = 4
MK_FLAG_NO_FOLD = 8
ERRNAMES = {MK_EINVAL: "MK_EINVAL", MK_ECUDA: "MK_ECUDA", MK_ETIMEOUT: "MK_ETIMEOUT",
            MK_ENORESIDENT: "MK_ENORESIDENT", MK_ENOTRACE: "MK_ENOTRACE", MK_EBOUNDS: "MK_EBOUNDS"}
TRACE_DTYPE = np.dtype([("gtime", "<u8"), ("clk", "<u8"), ("smid", "<u4"), ("cta", "<u2"),
                        ("phase", "u1"), ("kind", "u1")])
TRACE_PER_CTA = 2048  # records kept per CTA (the kernel's trace row length)
PHASES = {0: "qkv", 1: "attention", 2: "o_proj", 3: "gate_up", 4: "down", 5: "lm_head", 6: "embed"}


class MkError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{ERRNAMES.get(code, code)}: {msg}")
        self.code = code


class mk_mat(C.Structure):
    _fields_ = [("data", C.c_void_p), ("scale", C.c_void_p), ("tensor_scale", C.c_float), ("fmt", C.c_int)]


class mk_config(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("hidden", C.c_int), ("n_q_heads", C.c_int), ("n_kv_heads", C.c_int),
                ("head_dim", C.c_int), ("ffn", C.c_int), ("vocab", C.c_int), ("max_ctx", C.c_int),
                ("rope_theta", C.c_float), ("rms_eps", C.c_float)]


class mk_layer(C.Structure):
    _fields_ = [("q", mk_mat), ("k", mk_mat), ("v", mk_mat), ("o", mk_mat), ("gate", mk_mat), ("up", mk_mat),
                ("down", mk_mat), ("ln_in", C.c_void_p), ("ln_post", C.c_void_p), ("q_norm", C.c_void_p),
                ("k_norm", C.c_void_p)]


class mk_weights(C.Structure):
    _fields_ = [("layers", C.c_void_p), ("embed", mk_mat), ("final_norm", C.c_void_p)]


# every symbol include/mk.h declares
EXPORTS = ("mk_max_context", "mk_decode_grid", "mk_workspace_bytes", "mk_create", "mk_destroy", "mk_last_error", "mk_decode_step",
           "mk_decode_greedy", "mk_decode_next", "mk_sync", "mk_kv_cache", "mk_debug_hidden", "mk_trace_dump", "mk_debug_fault",
           "mk_pack_fp8_row", "mk_pack_fp8_row_bf16scale", "mk_pack_nvfp4", "mk_pack_nvfp4_mse", "mk_gemv", "mk_stream_read", "mk_probe_cvt",
           "mk_decode_step_static", "mk_debug_stress", "mk_verify_workspace_bytes", "mk_verify_attach", "mk_verify_step")
MK_VERIFY_MAX = 8

_lib = None


def lib():
    """The library, built if needed: libmk.so, or the bounds-checking libmk_debug.so when the
    environment variable MK_LIBRARY is "debug" (checked once, at the first call)."""
    global _lib
    if _lib is None:
        path = _build.build(debug=os.environ.get("MK_LIBRARY", "") == "debug")
        L = C.CDLL(path)
        vp, i32, sz = C.c_void_p, C.c_int32, C.c_size_t
        L.mk_max_context.restype = C.c_int
        L.mk_decode_grid.restype = C.c_int
        L.mk_workspace_bytes.restype = sz
        L.mk_workspace_bytes.argtypes = [C.POINTER(mk_config), C.c_uint]
        L.mk_create.argtypes = [C.POINTER(mk_config), C.POINTER(mk_weights), vp, sz, vp, C.c_uint, C.POINTER(vp)]
        L.mk_destroy.argtypes = [vp]
        L.mk_last_error.restype = C.c_char_p
        L.mk_last_error.argtypes = [vp]
        L.mk_decode_step.argtypes = [vp, i32, i32, C.POINTER(i32), vp]
        L.mk_decode_greedy.argtypes = [vp, i32, i32, i32, vp]
        L.mk_decode_next.argtypes = [vp, vp, i32, vp, vp]
        L.mk_sync.argtypes = [vp]
        L.mk_kv_cache.argtypes = [vp, C.c_int, C.POINTER(vp), C.POINTER(vp)]
        L.mk_debug_hidden.argtypes = [vp, vp]
        L.mk_trace_dump.argtypes = [vp, vp, sz, C.POINTER(sz)]
        L.mk_debug_fault.argtypes = [vp, C.c_int, C.c_int, C.c_int]
        L.mk_debug_stress.argtypes = [vp, C.c_uint32]
        L.mk_pack_fp8_row.argtypes = [vp, C.c_int, C.c_int, vp, vp, vp]
        L.mk_pack_fp8_row_bf16scale.argtypes = [vp, C.c_int, C.c_int, vp, vp, vp]
        L.mk_pack_nvfp4.argtypes = [vp, C.c_int, C.c_int, vp, vp, vp, vp]
        L.mk_pack_nvfp4_mse.argtypes = [vp, C.c_int, C.c_int, vp, vp, vp, vp]
        L.mk_gemv.argtypes = [C.POINTER(mk_mat), C.c_int, C.c_int, vp, vp, vp]
        L.mk_stream_read.argtypes = [vp, sz, vp]
        L.mk_probe_cvt.argtypes = [vp, vp, vp, C.c_int, vp, vp, vp]
        L.mk_verify_workspace_bytes.restype = sz
        L.mk_verify_workspace_bytes.argtypes = [vp]
        L.mk_verify_attach.argtypes = [vp, vp, sz]
        L.mk_verify_step.argtypes = [vp, vp, i32, i32, vp, vp]
        L.mk_decode_step_static.argtypes = [C.POINTER(mk_config), C.POINTER(mk_weights), vp, vp, i32, i32,
                                            C.POINTER(i32), vp, vp]
        _lib = L
    return _lib


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _check(rc, handle=None, what=""):
    if rc != MK_OK:
        raise MkError(rc, f"{what} {lib().mk_last_error(handle).decode()}".strip())


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("expected a CUDA tensor")


# ------------------------------------------------------------------ building blocks
class PackedMat:
    """A packed weight matrix in device memory (keeps its tensors alive)."""

    def __init__(self, fmt, rows, cols, data, scale=None, tensor_scale=0.0):
        self.fmt, self.rows, self.cols = fmt, rows, cols
        self.data, self.scale, self.tensor_scale = data, scale, float(tensor_scale)

    def c(self) -> mk_mat:
        return mk_mat(self.data.data_ptr(), None if self.scale is None else self.scale.data_ptr(),
                      self.tensor_scale, self.fmt)


def pack_fp8_row(w_bf16: torch.Tensor, stream=None, bf16_scale=False):
    """FP8-E4M3 codes and fp32 row scales; bf16_scale rounds each scale to bf16 first
    (mk_pack_fp8_row_bf16scale)."""
    _need_cuda(w_bf16)
    rows, cols = w_bf16.shape
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=w_bf16.device)
    scales = torch.empty(rows, dtype=torch.float32, device=w_bf16.device)
    fn, name = (lib().mk_pack_fp8_row_bf16scale, "mk_pack_fp8_row_bf16scale") if bf16_scale else \
        (lib().mk_pack_fp8_row, "mk_pack_fp8_row")
    _check(fn(_ptr(w_bf16.contiguous()), rows, cols, _ptr(codes), _ptr(scales), _stream(stream)), what=name)
    return codes, scales


def pack_nvfp4(w_bf16: torch.Tensor, stream=None, scale_search=False):
    """NVFP4 codes, E4M3 block scales and the fp32 tensor scale (a device scalar). With
    scale_search, each block's scale is the least-squared-error one (mk_pack_nvfp4_mse)."""
    _need_cuda(w_bf16)
    rows, cols = w_bf16.shape
    dev = w_bf16.device
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
    bscales = torch.empty((rows, cols // 16), dtype=torch.uint8, device=dev)
    t = torch.empty(1, dtype=torch.float32, device=dev)
    fn, name = (lib().mk_pack_nvfp4_mse, "mk_pack_nvfp4_mse") if scale_search else (lib().mk_pack_nvfp4,
                                                                                      "mk_pack_nvfp4")
    _check(fn(_ptr(w_bf16.contiguous()), rows, cols, _ptr(codes), _ptr(bscales), _ptr(t), _stream(stream)), what=name)
    return codes, bscales, t


def pack(w_bf16: torch.Tensor, fmt: int, stream=None, scale_search=False, bf16_scale=False) -> PackedMat:
    rows, cols = w_bf16.shape
    if fmt == FMT_BF16:
        return PackedMat(fmt, rows, cols, w_bf16.contiguous())
    if fmt == FMT_FP8_ROW:
        c, s = pack_fp8_row(w_bf16, stream, bf16_scale)
        return PackedMat(fmt, rows, cols, c, s)
    c, b, t = pack_nvfp4(w_bf16, stream, scale_search)
    torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
    return PackedMat(fmt, rows, cols, c, b, float(t.item()))


def gemv(m: PackedMat, x: torch.Tensor, stream=None) -> torch.Tensor:
    _need_cuda(x)
    y = torch.empty(m.rows, dtype=torch.float32, device=x.device)
    mc = m.c()
    _check(lib().mk_gemv(C.byref(mc), m.rows, m.cols, _ptr(x.contiguous()), _ptr(y), _stream(stream)),
           what="mk_gemv")
    return y


def stream_read(buf: torch.Tensor, nbytes: int | None = None, stream=None):
    _check(lib().mk_stream_read(_ptr(buf), buf.numel() * buf.element_size() if nbytes is None else nbytes,
                                _stream(stream)), what="mk_stream_read")


def probe_cvt(x_f32: torch.Tensor | None = None, stream=None):
    dev = torch.device("cuda")
    a = torch.empty(65536, dtype=torch.int32, device=dev)
    b = torch.empty(256, dtype=torch.int32, device=dev)
    n = 0 if x_f32 is None else x_f32.numel()
    e4 = torch.empty(max(n // 2, 1), dtype=torch.int16, device=dev)
    e2 = torch.empty(max(n // 2, 1), dtype=torch.uint8, device=dev)
    _check(lib().mk_probe_cvt(_ptr(a), _ptr(b), _ptr(x_f32), n, _ptr(e4) if n else None, _ptr(e2) if n else None,
                              _stream(stream)), what="mk_probe_cvt")
    return a, b, e4[: n // 2], e2[: n // 2]


def max_context() -> int:
    return lib().mk_max_context()


def decode_grid() -> int:
    return lib().mk_decode_grid()


# ------------------------------------------------------------------ the model
class Model:
    """A decode engine instance over packed device weights.

    `packed` = {"layers": [{name: PackedMat for LINEARS, "ln_in", "ln_post", "q_norm", "k_norm": bf16
    tensors}], "embed": PackedMat, "final_norm": bf16 tensor}, all on the current CUDA device.
    """

    def __init__(self, cfg: ModelConfig, packed, flags: int = 0, stream=None):
        self.cfg = cfg
        self.packed = packed
        self.flags = flags
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        L = lib()
        self._cfg = mk_config(cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn,
                              cfg.vocab, cfg.max_ctx, cfg.rope_theta, cfg.rms_eps)
        layers = (mk_layer * cfg.n_layers)()
        for i, Lp in enumerate(packed["layers"]):
            layers[i] = mk_layer(*(Lp[n].c() for n in LINEARS), Lp["ln_in"].data_ptr(), Lp["ln_post"].data_ptr(),
                                 Lp["q_norm"].data_ptr(), Lp["k_norm"].data_ptr())
        self._layers = layers
        self._w = mk_weights(C.cast(layers, C.c_void_p), packed["embed"].c(), packed["final_norm"].data_ptr())
        nbytes = L.mk_workspace_bytes(C.byref(self._cfg), flags)
        if nbytes == 0:
            raise MkError(MK_EINVAL, "mk_workspace_bytes rejected the config")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        h = C.c_void_p()
        rc = L.mk_create(C.byref(self._cfg), C.byref(self._w), _ptr(self.workspace), nbytes,
                         C.c_void_p(self.stream.cuda_stream), flags, C.byref(h))
        if rc != MK_OK:
            raise MkError(rc, L.mk_last_error(None).decode())
        self.h = h
        self._next = C.c_int32()

    def close(self):
        if getattr(self, "h", None):
            lib().mk_destroy(self.h)
            self.h = None

    __del__ = close

    def _err(self, rc, what):
        if rc != MK_OK:
            raise MkError(rc, f"{what}: {lib().mk_last_error(self.h).decode()}")

    def decode_step(self, token: int, pos: int, logits: torch.Tensor | None = None) -> int:
        rc = lib().mk_decode_step(self.h, int(token), int(pos), C.byref(self._next), _ptr(logits))
        self._err(rc, "mk_decode_step")
        return int(self._next.value)

    def decode_greedy(self, first_token: int, pos0: int, n: int, out: torch.Tensor | None = None) -> torch.Tensor:
        if out is None:
            out = torch.empty(n, dtype=torch.int32, device="cuda")
        self._err(lib().mk_decode_greedy(self.h, int(first_token), int(pos0), int(n), _ptr(out)), "mk_decode_greedy")
        return out

    def decode_next(self, token_dev: torch.Tensor, pos: int, next_dev: torch.Tensor, logits=None):
        """One launch; token_dev / next_dev are 1-element int32 CUDA tensors (or views)."""
        self._err(lib().mk_decode_next(self.h, _ptr(token_dev), int(pos), _ptr(next_dev), _ptr(logits)),
                  "mk_decode_next")

    def sync(self):
        self._err(lib().mk_sync(self.h), "mk_sync")

    def kv_cache(self, layer: int):
        """(K, V) bf16 views [n_kv_heads][max_ctx][head_dim] into the model's workspace."""
        k, v = C.c_void_p(), C.c_void_p()
        self._err(lib().mk_kv_cache(self.h, layer, C.byref(k), C.byref(v)), "mk_kv_cache")
        c = self.cfg
        n = c.n_kv_heads * c.max_ctx * c.head_dim
        base = self.workspace.data_ptr()
        ws = self.workspace
        kt = ws[k.value - base: k.value - base + 2 * n].view(torch.bfloat16).view(c.n_kv_heads, c.max_ctx, c.head_dim)
        vt = ws[v.value - base: v.value - base + 2 * n].view(torch.bfloat16).view(c.n_kv_heads, c.max_ctx, c.head_dim)
        return kt, vt

    def hidden(self) -> torch.Tensor:
        out = torch.empty((self.cfg.n_layers + 1, self.cfg.hidden), dtype=torch.float32, device="cuda")
        self._err(lib().mk_debug_hidden(self.h, _ptr(out)), "mk_debug_hidden")
        return out

    def trace(self) -> np.ndarray:
        cap = 0
        grid = torch.cuda.get_device_properties(0).multi_processor_count
        cap = grid * TRACE_PER_CTA * TRACE_DTYPE.itemsize
        buf = np.zeros(cap, dtype=np.uint8)
        written = C.c_size_t()
        self._err(lib().mk_trace_dump(self.h, buf.ctypes.data_as(C.c_void_p), cap, C.byref(written)), "mk_trace_dump")
        recs = buf[: written.value].view(TRACE_DTYPE)
        return recs.reshape(len(recs) // TRACE_PER_CTA, TRACE_PER_CTA)  # one row of records per CTA of the grid

    def debug_stress(self, seed: int):
        """Seeded 0..20 us per-CTA waits before every step (0 = off); results must not change."""
        self._err(lib().mk_debug_stress(self.h, int(seed)), "mk_debug_stress")

    def verify_attach(self):
        """Repack the weights for mk_verify_step into a workspace this object keeps."""
        n = lib().mk_verify_workspace_bytes(self.h)
        self.verify_workspace = torch.empty(n, dtype=torch.uint8, device="cuda")
        self._err(lib().mk_verify_attach(self.h, _ptr(self.verify_workspace), n), "mk_verify_attach")

    def verify_step(self, tokens_dev: torch.Tensor, pos0: int, next_dev: torch.Tensor, logits=None):
        """One batched verify launch over the k = len(tokens_dev) tokens (int32 CUDA tensors)."""
        self._err(lib().mk_verify_step(self.h, _ptr(tokens_dev), int(tokens_dev.numel()), int(pos0), _ptr(next_dev),
                                       _ptr(logits)), "mk_verify_step")

    def debug_fault(self, cta: int, phase: int, timeout_ms: int = 0):
        self._err(lib().mk_debug_fault(self.h, cta, phase, timeout_ms), "mk_debug_fault")


MK_STATIC_MAX_CTX = 4352


def decode_step_static(cfg: ModelConfig, packed, k_cache: torch.Tensor, v_cache: torch.Tensor, token: int,
                       pos: int, logits: torch.Tensor | None = None, stream=None) -> int:
    """mk_decode_step_static: one step with no model object and no workspace (the library keeps its
    scratch in a fixed device array). k_cache / v_cache: contiguous bf16 CUDA tensors of at least
    n_layers * n_kv_heads * max_ctx * head_dim elements (state the caller keeps between steps).
    The library cannot see the caches' size, so it is checked here before the call."""
    need = cfg.n_layers * cfg.n_kv_heads * cfg.max_ctx * cfg.head_dim
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
        if t.numel() < need:
            raise ValueError(f"{name} holds {t.numel()} elements, the model needs {need}")
    if logits is not None and not (logits.is_cuda and logits.dtype == torch.float32 and logits.is_contiguous()
                                   and logits.numel() >= cfg.vocab):
        raise ValueError("logits must be a contiguous fp32 CUDA tensor of at least vocab elements")
    ccfg = mk_config(cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn, cfg.vocab,
                     cfg.max_ctx, cfg.rope_theta, cfg.rms_eps)
    layers = (mk_layer * cfg.n_layers)()
    for i, Lp in enumerate(packed["layers"]):
        layers[i] = mk_layer(*(Lp[n].c() for n in LINEARS), Lp["ln_in"].data_ptr(), Lp["ln_post"].data_ptr(),
                             Lp["q_norm"].data_ptr(), Lp["k_norm"].data_ptr())
    w = mk_weights(C.cast(layers, C.c_void_p), packed["embed"].c(), packed["final_norm"].data_ptr())
    nxt = C.c_int32()
    rc = lib().mk_decode_step_static(C.byref(ccfg), C.byref(w), _ptr(k_cache), _ptr(v_cache), int(token), int(pos),
                                     C.byref(nxt), _ptr(logits), _stream(stream))
    if rc != MK_OK:
        raise MkError(rc, lib().mk_last_error(None).decode())
    return int(nxt.value)


def upload_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def pack_model(master, fmap, device="cuda"):
    """Upload bf16 master weights and quantise them on the device with the library's packers.
    fmap["scale_search"] (optional) selects the NVFP4 block-scale search, fmap["bf16_scale"]
    (optional) bf16 FP8 row scales."""
    search = bool(fmap.get("scale_search", False))
    bf16s = bool(fmap.get("bf16_scale", False))

    def pk(bits, fmt):
        return pack(upload_bf16(bits, device), fmt, scale_search=search, bf16_scale=bf16s)

    out = {"embed": pk(master["embed"], fmap["embed"]), "final_norm": upload_bf16(master["final_norm"], device),
           "layers": []}
    for L in master["layers"]:
        d = {n: pk(L[n], fmap[n]) for n in LINEARS}
        for n in ("ln_in", "ln_post", "q_norm", "k_norm"):
            d[n] = upload_bf16(L[n], device)
        out["layers"].append(d)
    torch.cuda.synchronize()
    return out
