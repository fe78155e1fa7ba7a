"""ctypes binding of liblora_mlp.so (include/lora_mlp.h).

Argument marshalling only: every function here checks the Python-side types, turns torch
tensors into device pointers and the current torch stream into a cudaStream_t, calls the C
entry point of the same name and raises ``LmError`` on a non-zero status.  All arithmetic
runs in the library's kernels.  There is no fallback: if the shared library is missing the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass
from typing import Optional

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "liblora_mlp.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "lora_mlp.h")

LM_OK, LM_ERR_NULL, LM_ERR_SHAPE, LM_ERR_ALIGN, LM_ERR_DTYPE, LM_ERR_ALIAS = 0, 1, 2, 3, 4, 5
LM_ERR_WORKSPACE, LM_ERR_CUDA, LM_ERR_TIMEOUT, LM_ERR_UNSUPPORTED = 6, 7, 8, 9
STATUS_NAMES = {0: "LM_OK", 1: "LM_ERR_NULL", 2: "LM_ERR_SHAPE", 3: "LM_ERR_ALIGN", 4: "LM_ERR_DTYPE",
                5: "LM_ERR_ALIAS", 6: "LM_ERR_WORKSPACE", 7: "LM_ERR_CUDA", 8: "LM_ERR_TIMEOUT",
                9: "LM_ERR_UNSUPPORTED"}
LM_WEIGHT_BF16, LM_WEIGHT_NF4, LM_WEIGHT_INT4, LM_WEIGHT_NVFP4 = 0, 1, 2, 3
LM_ACT_SWIGLU, LM_ACT_GEGLU_ERF = 0, 1
LM_OUT_F32, LM_OUT_BF16 = 0, 1
LM_AB_BF16, LM_AB_F32 = 0, 1
ACTS = {"swiglu": LM_ACT_SWIGLU, "geglu": LM_ACT_GEGLU_ERF}


class LmError(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        super().__init__("%s -> %s: %s" % (fn, STATUS_NAMES.get(status, status), msg))
        self.status = status


class lm_weight(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("group", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("w", ctypes.c_void_p), ("codes", ctypes.c_void_p),
                ("absmax_q", ctypes.c_void_p), ("group_scale", ctypes.c_void_p), ("scale_zero", ctypes.c_void_p),
                ("block_scale", ctypes.c_void_p), ("global_scale", ctypes.c_void_p)]


class lm_lora(ctypes.Structure):
    _fields_ = [("W", lm_weight), ("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("r", ctypes.c_int32),
                ("s", ctypes.c_float), ("ab_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t
_SZP = ctypes.POINTER(ctypes.c_size_t)
_LP = ctypes.POINTER(lm_lora)

_SIGS = {
    "lm_last_error": ([], ctypes.c_char_p),
    "lm_nf4_codebook": ([ctypes.POINTER(ctypes.c_float)], _I32),
    "lm_workspace_reset": ([_P, _P], _I32),
    "lm_workspace_check": ([_P, _P], _I32),
    "lm_profile_enable": ([_I32], _I32),
    "lm_profile_reset": ([], _I32),
    "lm_profile_summary": ([ctypes.c_char_p, _SZ], _I32),
    "lora_mlp_saved_size": ([_I64, _I32, _SZP], _I32),
    "lora_relu2_mlp_saved_size": ([_I64, _I32, _SZP], _I32),
    "lora_relu2_mlp_workspace_size": ([_I64, _I64, _I64, _I32, _SZP], _I32),
    "lora_relu2_mlp_fwd": ([_I64, _I64, _I64, _P, _LP, _LP, _P, _P, _P, _P, _SZ, _P, _SZ, _P], _I32),
    "lora_relu2_mlp_bwd": ([_I64, _I64, _I64, _P, _P, _P, _P, _P, _SZ, _LP, _LP, _P, _P, _P, _P, _P, _P, _SZ, _P],
                           _I32),
    "lora_mlp_workspace_size": ([_I64, _I64, _I64, _I32, _SZP], _I32),
    "lora_mlp_fwd": ([_I64, _I64, _I64, _I32, _P, _LP, _LP, _LP, _P, _P, _P, _P, _P, _SZ, _P, _SZ, _P], _I32),
    "lora_mlp_bwd": ([_I64, _I64, _I64, _I32, _P, _P, _P, _P, _P, _P, _SZ, _LP, _LP, _LP, _P, _P, _P, _P, _P,
                      _P, _P, _P, _SZ, _P], _I32),
    "lora_qkv_saved_size": ([_I64, _I32, _SZP], _I32),
    "lora_qkv_workspace_size": ([_I64, _I64, _I64, _I64, _I64, _I32, _SZP], _I32),
    "lora_qkv_fwd": ([_I64, _I64, _I64, _I64, _I64, _P, _LP, _LP, _LP, _P, _P, _P, _P, _SZ, _P, _SZ, _P], _I32),
    "lora_qkv_bwd": ([_I64, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P, _SZ, _LP, _LP, _LP, _P, _P, _P, _P, _P,
                      _P, _P, _P, _SZ, _P], _I32),
    "lora_o_saved_size": ([_I64, _I32, _SZP], _I32),
    "lora_o_workspace_size": ([_I64, _I64, _I64, _I32, _SZP], _I32),
    "lora_o_fwd": ([_I64, _I64, _I64, _P, _LP, _P, _P, _SZ, _P, _SZ, _P], _I32),
    "lora_o_bwd": ([_I64, _I64, _I64, _P, _P, _P, _SZ, _LP, _P, _P, _P, _P, _SZ, _P], _I32),
    "lora_o_bwd_static": ([_I64, _I64, _I64, _P, _P, _P, _SZ, _LP, _P, _P, _P, _P], _I32),
    "lm_static_scratch_check": ([_P], _I32),
    "lm_debug_inject": ([_I32, ctypes.c_uint64], _I32),
    "nf4_pack": ([_P, _I64, _P, _P, _P, _P], _I32),
    "nf4_dequant": ([_P, _P, _P, _I64, _I32, _P, _P], _I32),
    "int4_pack": ([_P, _I64, _I64, _I32, _P, _P, _P], _I32),
    "int4_dequant": ([_P, _P, _I64, _I64, _I32, _I32, _P, _P], _I32),
    "nvfp4_pack": ([_P, _I64, _I64, _P, _P, _P, _P], _I32),
    "nvfp4_dequant": ([_P, _P, _P, _I64, _I64, _I32, _P, _P], _I32),
}

_lib = None


def header_symbols() -> list:
    """Names of the entry points declared in include/lora_mlp.h."""
    with open(HEADER) as f:
        txt = f.read()
    return re.findall(r"LM_API\s+[\w\s\*]+?\b(\w+)\s*\(", txt)


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load liblora_mlp.so (built in-tree by bwd_lora_mlp_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError("liblora_mlp.so is not built (%s); run `python -m bwd_lora_mlp_gb300.build`" % p)
    lib = ctypes.CDLL(p)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def last_error() -> str:
    return load().lm_last_error().decode()


def _call(name: str, *args) -> None:
    st = getattr(load(), name)(*args)
    if st != LM_OK:
        raise LmError(st, name, last_error())


def call_status(name: str, *args) -> int:
    """Call an entry point and return its raw status (for tests of the error paths)."""
    return getattr(load(), name)(*args)


# ---------------------------------------------------------------------------------------------
# tensor marshalling


_EMPTY = {}


def _empty_ptr(device) -> int:
    """A valid device address for a zero-element tensor: torch gives those a null data pointer,
    the C ABI wants every buffer argument non-null, and a zero-byte buffer is never accessed."""
    key = device.index if device.index is not None else torch.cuda.current_device()
    if key not in _EMPTY:
        _EMPTY[key] = torch.empty(256, dtype=torch.uint8, device=device)
    return _EMPTY[key].data_ptr()


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor") -> int:
    if t is None:
        return 0
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.numel() == 0:  # (T == 0: the token-sized buffers of a call with no tokens)
        return _empty_ptr(t.device)
    return t.data_ptr()


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class NF4Weight:
    """An NF4-packed base weight (see nf4_pack)."""
    codes: torch.Tensor        # uint8, rows*cols/2
    absmax_q: torch.Tensor     # int8, rows*cols/64
    group_scale: torch.Tensor  # float32, rows*cols/16384
    rows: int
    cols: int


@dataclass
class Int4Weight:
    """A groupwise int4 base weight (see int4_pack)."""
    codes: torch.Tensor        # uint8, rows*cols/2
    scale_zero: torch.Tensor   # bfloat16, (cols/group, rows, 2): scale, zero
    rows: int
    cols: int
    group: int


@dataclass
class NVFP4Weight:
    """An NVFP4 weight-only base (see nvfp4_pack)."""
    codes: torch.Tensor         # uint8, rows*cols/2 (E2M1, element 2i in the low nibble)
    block_scale: torch.Tensor   # uint8 E4M3, (cols/64, rows, 4)
    global_scale: torch.Tensor  # float32, (1,)
    rows: int
    cols: int


_PACKED = (NF4Weight, Int4Weight, NVFP4Weight)


@dataclass
class Lora:
    """One adapted projection: W (out, in) bf16 tensor, NF4Weight, Int4Weight or NVFP4Weight, A (r, in),
    B (out, r), s.

    A and B are both bf16 or both fp32 (fp32 LoRA parameters; each call rounds them to bf16)."""
    W: object
    A: torch.Tensor
    B: torch.Tensor
    s: float

    @property
    def r(self) -> int:
        return int(self.A.shape[0])

    def c_struct(self) -> lm_lora:
        w = lm_weight()
        if isinstance(self.W, NF4Weight):
            w.kind = LM_WEIGHT_NF4
            w.rows, w.cols = self.W.rows, self.W.cols
            w.codes = _ptr(self.W.codes, torch.uint8, "codes")
            w.absmax_q = _ptr(self.W.absmax_q, torch.int8, "absmax_q")
            w.group_scale = _ptr(self.W.group_scale, torch.float32, "group_scale")
        elif isinstance(self.W, Int4Weight):
            w.kind = LM_WEIGHT_INT4
            w.rows, w.cols, w.group = self.W.rows, self.W.cols, self.W.group
            w.codes = _ptr(self.W.codes, torch.uint8, "codes")
            w.scale_zero = _ptr(self.W.scale_zero, torch.bfloat16, "scale_zero")
        elif isinstance(self.W, NVFP4Weight):
            w.kind = LM_WEIGHT_NVFP4
            w.rows, w.cols = self.W.rows, self.W.cols
            w.codes = _ptr(self.W.codes, torch.uint8, "codes")
            w.block_scale = _ptr(self.W.block_scale, torch.uint8, "block_scale")
            w.global_scale = _ptr(self.W.global_scale, torch.float32, "global_scale")
        else:
            w.kind = LM_WEIGHT_BF16
            w.rows, w.cols = int(self.W.shape[0]), int(self.W.shape[1])
            w.w = _ptr(self.W, torch.bfloat16, "W")
        L = lm_lora()
        L.W = w
        if self.A.dtype == torch.float32 and self.B.dtype == torch.float32:
            L.ab_dtype = LM_AB_F32
            L.A = _ptr(self.A, torch.float32, "A")
            L.B = _ptr(self.B, torch.float32, "B")
        else:
            L.ab_dtype = LM_AB_BF16
            L.A = _ptr(self.A, torch.bfloat16, "A")
            L.B = _ptr(self.B, torch.bfloat16, "B")
        L.r = self.r
        L.s = float(self.s)
        return L


def _size(fn: str, *args) -> int:
    out = ctypes.c_size_t(0)
    _call(fn, *args, ctypes.byref(out))
    return out.value


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-initialised device workspace (the zeroed head is the kernels' error word)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


# ---------------------------------------------------------------------------------------------
# entry points (same names as the C ABI)


def lm_nf4_codebook() -> list:
    arr = (ctypes.c_float * 16)()
    _call("lm_nf4_codebook", arr)
    return list(arr)


def lm_workspace_check(ws: torch.Tensor, stream=None) -> None:
    _call("lm_workspace_check", _ptr(ws, torch.uint8, "ws"), _stream(stream))


def lm_profile_enable(on: bool = True) -> None:
    _call("lm_profile_enable", 1 if on else 0)


def lm_profile_reset() -> None:
    _call("lm_profile_reset")


def lm_profile_summary() -> dict:
    """{tag: (launches, total_ms)} of the kernels launched while tracing was on."""
    buf = ctypes.create_string_buffer(1 << 16)
    _call("lm_profile_summary", buf, len(buf))
    out = {}
    for line in buf.value.decode().splitlines():
        tag, n, ms = line.split("\t")
        out[tag] = (int(n), float(ms))
    return out


def lora_mlp_saved_size(T: int, r: int) -> int:
    return _size("lora_mlp_saved_size", T, r)


def lora_mlp_workspace_size(T: int, d: int, n: int, r: int) -> int:
    return _size("lora_mlp_workspace_size", T, d, n, r)


def lora_mlp_fwd(X, gate: Lora, up: Lora, down: Lora, act="swiglu", y=None, e=None, u=None, h=None,
                 saved=None, ws=None, stream=None) -> dict:
    T, d = X.shape
    n = gate.W.rows if isinstance(gate.W, _PACKED) else gate.W.shape[0]
    r = gate.r
    dev = X.device
    bf = torch.bfloat16
    y = torch.empty((T, d), dtype=bf, device=dev) if y is None else y
    e = torch.empty((T, n), dtype=bf, device=dev) if e is None else e
    u = torch.empty((T, n), dtype=bf, device=dev) if u is None else u
    h = torch.empty((T, n), dtype=bf, device=dev) if h is None else h
    saved = torch.empty(lora_mlp_saved_size(T, r), dtype=torch.uint8, device=dev) if saved is None else saved
    ws = workspace(lora_mlp_workspace_size(T, d, n, r), dev) if ws is None else ws
    Lg, Lu, Ld = gate.c_struct(), up.c_struct(), down.c_struct()
    _call("lora_mlp_fwd", T, d, n, ACTS[act], _ptr(X, bf, "X"), ctypes.byref(Lg), ctypes.byref(Lu),
          ctypes.byref(Ld), _ptr(y, bf, "y"), _ptr(e, bf, "e"), _ptr(u, bf, "u"), _ptr(h, bf, "h"),
          _ptr(saved, torch.uint8, "saved"), saved.numel(), _ptr(ws, torch.uint8, "ws"), ws.numel(),
          _stream(stream))
    return {"y": y, "e": e, "u": u, "h": h, "saved": saved, "ws": ws}


def lora_mlp_bwd(X, dY, fwd: dict, gate: Lora, up: Lora, down: Lora, act="swiglu", dX=None, grads=None,
                 ws=None, stream=None) -> dict:
    T, d = X.shape
    n = fwd["e"].shape[1]
    r = gate.r
    dev = X.device
    bf, f32 = torch.bfloat16, torch.float32
    dX = torch.empty((T, d), dtype=bf, device=dev) if dX is None else dX
    if grads is None:
        grads = {"dA_gate": torch.empty((r, d), dtype=f32, device=dev),
                 "dB_gate": torch.empty((n, r), dtype=f32, device=dev),
                 "dA_up": torch.empty((r, d), dtype=f32, device=dev),
                 "dB_up": torch.empty((n, r), dtype=f32, device=dev),
                 "dA_down": torch.empty((r, n), dtype=f32, device=dev),
                 "dB_down": torch.empty((d, r), dtype=f32, device=dev)}
    ws = fwd["ws"] if ws is None else ws
    saved = fwd["saved"]
    Lg, Lu, Ld = gate.c_struct(), up.c_struct(), down.c_struct()
    g = grads
    _call("lora_mlp_bwd", T, d, n, ACTS[act], _ptr(X, bf, "X"), _ptr(dY, bf, "dY"), _ptr(fwd["e"], bf, "e"),
          _ptr(fwd["u"], bf, "u"), _ptr(fwd["h"], bf, "h"), _ptr(saved, torch.uint8, "saved"), saved.numel(),
          ctypes.byref(Lg), ctypes.byref(Lu), ctypes.byref(Ld), _ptr(dX, bf, "dX"),
          _ptr(g["dA_gate"], f32, "dA_gate"), _ptr(g["dB_gate"], f32, "dB_gate"), _ptr(g["dA_up"], f32, "dA_up"),
          _ptr(g["dB_up"], f32, "dB_up"), _ptr(g["dA_down"], f32, "dA_down"), _ptr(g["dB_down"], f32, "dB_down"),
          _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))
    return {"dX": dX, **grads}


def lora_relu2_mlp_saved_size(T: int, r: int) -> int:
    return _size("lora_relu2_mlp_saved_size", T, r)


def lora_relu2_mlp_workspace_size(T: int, d: int, n: int, r: int) -> int:
    return _size("lora_relu2_mlp_workspace_size", T, d, n, r)


def lora_relu2_mlp_fwd(X, up: Lora, down: Lora, y=None, u=None, h=None, saved=None, ws=None, stream=None) -> dict:
    T, d = X.shape
    n = up.W.rows if isinstance(up.W, _PACKED) else up.W.shape[0]
    r = up.r
    dev = X.device
    bf = torch.bfloat16
    y = torch.empty((T, d), dtype=bf, device=dev) if y is None else y
    u = torch.empty((T, n), dtype=bf, device=dev) if u is None else u
    h = torch.empty((T, n), dtype=bf, device=dev) if h is None else h
    saved = torch.empty(lora_relu2_mlp_saved_size(T, r), dtype=torch.uint8, device=dev) if saved is None else saved
    ws = workspace(lora_relu2_mlp_workspace_size(T, d, n, r), dev) if ws is None else ws
    Lu, Ld = up.c_struct(), down.c_struct()
    _call("lora_relu2_mlp_fwd", T, d, n, _ptr(X, bf, "X"), ctypes.byref(Lu), ctypes.byref(Ld), _ptr(y, bf, "y"),
          _ptr(u, bf, "u"), _ptr(h, bf, "h"), _ptr(saved, torch.uint8, "saved"), saved.numel(),
          _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))
    return {"y": y, "u": u, "h": h, "saved": saved, "ws": ws}


def lora_relu2_mlp_bwd(X, dY, fwd: dict, up: Lora, down: Lora, dX=None, grads=None, ws=None, stream=None) -> dict:
    T, d = X.shape
    n = fwd["u"].shape[1]
    r = up.r
    dev = X.device
    bf, f32 = torch.bfloat16, torch.float32
    dX = torch.empty((T, d), dtype=bf, device=dev) if dX is None else dX
    if grads is None:
        grads = {"dA_up": torch.empty((r, d), dtype=f32, device=dev),
                 "dB_up": torch.empty((n, r), dtype=f32, device=dev),
                 "dA_down": torch.empty((r, n), dtype=f32, device=dev),
                 "dB_down": torch.empty((d, r), dtype=f32, device=dev)}
    ws = fwd["ws"] if ws is None else ws
    saved = fwd["saved"]
    Lu, Ld = up.c_struct(), down.c_struct()
    g = grads
    _call("lora_relu2_mlp_bwd", T, d, n, _ptr(X, bf, "X"), _ptr(dY, bf, "dY"), _ptr(fwd["u"], bf, "u"),
          _ptr(fwd["h"], bf, "h"), _ptr(saved, torch.uint8, "saved"), saved.numel(), ctypes.byref(Lu),
          ctypes.byref(Ld), _ptr(dX, bf, "dX"), _ptr(g["dA_up"], f32, "dA_up"), _ptr(g["dB_up"], f32, "dB_up"),
          _ptr(g["dA_down"], f32, "dA_down"), _ptr(g["dB_down"], f32, "dB_down"), _ptr(ws, torch.uint8, "ws"),
          ws.numel(), _stream(stream))
    return {"dX": dX, **grads}


def lora_qkv_saved_size(T: int, r: int) -> int:
    return _size("lora_qkv_saved_size", T, r)


def lora_qkv_workspace_size(T, d, nq, nk, nv, r) -> int:
    return _size("lora_qkv_workspace_size", T, d, nq, nk, nv, r)


def _rows(L: Lora) -> int:
    return L.W.rows if isinstance(L.W, _PACKED) else int(L.W.shape[0])


def lora_qkv_fwd(X, q: Lora, k: Lora, v: Lora, out=None, saved=None, ws=None, stream=None) -> dict:
    T, d = X.shape
    nq, nk, nv = _rows(q), _rows(k), _rows(v)
    dev, bf = X.device, torch.bfloat16
    out = out or {"Q": torch.empty((T, nq), dtype=bf, device=dev), "K": torch.empty((T, nk), dtype=bf, device=dev),
                  "V": torch.empty((T, nv), dtype=bf, device=dev)}
    saved = torch.empty(lora_qkv_saved_size(T, q.r), dtype=torch.uint8, device=dev) if saved is None else saved
    ws = workspace(lora_qkv_workspace_size(T, d, nq, nk, nv, q.r), dev) if ws is None else ws
    Ls = [L.c_struct() for L in (q, k, v)]
    _call("lora_qkv_fwd", T, d, nq, nk, nv, _ptr(X, bf, "X"), *[ctypes.byref(L) for L in Ls],
          _ptr(out["Q"], bf, "Q"), _ptr(out["K"], bf, "K"), _ptr(out["V"], bf, "V"),
          _ptr(saved, torch.uint8, "saved"), saved.numel(), _ptr(ws, torch.uint8, "ws"), ws.numel(),
          _stream(stream))
    return {**out, "saved": saved, "ws": ws}


def lora_qkv_bwd(X, dQ, dK, dV, fwd: dict, q: Lora, k: Lora, v: Lora, dX=None, grads=None, ws=None,
                 stream=None) -> dict:
    T, d = X.shape
    nq, nk, nv = _rows(q), _rows(k), _rows(v)
    r = q.r
    dev, bf, f32 = X.device, torch.bfloat16, torch.float32
    dX = torch.empty((T, d), dtype=bf, device=dev) if dX is None else dX
    if grads is None:
        grads = {"dA_q": torch.empty((r, d), dtype=f32, device=dev), "dB_q": torch.empty((nq, r), dtype=f32, device=dev),
                 "dA_k": torch.empty((r, d), dtype=f32, device=dev), "dB_k": torch.empty((nk, r), dtype=f32, device=dev),
                 "dA_v": torch.empty((r, d), dtype=f32, device=dev), "dB_v": torch.empty((nv, r), dtype=f32, device=dev)}
    ws = fwd["ws"] if ws is None else ws
    saved = fwd["saved"]
    Ls = [L.c_struct() for L in (q, k, v)]
    g = grads
    _call("lora_qkv_bwd", T, d, nq, nk, nv, _ptr(X, bf, "X"), _ptr(dQ, bf, "dQ"), _ptr(dK, bf, "dK"),
          _ptr(dV, bf, "dV"), _ptr(saved, torch.uint8, "saved"), saved.numel(), *[ctypes.byref(L) for L in Ls],
          _ptr(dX, bf, "dX"), _ptr(g["dA_q"], f32), _ptr(g["dB_q"], f32), _ptr(g["dA_k"], f32),
          _ptr(g["dB_k"], f32), _ptr(g["dA_v"], f32), _ptr(g["dB_v"], f32), _ptr(ws, torch.uint8, "ws"),
          ws.numel(), _stream(stream))
    return {"dX": dX, **grads}


def lora_o_saved_size(T: int, r: int) -> int:
    return _size("lora_o_saved_size", T, r)


def lora_o_workspace_size(T, d_in, d_out, r) -> int:
    return _size("lora_o_workspace_size", T, d_in, d_out, r)


def lora_o_fwd(X, o: Lora, Y=None, saved=None, ws=None, stream=None) -> dict:
    T, d_in = X.shape
    d_out = _rows(o)
    dev, bf = X.device, torch.bfloat16
    Y = torch.empty((T, d_out), dtype=bf, device=dev) if Y is None else Y
    saved = torch.empty(lora_o_saved_size(T, o.r), dtype=torch.uint8, device=dev) if saved is None else saved
    ws = workspace(lora_o_workspace_size(T, d_in, d_out, o.r), dev) if ws is None else ws
    L = o.c_struct()
    _call("lora_o_fwd", T, d_in, d_out, _ptr(X, bf, "X"), ctypes.byref(L), _ptr(Y, bf, "Y"),
          _ptr(saved, torch.uint8, "saved"), saved.numel(), _ptr(ws, torch.uint8, "ws"), ws.numel(),
          _stream(stream))
    return {"Y": Y, "saved": saved, "ws": ws}


def lora_o_bwd(X, dY, fwd: dict, o: Lora, dX=None, dA=None, dB=None, ws=None, stream=None) -> dict:
    T, d_in = X.shape
    d_out = _rows(o)
    r = o.r
    dev, bf, f32 = X.device, torch.bfloat16, torch.float32
    dX = torch.empty((T, d_in), dtype=bf, device=dev) if dX is None else dX
    dA = torch.empty((r, d_in), dtype=f32, device=dev) if dA is None else dA
    dB = torch.empty((d_out, r), dtype=f32, device=dev) if dB is None else dB
    ws = fwd["ws"] if ws is None else ws
    saved = fwd["saved"]
    L = o.c_struct()
    _call("lora_o_bwd", T, d_in, d_out, _ptr(X, bf, "X"), _ptr(dY, bf, "dY"), _ptr(saved, torch.uint8, "saved"),
          saved.numel(), ctypes.byref(L), _ptr(dX, bf, "dX"), _ptr(dA, f32, "dA"), _ptr(dB, f32, "dB"),
          _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))
    return {"dX": dX, "dA": dA, "dB": dB}


def lora_o_bwd_static(X, dY, fwd: dict, o: Lora, dX=None, dA=None, dB=None, stream=None) -> dict:
    """lora_o_bwd with the library's static device scratch (no workspace argument)."""
    T, d_in = X.shape
    d_out = _rows(o)
    r = o.r
    dev, bf, f32 = X.device, torch.bfloat16, torch.float32
    dX = torch.empty((T, d_in), dtype=bf, device=dev) if dX is None else dX
    dA = torch.empty((r, d_in), dtype=f32, device=dev) if dA is None else dA
    dB = torch.empty((d_out, r), dtype=f32, device=dev) if dB is None else dB
    saved = fwd["saved"]
    L = o.c_struct()
    _call("lora_o_bwd_static", T, d_in, d_out, _ptr(X, bf, "X"), _ptr(dY, bf, "dY"),
          _ptr(saved, torch.uint8, "saved"), saved.numel(), ctypes.byref(L), _ptr(dX, bf, "dX"),
          _ptr(dA, f32, "dA"), _ptr(dB, f32, "dB"), _stream(stream))
    return {"dX": dX, "dA": dA, "dB": dB}


def nf4_pack(W: torch.Tensor, stream=None) -> NF4Weight:
    numel = W.numel()
    dev = W.device
    codes = torch.empty(numel // 2, dtype=torch.uint8, device=dev)
    absmax_q = torch.empty(numel // 64, dtype=torch.int8, device=dev)
    scale = torch.empty(numel // 16384, dtype=torch.float32, device=dev)
    _call("nf4_pack", _ptr(W, torch.bfloat16, "W"), numel, _ptr(codes, torch.uint8, "codes"),
          _ptr(absmax_q, torch.int8, "absmax_q"), _ptr(scale, torch.float32, "group_scale"), _stream(stream))
    rows, cols = (W.shape[0], W.shape[1]) if W.dim() == 2 else (1, numel)
    return NF4Weight(codes, absmax_q, scale, int(rows), int(cols))


def nf4_dequant(w: NF4Weight, out_dtype=torch.float32, out=None, stream=None) -> torch.Tensor:
    numel = w.rows * w.cols
    code = LM_OUT_F32 if out_dtype == torch.float32 else LM_OUT_BF16
    out = torch.empty(numel, dtype=out_dtype, device=w.codes.device) if out is None else out
    _call("nf4_dequant", _ptr(w.codes, torch.uint8, "codes"), _ptr(w.absmax_q, torch.int8, "absmax_q"),
          _ptr(w.group_scale, torch.float32, "group_scale"), numel, code, _ptr(out, out_dtype, "out"),
          _stream(stream))
    return out


def int4_pack(W: torch.Tensor, group: int = 128, stream=None) -> Int4Weight:
    rows, cols = int(W.shape[0]), int(W.shape[1])
    dev = W.device
    codes = torch.empty(rows * cols // 2, dtype=torch.uint8, device=dev)
    sz = torch.empty((cols // group if group > 0 else 0, rows, 2), dtype=torch.bfloat16, device=dev)
    _call("int4_pack", _ptr(W, torch.bfloat16, "W"), rows, cols, int(group), _ptr(codes, torch.uint8, "codes"),
          _ptr(sz, torch.bfloat16, "scale_zero"), _stream(stream))
    return Int4Weight(codes, sz, rows, cols, int(group))


def int4_dequant(w: Int4Weight, out_dtype=torch.float32, out=None, stream=None) -> torch.Tensor:
    code = LM_OUT_F32 if out_dtype == torch.float32 else LM_OUT_BF16
    out = torch.empty((w.rows, w.cols), dtype=out_dtype, device=w.codes.device) if out is None else out
    _call("int4_dequant", _ptr(w.codes, torch.uint8, "codes"), _ptr(w.scale_zero, torch.bfloat16, "scale_zero"),
          w.rows, w.cols, w.group, code, _ptr(out, out_dtype, "out"), _stream(stream))
    return out


def nvfp4_pack(W: torch.Tensor, stream=None) -> NVFP4Weight:
    rows, cols = int(W.shape[0]), int(W.shape[1])
    dev = W.device
    codes = torch.empty(rows * cols // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty((cols // 64, rows, 4), dtype=torch.uint8, device=dev)
    gs = torch.empty(1, dtype=torch.float32, device=dev)
    _call("nvfp4_pack", _ptr(W, torch.bfloat16, "W"), rows, cols, _ptr(codes, torch.uint8, "codes"),
          _ptr(sf, torch.uint8, "block_scale"), _ptr(gs, torch.float32, "global_scale"), _stream(stream))
    return NVFP4Weight(codes, sf, gs, rows, cols)


def nvfp4_dequant(w: NVFP4Weight, out_dtype=torch.float32, out=None, stream=None) -> torch.Tensor:
    code = LM_OUT_F32 if out_dtype == torch.float32 else LM_OUT_BF16
    out = torch.empty((w.rows, w.cols), dtype=out_dtype, device=w.codes.device) if out is None else out
    _call("nvfp4_dequant", _ptr(w.codes, torch.uint8, "codes"), _ptr(w.block_scale, torch.uint8, "block_scale"),
          _ptr(w.global_scale, torch.float32, "global_scale"), w.rows, w.cols, code, _ptr(out, out_dtype, "out"),
          _stream(stream))
    return out
