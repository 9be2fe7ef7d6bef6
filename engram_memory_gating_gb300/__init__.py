"""Python binding of libengram.so (the GB300 Engram gate library).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/engram.h.  PyTorch provides
device memory and the current stream.  There is no CPU fallback: if the
library is missing or the device is not sm_103, calls raise.

Entry points (same names as the C ABI):
  engram_gate_fwd, engram_gate_bwd, engram_gate_bwd_workspace_size,
  engram_gateconv_fwd, engram_gateconv_bwd, engram_gateconv_bwd_workspace_size,
  engram_device_error, engram_launch_info.
Convenience wrappers that allocate their outputs (like the eager wrappers of
the cuDNN Frontend page): gate_forward, gate_backward, gateconv_forward,
gateconv_backward.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from ._build import LIB as _LIB_PATH
from ._build import build as _build_lib

__all__ = [
    "EngramError", "load", "build",
    "engram_gate_fwd", "engram_gate_bwd", "engram_gate_bwd_workspace_size",
    "engram_gateconv_fwd", "engram_gateconv_bwd", "engram_gateconv_bwd_workspace_size",
    "engram_device_error", "engram_launch_info", "engram_gate_bwd_noalloc",
    "engram_gate_sep_fwd", "engram_gate_sep_bwd", "engram_gate_sep_bwd_workspace_size",
    "engram_gate_bwd_fused_weight", "gate_backward_fused_weight",
    "gate_forward", "gate_backward", "gateconv_forward", "gateconv_backward",
    "gate_sep_forward", "gate_sep_backward", "engram_fused_weight", "engram_fused_weight_bwd",
    "fused_weight", "fused_weight_backward", "engram_decode_fwd", "engram_decode_workspace_size",
    "decode_forward",
    "GATE_EPS", "GATE_CLAMP", "GATECONV_EPS", "EXPORTED_SYMBOLS",
]

GATE_EPS = 1e-20     # default RMS-norm epsilon of the saved-state gate
GATE_CLAMP = 1e-6    # clamp of the gate's signed square root
GATECONV_EPS = 1e-6  # default RMSNorm epsilon of GateConv
D_GATE = 5120
S_GATE = 4

EXPORTED_SYMBOLS = (
    "engram_status_string", "engram_gate_fwd", "engram_gate_bwd_workspace_size",
    "engram_gate_bwd", "engram_gateconv_fwd", "engram_gateconv_bwd_workspace_size",
    "engram_gateconv_bwd", "engram_device_error", "engram_launch_info",
    "engram_gate_bwd_noalloc", "engram_gate_sep_fwd", "engram_gate_sep_bwd_workspace_size",
    "engram_gate_sep_bwd", "engram_fused_weight", "engram_fused_weight_bwd",
    "engram_decode_workspace_size", "engram_decode_fwd", "engram_gate_bwd_fused_weight",
)

_STATUS = {0: "ok", 1: "null pointer", 2: "misaligned pointer", 3: "size out of range",
           4: "overlap", 5: "workspace too small", 6: "no usable sm_103 device",
           7: "kernel launch failed"}


class EngramError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: status {code} ({_STATUS.get(code, 'unknown')})")
        self.code = code


class _LaunchInfo(ctypes.Structure):
    _fields_ = [("cluster", ctypes.c_int), ("threads", ctypes.c_int),
                ("clusters", ctypes.c_int), ("stages", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("resident", ctypes.c_int),
                ("kernels", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile libengram.so for sm_103a (nvcc) and return its path."""
    return _build_lib(force=force)


def load(path: str | None = None):
    """Load libengram.so (building it first if it is absent or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _LIB_PATH
        if path is None:
            _build_lib()
        if not os.path.exists(p):
            raise RuntimeError(f"libengram.so not found at {p}")
        lib = ctypes.CDLL(p)
        P, I64, F, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        lib.engram_status_string.restype = ctypes.c_char_p
        lib.engram_status_string.argtypes = [ctypes.c_int]
        lib.engram_gate_fwd.argtypes = [P, P, P, P, P, P, I64, F, P]
        lib.engram_gate_bwd_workspace_size.argtypes = [I64]
        lib.engram_gate_bwd_workspace_size.restype = SZ
        lib.engram_gate_bwd.argtypes = [P, P, P, P, P, P, P, P, P, SZ, I64, P]
        lib.engram_gate_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, I64, P]
        lib.engram_gate_bwd_fused_weight.argtypes = [P] * 13 + [SZ, I64, P]
        lib.engram_gate_sep_fwd.argtypes = [P] * 9 + [I64, I64, F, F, P]
        lib.engram_gate_sep_bwd_workspace_size.argtypes = [I64]
        lib.engram_gate_sep_bwd_workspace_size.restype = SZ
        lib.engram_gate_sep_bwd.argtypes = [P] * 14 + [SZ, I64, I64, F, P]
        lib.engram_fused_weight.argtypes = [P, P, P, I64, P]
        lib.engram_decode_workspace_size.argtypes = [I64, I64, I64]
        lib.engram_decode_workspace_size.restype = SZ
        lib.engram_decode_fwd.argtypes = [P, P, P, I64] + [P] * 8 + [SZ, I64, I64, I64, I64, I64, I64, F, P]
        lib.engram_fused_weight_bwd.argtypes = [P, I64, P, P, P, P, P, I64, P]
        lib.engram_gateconv_fwd.argtypes = [P] * 12 + [I64, I64, I64, F, P]
        lib.engram_gateconv_bwd_workspace_size.argtypes = [I64, I64, I64]
        lib.engram_gateconv_bwd_workspace_size.restype = SZ
        lib.engram_gateconv_bwd.argtypes = [P] * 19 + [SZ, I64, I64, I64, F, P]
        lib.engram_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        lib.engram_launch_info.argtypes = [ctypes.c_int, I64, I64, I64,
                                           ctypes.POINTER(_LaunchInfo)]
        for name in ("engram_gate_fwd", "engram_gate_bwd", "engram_gate_bwd_noalloc",
                     "engram_gate_bwd_fused_weight",
                     "engram_gate_sep_fwd", "engram_gate_sep_bwd", "engram_fused_weight",
                     "engram_fused_weight_bwd", "engram_decode_fwd", "engram_gateconv_fwd",
                     "engram_gateconv_bwd", "engram_device_error", "engram_launch_info"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        return ctypes.c_void_p(int(t))
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(fn, code):
    if code != 0:
        raise EngramError(fn, code)


def _need(t, dtype, shape, name):
    if t.dtype != dtype or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected {dtype} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")


# ------------------------------------------------------------ C ABI wrappers

def engram_gate_fwd(x, kv, weight, mask, out, saved, eps: float = GATE_EPS, stream=None):
    N = x.shape[0]
    _need(x, torch.bfloat16, (N, S_GATE, D_GATE), "x")
    _need(kv, torch.bfloat16, (N, (S_GATE + 1) * D_GATE), "kv")
    _need(weight, torch.float32, (S_GATE, D_GATE), "weight")
    _need(out, torch.bfloat16, (N, S_GATE, D_GATE), "out")
    if mask is not None:
        _need(mask, torch.bool, (N,), "mask")
    if saved is not None:
        _need(saved, torch.float32, (N, S_GATE, 4), "saved")
    _check("engram_gate_fwd", load().engram_gate_fwd(
        _ptr(x), _ptr(kv), _ptr(weight), _ptr(mask), _ptr(out), _ptr(saved), N,
        float(eps), _stream(stream)))


def engram_gate_bwd_workspace_size(N: int) -> int:
    return int(load().engram_gate_bwd_workspace_size(int(N)))


def engram_gate_bwd(x, kv, weight, saved, grad_out, grad_x, grad_kv, grad_weight, workspace,
                    stream=None):
    N = x.shape[0]
    _need(saved, torch.float32, (N, S_GATE, 4), "saved")
    _need(grad_out, torch.bfloat16, (N, S_GATE, D_GATE), "grad_out")
    _need(grad_x, torch.bfloat16, (N, S_GATE, D_GATE), "grad_x")
    _need(grad_kv, torch.bfloat16, (N, (S_GATE + 1) * D_GATE), "grad_kv")
    _need(grad_weight, torch.float32, (S_GATE, D_GATE), "grad_weight")
    nbytes = workspace.numel() * workspace.element_size()
    _check("engram_gate_bwd", load().engram_gate_bwd(
        _ptr(x), _ptr(kv), _ptr(weight), _ptr(saved), _ptr(grad_out), _ptr(grad_x),
        _ptr(grad_kv), _ptr(grad_weight), _ptr(workspace), nbytes, N, _stream(stream)))


def engram_gate_bwd_fused_weight(x, kv, weight, saved, grad_out, wh, we, grad_x, grad_kv,
                                 grad_weight, grad_wh, grad_we, workspace, stream=None):
    """engram_gate_bwd for weight = wh * we (bf16 (4, 5120) factors): the
    grad_weight merge also writes grad_wh = grad_weight * we and grad_we =
    grad_weight * wh.  grad_weight may be None."""
    N = x.shape[0]
    _need(saved, torch.float32, (N, S_GATE, 4), "saved")
    _need(grad_out, torch.bfloat16, (N, S_GATE, D_GATE), "grad_out")
    _need(grad_x, torch.bfloat16, (N, S_GATE, D_GATE), "grad_x")
    _need(grad_kv, torch.bfloat16, (N, (S_GATE + 1) * D_GATE), "grad_kv")
    for t, n in ((wh, "wh"), (we, "we")):
        _need(t, torch.bfloat16, (S_GATE, D_GATE), n)
    for t, n in ((grad_wh, "grad_wh"), (grad_we, "grad_we")) + (
            ((grad_weight, "grad_weight"),) if grad_weight is not None else ()):
        _need(t, torch.float32, (S_GATE, D_GATE), n)
    nbytes = workspace.numel() * workspace.element_size()
    _check("engram_gate_bwd_fused_weight", load().engram_gate_bwd_fused_weight(
        _ptr(x), _ptr(kv), _ptr(weight), _ptr(saved), _ptr(grad_out), _ptr(wh), _ptr(we),
        _ptr(grad_x), _ptr(grad_kv), _ptr(grad_weight), _ptr(grad_wh), _ptr(grad_we),
        _ptr(workspace), nbytes, N, _stream(stream)))


def engram_gate_bwd_noalloc(x, kv, weight, saved, grad_out, grad_x, grad_kv, grad_weight,
                            stream=None):
    """engram_gate_bwd without a workspace argument, for callers that cannot
    allocate: the library's own fixed device array serves as the workspace
    (N <= 2048).  Calls that can overlap on the GPU must be serialised."""
    N = x.shape[0]
    _need(saved, torch.float32, (N, S_GATE, 4), "saved")
    _need(grad_out, torch.bfloat16, (N, S_GATE, D_GATE), "grad_out")
    _need(grad_x, torch.bfloat16, (N, S_GATE, D_GATE), "grad_x")
    _need(grad_kv, torch.bfloat16, (N, (S_GATE + 1) * D_GATE), "grad_kv")
    _need(grad_weight, torch.float32, (S_GATE, D_GATE), "grad_weight")
    _check("engram_gate_bwd_noalloc", load().engram_gate_bwd_noalloc(
        _ptr(x), _ptr(kv), _ptr(weight), _ptr(saved), _ptr(grad_out), _ptr(grad_x),
        _ptr(grad_kv), _ptr(grad_weight), N, _stream(stream)))


def engram_gate_sep_fwd(x, k, v, weight, out, dot=None, gate=None, rstd_x=None, rstd_k=None,
                        eps: float = GATE_EPS, clamp: float = GATE_CLAMP, stream=None):
    """Separate key / value tensors, any hidden size H (multiple of 8); the
    saved state is four (N, 4) arrays, all given or all None."""
    N, _, H = x.shape
    _need(x, torch.bfloat16, (N, S_GATE, H), "x")
    _need(k, torch.bfloat16, (N, S_GATE, H), "k")
    _need(v, torch.bfloat16, (N, H), "v")
    _need(weight, torch.float32, (S_GATE, H), "weight")
    _need(out, torch.bfloat16, (N, S_GATE, H), "out")
    for t, n in ((dot, "dot"), (gate, "gate"), (rstd_x, "rstd_x"), (rstd_k, "rstd_k")):
        if t is not None:
            _need(t, torch.float32, (N, S_GATE), n)
    _check("engram_gate_sep_fwd", load().engram_gate_sep_fwd(
        _ptr(x), _ptr(k), _ptr(v), _ptr(weight), _ptr(out), _ptr(dot), _ptr(gate), _ptr(rstd_x),
        _ptr(rstd_k), N, H, float(eps), float(clamp), _stream(stream)))


def engram_gate_sep_bwd_workspace_size(N: int) -> int:
    return int(load().engram_gate_sep_bwd_workspace_size(int(N)))


def engram_gate_sep_bwd(grad_out, x, k, v, weight, dot, gate, rstd_x, rstd_k, grad_x, grad_k,
                        grad_v, grad_w_partial, workspace, clamp: float = GATE_CLAMP, stream=None):
    N, _, H = x.shape
    for t, n in ((grad_out, "grad_out"), (grad_x, "grad_x"), (grad_k, "grad_k")):
        _need(t, torch.bfloat16, (N, S_GATE, H), n)
    _need(grad_v, torch.bfloat16, (N, H), "grad_v")
    _need(grad_w_partial, torch.float32, ((N + 63) // 64, S_GATE, H), "grad_w_partial")
    nbytes = workspace.numel() * workspace.element_size()
    _check("engram_gate_sep_bwd", load().engram_gate_sep_bwd(
        _ptr(grad_out), _ptr(x), _ptr(k), _ptr(v), _ptr(weight), _ptr(dot), _ptr(gate),
        _ptr(rstd_x), _ptr(rstd_k), _ptr(grad_x), _ptr(grad_k), _ptr(grad_v), _ptr(grad_w_partial),
        _ptr(workspace), nbytes, N, H, float(clamp), _stream(stream)))


def engram_fused_weight(wh, we, weight, stream=None):
    n = wh.numel()
    _need(wh, torch.bfloat16, tuple(wh.shape), "wh")
    _need(we, torch.bfloat16, tuple(wh.shape), "we")
    _need(weight, torch.float32, tuple(wh.shape), "weight")
    _check("engram_fused_weight", load().engram_fused_weight(_ptr(wh), _ptr(we), _ptr(weight), n,
                                                             _stream(stream)))


def engram_fused_weight_bwd(grad_w_partial, wh, we, grad_w, grad_wh, grad_we, stream=None):
    """grad_w_partial (nblocks, *wh.shape); grad_w may be None."""
    n = wh.numel()
    nblocks = grad_w_partial.numel() // n
    _need(grad_w_partial, torch.float32, (nblocks,) + tuple(wh.shape), "grad_w_partial")
    for t, nm in ((grad_wh, "grad_wh"), (grad_we, "grad_we")) + (((grad_w, "grad_w"),) if grad_w is not None else ()):
        _need(t, torch.float32, tuple(wh.shape), nm)
    _check("engram_fused_weight_bwd", load().engram_fused_weight_bwd(
        _ptr(grad_w_partial), nblocks, _ptr(wh), _ptr(we), _ptr(grad_w), _ptr(grad_wh), _ptr(grad_we),
        n, _stream(stream)))


def engram_decode_workspace_size(B: int, d_mem: int, d: int) -> int:
    return int(load().engram_decode_workspace_size(int(B), int(d_mem), int(d)))


def engram_decode_fwd(e, h, conv_state, W_K, W_V, rms_w_h, rms_w_v, conv_w, y, new_state,
                      workspace, dilation: int, eps: float = GATECONV_EPS, stream=None):
    """conv_state (B, L, d) with L <= new_state.shape[1] (None or L = 0 for an
    empty cache)."""
    B, d_mem = e.shape
    d = h.shape[1]
    max_len = new_state.shape[1]
    w = conv_w.shape[0]
    L = 0 if conv_state is None else conv_state.shape[1]
    _need(e, torch.bfloat16, (B, d_mem), "e")
    _need(h, torch.bfloat16, (B, d), "h")
    if conv_state is not None:
        _need(conv_state, torch.bfloat16, (B, L, d), "conv_state")
    for t, n in ((W_K, "W_K"), (W_V, "W_V")):
        _need(t, torch.bfloat16, (d_mem, d), n)
    _need(rms_w_h, torch.float32, (d,), "rms_w_h")
    _need(rms_w_v, torch.float32, (d,), "rms_w_v")
    _need(conv_w, torch.float32, (w, d), "conv_w")
    _need(y, torch.bfloat16, (B, d), "y")
    _need(new_state, torch.bfloat16, (B, max_len, d), "new_state")
    st = conv_state if (conv_state is not None and L > 0) else None
    nbytes = workspace.numel() * workspace.element_size()
    _check("engram_decode_fwd", load().engram_decode_fwd(
        _ptr(e), _ptr(h), _ptr(st), L, _ptr(W_K), _ptr(W_V), _ptr(rms_w_h), _ptr(rms_w_v),
        _ptr(conv_w), _ptr(y), _ptr(new_state), _ptr(workspace), nbytes, B, d_mem, d, max_len, w,
        int(dilation), float(eps), _stream(stream)))


def engram_gateconv_fwd(H, k, v, rms_w_h, rms_w_v, conv_w, Y, vhat, alpha, rrms_h, rrms_k,
                        rrms_v, eps: float = GATECONV_EPS, stream=None):
    M, T, d = H.shape
    for t, n in ((H, "H"), (k, "k"), (v, "v"), (Y, "Y"), (vhat, "vhat")):
        _need(t, torch.bfloat16, (M, T, d), n)
    for t, n in ((alpha, "alpha"), (rrms_h, "rrms_h"), (rrms_k, "rrms_k"), (rrms_v, "rrms_v")):
        _need(t, torch.float32, (M, T), n)
    _need(rms_w_h, torch.float32, (d,), "rms_w_h")
    _need(rms_w_v, torch.float32, (d,), "rms_w_v")
    _need(conv_w, torch.float32, (4, d), "conv_w")
    _check("engram_gateconv_fwd", load().engram_gateconv_fwd(
        _ptr(H), _ptr(k), _ptr(v), _ptr(rms_w_h), _ptr(rms_w_v), _ptr(conv_w), _ptr(Y),
        _ptr(vhat), _ptr(alpha), _ptr(rrms_h), _ptr(rrms_k), _ptr(rrms_v), M, T, d,
        float(eps), _stream(stream)))


def engram_gateconv_bwd_workspace_size(M: int, T: int, d: int) -> int:
    return int(load().engram_gateconv_bwd_workspace_size(int(M), int(T), int(d)))


def engram_gateconv_bwd(dY, H, k, v, rms_w_h, rms_w_v, conv_w, vhat, alpha, rrms_h, rrms_k,
                        rrms_v, dH, dk, dv, drms_w_h, drms_w_v, dconv_w, workspace,
                        eps: float = GATECONV_EPS, stream=None):
    M, T, d = H.shape
    for t, n in ((dY, "dY"), (k, "k"), (v, "v"), (vhat, "vhat"), (dH, "dH"), (dk, "dk"),
                 (dv, "dv")):
        _need(t, torch.bfloat16, (M, T, d), n)
    _need(drms_w_h, torch.float32, (d,), "drms_w_h")
    _need(drms_w_v, torch.float32, (d,), "drms_w_v")
    _need(dconv_w, torch.float32, (4, d), "dconv_w")
    nbytes = workspace.numel() * workspace.element_size()
    _check("engram_gateconv_bwd", load().engram_gateconv_bwd(
        _ptr(dY), _ptr(H), _ptr(k), _ptr(v), _ptr(rms_w_h), _ptr(rms_w_v), _ptr(conv_w),
        _ptr(vhat), _ptr(alpha), _ptr(rrms_h), _ptr(rrms_k), _ptr(rrms_v), _ptr(dH), _ptr(dk),
        _ptr(dv), _ptr(drms_w_h), _ptr(drms_w_v), _ptr(dconv_w), _ptr(workspace), nbytes,
        M, T, d, float(eps), _stream(stream)))


def engram_device_error() -> int:
    v = ctypes.c_uint32(0)
    _check("engram_device_error", load().engram_device_error(ctypes.byref(v)))
    return int(v.value)


def engram_launch_info(op: int, n0: int, n1: int = 0, n2: int = 0) -> dict:
    info = _LaunchInfo()
    _check("engram_launch_info", load().engram_launch_info(int(op), int(n0), int(n1), int(n2),
                                                           ctypes.byref(info)))
    return {f: getattr(info, f) for f, _ in _LaunchInfo._fields_}


# ------------------------------------------------- allocating convenience API

def gate_forward(x, kv, weight, mask=None, eps: float = GATE_EPS, save: bool = True):
    out = torch.empty_like(x)
    saved = torch.empty((x.shape[0], S_GATE, 4), device=x.device, dtype=torch.float32) \
        if save else None
    engram_gate_fwd(x, kv, weight, mask, out, saved, eps)
    return out, saved


def gate_backward(x, kv, weight, saved, grad_out):
    N = x.shape[0]
    gx = torch.empty_like(x)
    gkv = torch.empty_like(kv)
    gw = torch.empty_like(weight)
    ws = torch.empty(engram_gate_bwd_workspace_size(N), device=x.device, dtype=torch.uint8)
    engram_gate_bwd(x, kv, weight, saved, grad_out, gx, gkv, gw, ws)
    return gx, gkv, gw


def gate_backward_fused_weight(x, kv, weight, saved, grad_out, wh, we):
    """Returns grad_x, grad_kv, grad_weight, grad_wh, grad_we for weight = wh * we."""
    N = x.shape[0]
    gx, gkv = torch.empty_like(x), torch.empty_like(kv)
    gw, gwh, gwe = (torch.empty(weight.shape, device=x.device, dtype=torch.float32) for _ in range(3))
    ws = torch.empty(engram_gate_bwd_workspace_size(N), device=x.device, dtype=torch.uint8)
    engram_gate_bwd_fused_weight(x, kv, weight, saved, grad_out, wh, we, gx, gkv, gw, gwh, gwe, ws)
    return gx, gkv, gw, gwh, gwe


def gate_sep_forward(x, k, v, weight, eps: float = GATE_EPS, clamp: float = GATE_CLAMP,
                     save: bool = True):
    """Returns out and, with save, (dot, gate, rstd_x, rstd_k), each (N, 4)."""
    out = torch.empty_like(x)
    sv = [torch.empty((x.shape[0], S_GATE), device=x.device, dtype=torch.float32)
          for _ in range(4)] if save else [None] * 4
    engram_gate_sep_fwd(x, k, v, weight, out, *sv, eps=eps, clamp=clamp)
    return (out, *sv) if save else (out,)


def gate_sep_backward(grad_out, x, k, v, weight, dot, gate, rstd_x, rstd_k,
                      clamp: float = GATE_CLAMP):
    """Returns grad_x, grad_k, grad_v and grad_w_partial (ceil(N/64), 4, H)."""
    N, _, H = x.shape
    gx, gk, gv = torch.empty_like(x), torch.empty_like(k), torch.empty_like(v)
    gwp = torch.empty(((N + 63) // 64, S_GATE, H), device=x.device, dtype=torch.float32)
    ws = torch.empty(engram_gate_sep_bwd_workspace_size(N), device=x.device, dtype=torch.uint8)
    engram_gate_sep_bwd(grad_out, x, k, v, weight, dot, gate, rstd_x, rstd_k, gx, gk, gv, gwp, ws,
                        clamp=clamp)
    return gx, gk, gv, gwp


def fused_weight(wh, we):
    """fp32 (4, H) fused weight wh * we from bf16 (4, H) weights."""
    w = torch.empty(wh.shape, device=wh.device, dtype=torch.float32)
    engram_fused_weight(wh, we, w)
    return w


def fused_weight_backward(grad_w_partial, wh, we):
    """Returns (grad_w, grad_wh, grad_we) from per-block grad_w partials."""
    out = [torch.empty(wh.shape, device=wh.device, dtype=torch.float32) for _ in range(3)]
    engram_fused_weight_bwd(grad_w_partial, wh, we, *out)
    return tuple(out)


def decode_forward(e, h, conv_state, W_K, W_V, rms_w_h, rms_w_v, conv_w, max_len: int,
                   dilation: int, eps: float = GATECONV_EPS):
    """One decode step: returns y (B, d) and the new cache (B, max_len, d)."""
    B, d = h.shape
    y = torch.empty_like(h)
    ns = torch.empty((B, max_len, d), device=h.device, dtype=torch.bfloat16)
    ws = torch.empty(engram_decode_workspace_size(B, e.shape[1], d), device=h.device, dtype=torch.uint8)
    engram_decode_fwd(e, h, conv_state, W_K, W_V, rms_w_h, rms_w_v, conv_w, y, ns, ws, dilation, eps)
    return y, ns


def gateconv_forward(H, k, v, rms_w_h, rms_w_v, conv_w, eps: float = GATECONV_EPS):
    M, T, d = H.shape
    Y = torch.empty_like(H)
    vhat = torch.empty_like(H)
    sc = [torch.empty((M, T), device=H.device, dtype=torch.float32) for _ in range(4)]
    engram_gateconv_fwd(H, k, v, rms_w_h, rms_w_v, conv_w, Y, vhat, *sc, eps=eps)
    return (Y, vhat, *sc)


def gateconv_backward(dY, H, k, v, rms_w_h, rms_w_v, conv_w, vhat, alpha, rrms_h, rrms_k,
                      rrms_v, eps: float = GATECONV_EPS):
    M, T, d = H.shape
    dH, dk, dv = torch.empty_like(H), torch.empty_like(H), torch.empty_like(H)
    dwh = torch.empty(d, device=H.device, dtype=torch.float32)
    dwv = torch.empty(d, device=H.device, dtype=torch.float32)
    dcw = torch.empty((4, d), device=H.device, dtype=torch.float32)
    ws = torch.empty(engram_gateconv_bwd_workspace_size(M, T, d), device=H.device,
                     dtype=torch.uint8)
    engram_gateconv_bwd(dY, H, k, v, rms_w_h, rms_w_v, conv_w, vhat, alpha, rrms_h, rrms_k,
                        rrms_v, dH, dk, dv, dwh, dwv, dcw, ws, eps=eps)
    return dH, dk, dv, dwh, dwv, dcw
