"""Engram gate oracle: plain fp64 CPU definitions (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
path (``engram_memory_gating_gb300``) never imports it and shares no code with
it.  The arithmetic lives in ``engram_oracle.cpp``; this module only builds
that file with g++ and marshals numpy arrays through ctypes.

Each function follows the page and section cited in the C++ source:
  * gate_fwd / gate_bwd  -- cuDNN Frontend "Engram saved-state gate"
    (semantics, layout and saved-state paragraphs) and the tile-kernels 1.0.0
    engram gate tests;
  * gateconv_fwd / gateconv_bwd -- TileOPs "Engram Operators", GateConv
    section (EngramGateConvFwdOp / EngramGateConvBwdOp).

Parity status: gate_fwd, gate_bwd and the bf16 helpers are pinned by the
tests in ``tests/test_oracle_*.py`` (closed forms, invariants, brute-force
finite differences, library rounding).  gateconv_fwd / gateconv_bwd are
pinned by closed forms, causality and finite differences, and their conv
(tap order, causal padding; with a dilation in decode_fwd) against the
standard causal depthwise conv1d of torch.  The gate formula inside them (a
plain sigmoid of the normalised dot scaled by 1/sqrt(d)) is a reading the
page does not print: for that choice parity is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "engram_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

GATE_EPS = 1e-20     # cuDNN "Engram saved-state gate": default epsilon
GATE_CLAMP = 1e-6    # cuDNN "Engram saved-state gate": signed-sqrt clamp
GATECONV_EPS = 1e-6  # TileOPs EngramGateConvFwdOp: RMSNorm epsilon default


def build(force: bool = False) -> str:
    """Compile ``engram_oracle.cpp`` into ``liboracle.so`` (g++, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fopenmp",
           "-shared", "-fPIC", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            D = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [P, P, I64]
            lib.oracle_f64_to_bf16.argtypes = [P, P, I64]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            lib.oracle_gate_fwd.argtypes = [P, P, P, P, I64, I64, I64, D, D, P, P]
            lib.oracle_gate_bwd.argtypes = [P, P, P, P, P, I64, I64, I64, D, P, P, P]
            lib.oracle_gateconv_fwd.argtypes = [P, P, P, P, P, P, I64, I64, I64, D,
                                                P, P, P, P, P, P]
            lib.oracle_gateconv_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P,
                                                I64, I64, I64, P, P, P, P, P, P]
            lib.oracle_fused_weight.argtypes = [P, P, I64, P]
            lib.oracle_decode_fwd.argtypes = [P, P, P, I64, P, P, P, P, P, I64, I64, I64, I64, I64,
                                              I64, D, P, P]
            lib.oracle_fused_weight_bwd.argtypes = [P, I64, P, P, I64, P, P, P]
            for f in (lib.oracle_gate_fwd, lib.oracle_gate_bwd, lib.oracle_fused_weight, lib.oracle_decode_fwd,
                      lib.oracle_fused_weight_bwd, lib.oracle_gateconv_fwd, lib.oracle_gateconv_bwd):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_bf16_to_f64(_p(b), _p(out), b.size)
    return out


def round_bf16(values) -> np.ndarray:
    """One round-to-nearest-even step from float64 to bf16 bits (uint16)."""
    v = _f64(values)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_f64_to_bf16(_p(v), _p(out), v.size)
    return out


def gate_fwd(x, kv, w, mask=None, eps: float = GATE_EPS, clamp: float = GATE_CLAMP):
    """Saved-state gate forward in fp64.

    x (N,S,d), kv (N,(S+1)*d), w (S,d), mask (N,) bool/uint8 or None.
    Returns (out (N,S,d) exact fp64, saved (N,S,4) = gate, dot, rstd_X, rstd_key).
    """
    x = _f64(x)
    N, S, d = x.shape
    kv = _f64(kv).reshape(N, (S + 1) * d)
    w = _f64(w).reshape(S, d)
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8).reshape(N)
    out = np.empty_like(x)
    saved = np.empty((N, S, 4), dtype=np.float64)
    rc = _load().oracle_gate_fwd(_p(x), _p(kv), _p(w), None if m is None else _p(m),
                                 N, S, d, float(eps), float(clamp), _p(out), _p(saved))
    if rc != 0:
        raise ValueError("oracle_gate_fwd: bad shape")
    return out, saved


def gate_bwd(x, kv, w, saved, grad_out, clamp: float = GATE_CLAMP):
    """Saved-state gate backward in fp64.

    Returns (grad_x (N,S,d), grad_kv (N,(S+1)*d), grad_w (S,d)).
    """
    x = _f64(x)
    N, S, d = x.shape
    kv = _f64(kv).reshape(N, (S + 1) * d)
    w = _f64(w).reshape(S, d)
    sv = _f64(saved).reshape(N, S, 4)
    g = _f64(grad_out).reshape(N, S, d)
    gx = np.empty_like(x)
    gkv = np.empty_like(kv)
    gw = np.empty_like(w)
    rc = _load().oracle_gate_bwd(_p(x), _p(kv), _p(w), _p(sv), _p(g), N, S, d,
                                 float(clamp), _p(gx), _p(gkv), _p(gw))
    if rc != 0:
        raise ValueError("oracle_gate_bwd: bad shape")
    return gx, gkv, gw


def fused_weight(wh, we):
    """The gate's fused weight wh * we (fp64; exact for bf16 inputs)."""
    wh = _f64(wh)
    we = _f64(we).reshape(wh.shape)
    out = np.empty_like(wh)
    if _load().oracle_fused_weight(_p(wh), _p(we), wh.size, _p(out)) != 0:
        raise ValueError("oracle_fused_weight: bad shape")
    return out


def fused_weight_bwd(partial, wh, we):
    """partial (B, ...) per-block grad_weight; returns (grad_w, grad_wh, grad_we)
    with grad_w = sum over blocks and the product rule for wh, we."""
    wh = _f64(wh)
    we = _f64(we).reshape(wh.shape)
    pa = _f64(partial).reshape((-1,) + wh.shape)
    gw, gwh, gwe = np.empty_like(wh), np.empty_like(wh), np.empty_like(wh)
    if _load().oracle_fused_weight_bwd(_p(pa), pa.shape[0], _p(wh), _p(we), wh.size, _p(gw),
                                       _p(gwh), _p(gwe)) != 0:
        raise ValueError("oracle_fused_weight_bwd: bad shape")
    return gw, gwh, gwe


def gateconv_fwd(H, k, v, rms_w_h, rms_w_v, conv_w, eps: float = GATECONV_EPS):
    """GateConv forward in fp64.

    H, k, v (M,T,d); rms_w_h, rms_w_v (d,); conv_w (4,d).
    Returns (Y, vhat) exact fp64 (M,T,d) and (alpha, rrms_h, rrms_k, rrms_v) (M,T).
    """
    H = _f64(H)
    M, T, d = H.shape
    k = _f64(k).reshape(M, T, d)
    v = _f64(v).reshape(M, T, d)
    wh = _f64(rms_w_h).reshape(d)
    wv = _f64(rms_w_v).reshape(d)
    cw = _f64(conv_w).reshape(4, d)
    Y = np.empty_like(H)
    vhat = np.empty_like(H)
    alpha = np.empty((M, T))
    rh = np.empty((M, T))
    rk = np.empty((M, T))
    rv = np.empty((M, T))
    rc = _load().oracle_gateconv_fwd(_p(H), _p(k), _p(v), _p(wh), _p(wv), _p(cw),
                                     M, T, d, float(eps), _p(Y), _p(vhat), _p(alpha),
                                     _p(rh), _p(rk), _p(rv))
    if rc != 0:
        raise ValueError("oracle_gateconv_fwd: bad shape")
    return Y, vhat, alpha, rh, rk, rv


def gateconv_bwd(dY, H, k, v, rms_w_h, rms_w_v, conv_w, vhat, alpha, rrms_h, rrms_k,
                 rrms_v):
    """GateConv backward in fp64 at the given saved activations.

    Returns (dH, dk, dv) (M,T,d) and (drms_w_h (d,), drms_w_v (d,), dconv_w (4,d)).
    """
    H = _f64(H)
    M, T, d = H.shape
    args = [_f64(dY).reshape(M, T, d), H, _f64(k).reshape(M, T, d),
            _f64(v).reshape(M, T, d), _f64(rms_w_h).reshape(d), _f64(rms_w_v).reshape(d),
            _f64(conv_w).reshape(4, d), _f64(vhat).reshape(M, T, d),
            _f64(alpha).reshape(M, T), _f64(rrms_h).reshape(M, T),
            _f64(rrms_k).reshape(M, T), _f64(rrms_v).reshape(M, T)]
    dH = np.empty_like(H)
    dk = np.empty_like(H)
    dv = np.empty_like(H)
    dwh = np.empty(d)
    dwv = np.empty(d)
    dcw = np.empty((4, d))
    rc = _load().oracle_gateconv_bwd(*[_p(a) for a in args], M, T, d, _p(dH), _p(dk),
                                     _p(dv), _p(dwh), _p(dwv), _p(dcw))
    if rc != 0:
        raise ValueError("oracle_gateconv_bwd: bad shape")
    return dH, dk, dv, dwh, dwv, dcw


def decode_fwd(e, h, conv_state, W_K, W_V, rms_w_h, rms_w_v, conv_w, max_len: int, dilation: int,
               eps: float = GATECONV_EPS):
    """GateConv decode step in fp64.

    e (B,d_mem), h (B,d), conv_state (B,L,d) with L <= max_len, W_K, W_V (d_mem,d),
    rms_w_h, rms_w_v (d,), conv_w (w,d).  Returns y (B,d) and new_state
    (B,max_len,d), exact (the last state row is this token's exact u).
    """
    e = _f64(e)
    B, dmem = e.shape
    h = _f64(h).reshape(B, -1)
    d = h.shape[1]
    st = _f64(conv_state).reshape(B, -1, d)
    L = st.shape[1]
    WK = _f64(W_K).reshape(dmem, d)
    WV = _f64(W_V).reshape(dmem, d)
    wh = _f64(rms_w_h).reshape(d)
    wv = _f64(rms_w_v).reshape(d)
    cw = _f64(conv_w).reshape(-1, d)
    y = np.empty((B, d))
    ns = np.empty((B, max_len, d))
    rc = _load().oracle_decode_fwd(_p(e), _p(h), _p(st), L, _p(WK), _p(WV), _p(wh), _p(wv), _p(cw),
                                   B, dmem, d, int(max_len), cw.shape[0], int(dilation), float(eps),
                                   _p(y), _p(ns))
    if rc != 0:
        raise ValueError("oracle_decode_fwd: bad shape")
    return y, ns
