"""Host-side tests of the C ABI (no GPU needed).

The library must load and export every function include/engram.h declares,
and argument validation must reject bad calls before any device work.  The
fake pointers used here are never valid for a kernel: every call below fails
validation, so nothing is enqueued even on a machine with a GPU.
"""
import ctypes
import os
import re

import pytest
import torch

import engram_memory_gating_gb300 as eg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "include", "engram.h")

OK, ENULL, EALIGN, ESHAPE, EOVERLAP, EWS, EDEV = 0, 1, 2, 3, 4, 5, 6


def declared_functions():
    text = open(HDR).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(engram_[a-z0-9_]+)\s*\(", text)))


def test_library_loads_and_exports_every_declared_symbol():
    lib = eg.load()
    names = declared_functions()
    assert len(names) >= 9
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(names) == set(eg.EXPORTED_SYMBOLS)


def test_status_strings():
    lib = eg.load()
    for code in range(8):
        assert lib.engram_status_string(code)


def test_gate_bwd_workspace_size_formula():
    # 4 * (16 N + 4 * 5120 * (N // 64)) bytes
    for N in (64, 128, 4096, 8192, 8256, 65536, 4194240):
        assert eg.engram_gate_bwd_workspace_size(N) == 4 * (16 * N + 4 * 5120 * (N // 64))
    assert eg.engram_gate_bwd_workspace_size(8192) == 11010048
    for N in (0, 1, 63, 100, 8200, -64, 4194304):
        assert eg.engram_gate_bwd_workspace_size(N) == 0


def test_gateconv_bwd_workspace_size():
    # one 6*d fp32 slot per token range: up to 256 ranges of >= 16 tokens, but
    # at least enough for ranges of at most 1024 tokens; then the exchange
    # records of up to 1024 CTAs (2 x 16 eight-byte words each)
    def slots(M, T):
        return max(M * ((T + 1023) // 1024), min(256, M * ((T + 15) // 16)))

    xrec = 1024 * 2 * 16 * 8
    for M, T, d in ((4, 4096, 4096), (8, 8192, 7168), (1, 1, 8), (2, 96, 512), (300, 4, 64),
                    (1, 5, 8192), (2, 300000, 64)):
        assert eg.engram_gateconv_bwd_workspace_size(M, T, d) == slots(M, T) * 6 * d * 4 + xrec
    assert eg.engram_gateconv_bwd_workspace_size(8, 8192, 7168) == 256 * 6 * 7168 * 4 + 262144
    for shape in ((0, 4, 64), (1, 0, 64), (1, 4, 12), (1, 4, 0), (1, 4, 8200), (1, 4, 8 * 1031)):
        assert eg.engram_gateconv_bwd_workspace_size(*shape) == 0


A = 1 << 20  # fake, 16-byte aligned, never dereferenced


def p(v):
    return ctypes.c_void_p(v)


def gate_fwd(x=A, kv=2 * A * 1024, w=3 * A * 2048, mask=None, out=4 * A * 4096, saved=None,
             N=4, eps=1e-20):
    return eg.load().engram_gate_fwd(p(x), p(kv), p(w), p(mask) if mask else None, p(out),
                                     p(saved) if saved else None, N, eps, None)


def test_gate_fwd_validation():
    assert gate_fwd(x=0) == ENULL
    assert gate_fwd(out=0) == ENULL
    assert gate_fwd(x=A + 8) == EALIGN
    assert gate_fwd(saved=5 * A * 8192 + 4) == EALIGN
    assert gate_fwd(N=0) == ESHAPE
    assert gate_fwd(N=4194241) == ESHAPE
    assert gate_fwd(out=A) == EOVERLAP                       # out aliases x
    assert gate_fwd(out=A + 4 * 40960 - 16) == EOVERLAP      # partial overlap
    assert gate_fwd(saved=4 * A * 4096 + 16) == EOVERLAP     # saved inside out


def gate_bwd(N=64, ws_bytes=None, **kw):
    lib = eg.load()
    args = dict(x=A, kv=A * 100, w=A * 200, saved=A * 300, g=A * 400, gx=A * 500,
                gkv=A * 600, gw=A * 700, ws=A * 800)
    args.update(kw)
    wsb = eg.engram_gate_bwd_workspace_size(N) if ws_bytes is None else ws_bytes
    return lib.engram_gate_bwd(*(p(args[k]) for k in ("x", "kv", "w", "saved", "g", "gx",
                                                      "gkv", "gw", "ws")), wsb, N, None)


def test_gate_bwd_validation():
    assert gate_bwd(ws=0) == ENULL
    assert gate_bwd(N=100, ws_bytes=1 << 30) == ESHAPE
    assert gate_bwd(N=4194304, ws_bytes=1 << 40) == ESHAPE    # 65536 * 64: past the limit
    assert gate_bwd(N=8200, ws_bytes=1 << 30) == ESHAPE       # not a multiple of 64
    assert gate_bwd(N=0, ws_bytes=1 << 30) == ESHAPE
    assert gate_bwd(gx=A * 500 + 2) == EALIGN
    assert gate_bwd(ws_bytes=eg.engram_gate_bwd_workspace_size(64) - 16) == EWS
    assert gate_bwd(gkv=A * 100) == EOVERLAP                 # grad_kv aliases kv
    assert gate_bwd(ws=A * 700 + 1024) == EOVERLAP           # workspace inside grad_weight


def test_gateconv_validation():
    lib = eg.load()
    base = [A * i for i in range(1, 13)]

    def call(ptrs, M=2, T=8, d=64):
        return lib.engram_gateconv_fwd(*(p(v) for v in ptrs), M, T, d, 1e-6, None)

    assert call([0] + base[1:]) == ENULL
    assert call(base, d=12) == ESHAPE
    assert call(base, M=0) == ESHAPE
    assert call(base, d=8 * 1031) == ESHAPE
    bad = list(base)
    bad[7] = base[7] + 4
    assert call(bad) == EALIGN
    ov = list(base)
    ov[6] = base[0]                                          # Y aliases H
    assert call(ov) == EOVERLAP


@pytest.mark.skipif(torch.cuda.is_available(), reason="needs a host without a GPU")
def test_valid_arguments_without_a_device_report_device_error():
    assert gate_fwd() == EDEV
    info = eg._LaunchInfo()
    assert eg.load().engram_launch_info(0, 64, 0, 0, ctypes.byref(info)) == EDEV


def test_binding_has_no_cpu_fallback():
    # the product package never imports the oracle
    import engram_memory_gating_gb300 as pkg
    src_dir = os.path.dirname(pkg.__file__)
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle|from\s+\.\.\s*import\s+oracle)",
                     re.M)
    for name in os.listdir(src_dir):
        if name.endswith(".py"):
            assert not pat.search(open(os.path.join(src_dir, name)).read()), name


def test_gate_sep_validation_and_workspace():
    lib = eg.load()
    assert eg.engram_gate_sep_bwd_workspace_size(1) == 64
    assert eg.engram_gate_sep_bwd_workspace_size(8192) == 64 * 8192
    assert eg.engram_gate_sep_bwd_workspace_size(0) == 0

    def fwd(ptrs, N=4, H=64):
        return lib.engram_gate_sep_fwd(*(p(v) if v else None for v in ptrs), N, H, 1e-20, 1e-6, None)

    base = [A * i for i in range(1, 10)]       # x, k, v, weight, out, dot, gate, rstd_x, rstd_k
    assert fwd([0] + base[1:]) == ENULL
    partial = list(base)
    partial[6] = 0                             # three of the four saved arrays
    assert fwd(partial) == ENULL
    assert fwd(base, H=12) == ESHAPE
    assert fwd(base, H=0) == ESHAPE
    assert fwd(base, N=0) == ESHAPE
    bad = list(base)
    bad[2] = base[2] + 8
    assert fwd(bad) == EALIGN
    ov = list(base)
    ov[4] = base[1]                            # out aliases k
    assert fwd(ov) == EOVERLAP

    def bwd(ptrs, ws_bytes=1 << 20, N=4, H=64):
        return lib.engram_gate_sep_bwd(*(p(v) if v else None for v in ptrs), ws_bytes, N, H, 1e-6, None)

    b14 = [A * i for i in range(1, 15)]
    assert bwd([0] + b14[1:]) == ENULL
    assert bwd(b14, H=7) == ESHAPE
    assert bwd(b14, ws_bytes=64 * 4 - 16) == EWS
    ov = list(b14)
    ov[12] = b14[0]                            # grad_w_partial aliases grad_out
    assert bwd(ov) == EOVERLAP


def test_fused_weight_validation():
    lib = eg.load()
    assert lib.engram_fused_weight(None, p(A), p(2 * A), 64, None) == ENULL
    assert lib.engram_fused_weight(p(A), p(2 * A), p(3 * A), 0, None) == ESHAPE
    assert lib.engram_fused_weight(p(A + 2), p(2 * A), p(3 * A), 64, None) == EALIGN
    assert lib.engram_fused_weight(p(A), p(2 * A), p(A + 16), 64, None) == EOVERLAP
    bwd = lib.engram_fused_weight_bwd
    assert bwd(p(A), 1, p(2 * A), p(3 * A), None, None, p(5 * A), 64, None) == ENULL
    assert bwd(p(A), 0, p(2 * A), p(3 * A), None, p(4 * A), p(5 * A), 64, None) == ESHAPE
    assert bwd(p(A), 2, p(2 * A), p(3 * A), None, p(A + 256), p(5 * A), 64, None) == EOVERLAP


def test_decode_validation_and_workspace():
    lib = eg.load()
    assert eg.engram_decode_workspace_size(8, 1024, 4096) > 0
    for shape in ((0, 64, 64), (1, 12, 64), (1, 64, 100), (1, 64, 32)):
        assert eg.engram_decode_workspace_size(*shape) == 0
    ws = eg.engram_decode_workspace_size(2, 64, 64)
    ptrs = [A * i for i in range(1, 13)]   # e, h, state, W_K, W_V, wh, wv, cw, y, new_state, workspace

    def call(pt=ptrs, L=2, B=2, dmem=64, d=64, max_len=4, w=4, dil=1, wsb=ws):
        return lib.engram_decode_fwd(p(pt[0]), p(pt[1]), p(pt[2]) if pt[2] else None, L,
                                     *(p(v) if v else None for v in pt[3:11]), wsb, B, dmem, d,
                                     max_len, w, dil, 1e-6, None)

    assert call(pt=[0] + ptrs[1:]) == ENULL
    no_state = list(ptrs)
    no_state[2] = 0
    assert call(pt=no_state, L=1) == ENULL          # a non-empty cache needs its pointer
    assert call(L=5) == ESHAPE                      # L > max_len
    assert call(w=0) == ESHAPE
    assert call(dil=0) == ESHAPE
    assert call(wsb=ws - 16) == EWS
    ov = list(ptrs)
    ov[9] = ptrs[2]                                 # the new cache aliases the old one
    assert call(pt=ov) == EOVERLAP
