"""Guard bands around every output and workspace (a stand-in for a memory
checker): each buffer an entry point writes is placed inside a larger device
buffer whose 4 KB margins on both sides, and the buffer itself, are filled
with seeded random bytes.  After the call the margins must be unchanged (no
store ran past either end of any output row slice, ring refill or workspace
slot), and the outputs must equal, bit for bit, those of an ordinary call with
freshly allocated buffers (so every element was written: a skipped element
would still hold the poison).  One ragged and one full-size shape per entry
point, through the C ABI.
"""
import pytest
import torch

import engram_memory_gating_gb300 as eg
from engram_memory_gating_gb300.inputs import decode_inputs, gate_inputs, gateconv_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
MARGIN = 4096


class Guarded:
    """A tensor of `shape` / `dtype` at byte offset MARGIN of a poisoned buffer."""

    def __init__(self, shape, dtype, seed):
        n = 1
        for s in shape:
            n *= s
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        g = torch.Generator(device="cpu").manual_seed(seed)
        poison = torch.randint(0, 256, (self.nbytes + 2 * MARGIN,), generator=g, dtype=torch.uint8)
        self.base = poison.to(DEV)
        self.head = poison[:MARGIN].clone()
        self.tail = poison[MARGIN + self.nbytes:].clone()
        self.t = self.base[MARGIN:MARGIN + self.nbytes].view(dtype).view(shape)

    def check(self, name):
        got = self.base.cpu()
        assert torch.equal(got[:MARGIN], self.head), f"{name}: bytes before the buffer changed"
        assert torch.equal(got[MARGIN + self.nbytes:], self.tail), f"{name}: bytes after the buffer changed"


def like(t, seed):
    return Guarded(tuple(t.shape), t.dtype, seed)


def ws_guard(nbytes, seed):
    return Guarded((max(1, nbytes),), torch.uint8, seed)


def same_bits(a, b, name):
    if a.dtype in (torch.bfloat16, torch.float16):
        a, b = a.view(torch.int16), b.view(torch.int16)
    elif a.dtype == torch.float32:
        a, b = a.view(torch.int32), b.view(torch.int32)
    assert torch.equal(a, b), f"{name}: differs from an ordinary call"


@pytest.fixture(autouse=True)
def no_device_error():
    yield
    assert eg.engram_device_error() == 0


@pytest.mark.parametrize("N", [321, 8192])
def test_gate_fwd_bwd(N):
    inp = gate_inputs(N, 60 + N % 7, device=DEV, mask="bern0.9")
    out, saved = eg.gate_forward(inp["x"], inp["kv"], inp["weight"], inp["mask"])
    go, gs = like(out, 1), like(saved, 2)
    eg.engram_gate_fwd(inp["x"], inp["kv"], inp["weight"], inp["mask"], go.t, gs.t)
    torch.cuda.synchronize()
    go.check("out"), gs.check("saved")
    same_bits(go.t, out, "out"), same_bits(gs.t, saved, "saved")
    Nb = N // 64 * 64
    x, kv, sv, gout = inp["x"][:Nb], inp["kv"][:Nb], saved[:Nb], inp["grad_out"][:Nb]
    ref = eg.gate_backward(x, kv, inp["weight"], sv, gout)
    gx, gkv, gw = like(ref[0], 3), like(ref[1], 4), like(ref[2], 5)
    ws = ws_guard(eg.engram_gate_bwd_workspace_size(Nb), 6)
    eg.engram_gate_bwd(x, kv, inp["weight"], sv, gout, gx.t, gkv.t, gw.t, ws.t)
    torch.cuda.synchronize()
    for g, r, name in ((gx, ref[0], "grad_x"), (gkv, ref[1], "grad_kv"), (gw, ref[2], "grad_weight")):
        g.check(name)
        same_bits(g.t, r, name)
    ws.check("workspace")
    # the entry point without a workspace argument (its array is internal)
    if Nb <= 2048:
        gx2, gkv2, gw2 = like(ref[0], 7), like(ref[1], 8), like(ref[2], 9)
        eg.engram_gate_bwd_noalloc(x, kv, inp["weight"], sv, gout, gx2.t, gkv2.t, gw2.t)
        torch.cuda.synchronize()
        for g, r, name in ((gx2, ref[0], "grad_x"), (gkv2, ref[1], "grad_kv"), (gw2, ref[2], "grad_weight")):
            g.check(name + " (noalloc)")
            same_bits(g.t, r, name + " (noalloc)")


@pytest.mark.parametrize("N,H", [(100, 264), (8192, 4096)])
def test_gate_sep_fwd_bwd(N, H):
    inp = gate_inputs(N, 70, device=DEV, d=H)
    k = inp["kv"][:, :4 * H].reshape(N, 4, H).contiguous()
    v = inp["kv"][:, 4 * H:].contiguous()
    ref = eg.gate_sep_forward(inp["x"], k, v, inp["weight"])
    gd = [like(t, 10 + i) for i, t in enumerate(ref)]
    eg.engram_gate_sep_fwd(inp["x"], k, v, inp["weight"], *(g.t for g in gd))
    torch.cuda.synchronize()
    for g, r, name in zip(gd, ref, ("out", "dot", "gate", "rstd_x", "rstd_k")):
        g.check(name)
        same_bits(g.t, r, name)
    rb = eg.gate_sep_backward(inp["grad_out"], inp["x"], k, v, inp["weight"], *ref[1:])
    gb = [like(t, 20 + i) for i, t in enumerate(rb)]
    ws = ws_guard(eg.engram_gate_sep_bwd_workspace_size(N), 25)
    eg.engram_gate_sep_bwd(inp["grad_out"], inp["x"], k, v, inp["weight"], *ref[1:],
                           *(g.t for g in gb), ws.t)
    torch.cuda.synchronize()
    for g, r, name in zip(gb, rb, ("grad_x", "grad_k", "grad_v", "grad_w_partial")):
        g.check(name)
        same_bits(g.t, r, name)
    ws.check("workspace")


@pytest.mark.parametrize("n,nblocks", [(4 * 264, 2), (4 * 5120, 128)])
def test_fused_weight(n, nblocks):
    g = torch.Generator(device="cpu").manual_seed(n)
    wh = (1 + 0.1 * torch.randn(n, generator=g)).to(torch.bfloat16).to(DEV)
    we = (1 + 0.1 * torch.randn(n, generator=g)).to(torch.bfloat16).to(DEV)
    part = torch.randn((nblocks, n), generator=g).to(DEV)
    w_ref = eg.fused_weight(wh, we)
    gw = like(w_ref, 30)
    eg.engram_fused_weight(wh, we, gw.t)
    torch.cuda.synchronize()
    gw.check("weight")
    same_bits(gw.t, w_ref, "weight")
    rb = eg.fused_weight_backward(part, wh, we)
    gb = [like(t, 31 + i) for i, t in enumerate(rb)]
    eg.engram_fused_weight_bwd(part, wh, we, *(x.t for x in gb))
    torch.cuda.synchronize()
    for x, r, name in zip(gb, rb, ("grad_w", "grad_wh", "grad_we")):
        x.check(name)
        same_bits(x.t, r, name)


@pytest.mark.parametrize("M,T,d", [(2, 45, 1032), (4, 4096, 4096), (3, 70, 7168)])
def test_gateconv_fwd_bwd(M, T, d):
    """Guard bands around every output and the workspace; d = 7168 runs the
    backward as groups of CTAs exchanging through the workspace's records,
    the other shapes as thread-block clusters."""
    ci = gateconv_inputs(M, T, d, 80, device=DEV)
    ref = eg.gateconv_forward(ci["H"], ci["k"], ci["v"], ci["rms_w_h"], ci["rms_w_v"], ci["conv_w"])
    gf = [like(t, 40 + i) for i, t in enumerate(ref)]
    eg.engram_gateconv_fwd(ci["H"], ci["k"], ci["v"], ci["rms_w_h"], ci["rms_w_v"], ci["conv_w"],
                           *(g.t for g in gf))
    torch.cuda.synchronize()
    for g, r, name in zip(gf, ref, ("Y", "vhat", "alpha", "rrms_h", "rrms_k", "rrms_v")):
        g.check(name)
        same_bits(g.t, r, name)
    args = (ci["dY"], ci["H"], ci["k"], ci["v"], ci["rms_w_h"], ci["rms_w_v"], ci["conv_w"], *ref[1:])
    rb = eg.gateconv_backward(*args)
    gb = [like(t, 50 + i) for i, t in enumerate(rb)]
    ws = ws_guard(eg.engram_gateconv_bwd_workspace_size(M, T, d), 56)
    eg.engram_gateconv_bwd(*args, *(g.t for g in gb), ws.t)
    torch.cuda.synchronize()
    for g, r, name in zip(gb, rb, ("dH", "dk", "dv", "drms_w_h", "drms_w_v", "dconv_w")):
        g.check(name)
        same_bits(g.t, r, name)
    ws.check("workspace")


@pytest.mark.parametrize("B,dm,d,L,max_len,w,dil", [(3, 72, 192, 5, 8, 4, 2),
                                                    (8, 1024, 4096, 16, 16, 4, 3)])
def test_decode(B, dm, d, L, max_len, w, dil):
    di = decode_inputs(B, dm, d, L, w, seed=90, device=DEV)
    y_ref, ns_ref = eg.decode_forward(di["e"], di["h"], di["conv_state"], di["W_K"], di["W_V"],
                                      di["rms_w_h"], di["rms_w_v"], di["conv_w"], max_len, dil)
    gy, gns = like(y_ref, 60), like(ns_ref, 61)
    ws = ws_guard(eg.engram_decode_workspace_size(B, dm, d), 62)
    eg.engram_decode_fwd(di["e"], di["h"], di["conv_state"], di["W_K"], di["W_V"], di["rms_w_h"],
                         di["rms_w_v"], di["conv_w"], gy.t, gns.t, ws.t, dil)
    torch.cuda.synchronize()
    gy.check("y"), gns.check("new_state"), ws.check("workspace")
    same_bits(gy.t, y_ref, "y")
    same_bits(gns.t, ns_ref, "new_state")
