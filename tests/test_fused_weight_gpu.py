"""GPU parity of the gate's fused weight and its product rule (cuDNN Frontend
"Engram saved-state gate", semantics paragraph; tile-kernels engram
fused-weight and backward tests) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import engram_memory_gating_gb300 as eg
import oracle
from engram_memory_gating_gb300.inputs import bf16_bits, gate_inputs
from tolerance import bf16_bits_to_f64, check_f32

pytestmark = pytest.mark.gpu


def f64(t):
    if t.dtype == torch.bfloat16:
        return bf16_bits_to_f64(bf16_bits(t)).reshape(tuple(t.shape))
    return t.detach().double().cpu().numpy()


@pytest.mark.parametrize("H", [8, 800, 5120])
def test_fused_weight_is_bit_exact(H):
    g = torch.Generator().manual_seed(H)
    wh = torch.randn((4, H), generator=g).to(torch.bfloat16).cuda()
    we = (3 * torch.randn((4, H), generator=g)).to(torch.bfloat16).cuda()
    w = eg.fused_weight(wh, we)
    torch.cuda.synchronize()
    assert np.array_equal(w.cpu().double().numpy(), oracle.fused_weight(f64(wh), f64(we)))


@pytest.mark.parametrize("nblocks,H", [(1, 64), (3, 1000), (129, 5120)])
def test_fused_weight_backward_sums_and_product_rule(nblocks, H):
    g = torch.Generator().manual_seed(nblocks)
    wh = torch.randn((4, H), generator=g).to(torch.bfloat16).cuda()
    we = torch.randn((4, H), generator=g).to(torch.bfloat16).cuda()
    parts = torch.randn((nblocks, 4, H), generator=g).cuda()
    gw, gwh, gwe = eg.fused_weight_backward(parts, wh, we)
    torch.cuda.synchronize()
    egw, egwh, egwe = oracle.fused_weight_bwd(f64(parts), f64(wh), f64(we))
    # fp32 results of exact fp64 values: within a few fp32 ulps
    check_f32("grad_w", gw.cpu().numpy(), egw, rel=1e-6, abs_=1e-6)
    check_f32("grad_wh", gwh.cpu().numpy(), egwh, rel=1e-6, abs_=1e-6)
    check_f32("grad_we", gwe.cpu().numpy(), egwe, rel=1e-6, abs_=1e-6)


def test_chain_through_the_separate_tensor_gate():
    """w = wh * we -> gate forward / backward -> per-block partials -> grad_wh,
    grad_we, against the oracle's gate backward and product rule."""
    N, H = 200, 512
    inp = gate_inputs(N, 41, d=H)
    g = torch.Generator().manual_seed(41)
    wh = (1 + 0.3 * torch.randn((4, H), generator=g)).to(torch.bfloat16)
    we = (1 + 0.3 * torch.randn((4, H), generator=g)).to(torch.bfloat16)
    k = inp["kv"][:, :4 * H].reshape(N, 4, H).contiguous()
    v = inp["kv"][:, 4 * H:].contiguous()
    d = {n: t.cuda() for n, t in (("x", inp["x"]), ("k", k), ("v", v), ("g", inp["grad_out"]),
                                  ("wh", wh), ("we", we))}
    w = eg.fused_weight(d["wh"], d["we"])
    out, dot, gate, rx, rk = eg.gate_sep_forward(d["x"], d["k"], d["v"], w)
    _, _, _, parts = eg.gate_sep_backward(d["g"], d["x"], d["k"], d["v"], w, dot, gate, rx, rk)
    gw, gwh, gwe = eg.fused_weight_backward(parts, d["wh"], d["we"])
    torch.cuda.synchronize()
    saved = np.stack([f64(t) for t in (gate, dot, rx, rk)], axis=-1)
    w64 = oracle.fused_weight(f64(wh), f64(we))
    _, _, egw = oracle.gate_bwd(f64(inp["x"]), f64(inp["kv"]), w64, saved, f64(inp["grad_out"]))
    check_f32("grad_w", gw.cpu().numpy(), egw)
    check_f32("grad_wh", gwh.cpu().numpy(), egw * f64(we))
    check_f32("grad_we", gwe.cpu().numpy(), egw * f64(wh))


@pytest.mark.parametrize("N,mask", [(64, "all"), (320, "bern0.9"), (8192, "bern0.9")])
def test_packed_backward_applies_the_product_rule_in_its_merge(N, mask):
    """engram_gate_bwd_fused_weight: w = wh * we -> packed gate forward ->
    backward whose grad_weight merge also writes grad_wh = grad_w * we and
    grad_we = grad_w * wh.  Against the oracle's gate backward and product
    rule, and bitwise against engram_gate_bwd followed by the separate product
    rule call (one block holding grad_weight), which it replaces."""
    inp = gate_inputs(N, 50 + N % 11, device="cuda", mask=mask)
    g = torch.Generator(device="cuda").manual_seed(N)
    wh = (1 + 0.3 * torch.randn((4, 5120), generator=g, device="cuda")).to(torch.bfloat16)
    we = (1 + 0.3 * torch.randn((4, 5120), generator=g, device="cuda")).to(torch.bfloat16)
    w = eg.fused_weight(wh, we)
    out, saved = eg.gate_forward(inp["x"], inp["kv"], w, inp["mask"])
    gx, gkv, gw, gwh, gwe = eg.gate_backward_fused_weight(inp["x"], inp["kv"], w, saved,
                                                          inp["grad_out"], wh, we)
    rx, rkv, rw = eg.gate_backward(inp["x"], inp["kv"], w, saved, inp["grad_out"])
    _, rwh, rwe = eg.fused_weight_backward(rw.unsqueeze(0), wh, we)
    # grad_weight may be skipped: the product-rule outputs are unchanged
    gwh2, gwe2 = torch.empty_like(gwh), torch.empty_like(gwe)
    ws = torch.empty(eg.engram_gate_bwd_workspace_size(N), device="cuda", dtype=torch.uint8)
    eg.engram_gate_bwd_fused_weight(inp["x"], inp["kv"], w, saved, inp["grad_out"], wh, we,
                                    torch.empty_like(gx), torch.empty_like(gkv), None, gwh2, gwe2, ws)
    torch.cuda.synchronize()
    for a, b in ((gx, rx), (gkv, rkv)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for a, b in ((gw, rw), (gwh, rwh), (gwe, rwe), (gwh2, gwh), (gwe2, gwe)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    _, _, egw = oracle.gate_bwd(f64(inp["x"]), f64(inp["kv"]), f64(w), f64(saved),
                                f64(inp["grad_out"]))
    _, egwh, egwe = oracle.fused_weight_bwd(egw[None], f64(wh), f64(we))
    check_f32("grad_weight (fused-weight bwd)", gw.cpu().numpy(), egw)
    check_f32("grad_wh (fused-weight bwd)", gwh.cpu().numpy(), egwh)
    check_f32("grad_we (fused-weight bwd)", gwe.cpu().numpy(), egwe)
