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
