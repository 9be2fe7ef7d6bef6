"""GPU parity of GateConv (TileOPs "Engram Operators", GateConv section)
against the fp64 oracle, through the C ABI.

Workloads: H, k, v ~N(0,1) bf16, rms weights 1 + 0.1 N(0,1), conv_w ~N(0, 0.25)
(variance), dY ~N(0,1), eps 1e-6; the large case scales H by 10 and draws v
~N(0, 0.1).  Tolerances are in tests/tolerance.py.
"""
import numpy as np
import pytest
import torch

import engram_memory_gating_gb300 as eg
import oracle
from engram_memory_gating_gb300.inputs import bf16_bits, gateconv_inputs
from tolerance import bf16_bits_to_f64, check_bf16, check_f32, check_f32_sum

pytestmark = pytest.mark.gpu
DEV = "cuda"


def f64(t):
    if t.dtype == torch.bfloat16:
        return bf16_bits_to_f64(bf16_bits(t)).reshape(tuple(t.shape))
    return t.detach().double().cpu().numpy()


@pytest.fixture(autouse=True)
def no_device_error():
    yield
    assert eg.engram_device_error() == 0


def oracle_fwd(inp):
    return oracle.gateconv_fwd(*(f64(inp[k]) for k in ("H", "k", "v", "rms_w_h", "rms_w_v",
                                                        "conv_w")))


def check_fwd(res, exact):
    Y, vhat, alpha, rh, rk, rv = res
    eY, evh, ea, erh, erk, erv = exact
    check_bf16("Y", bf16_bits(Y), eY)
    check_bf16("vhat", bf16_bits(vhat), evh)
    check_f32("alpha", alpha.cpu().numpy(), ea)
    check_f32("rrms_h", rh.cpu().numpy(), erh)
    check_f32("rrms_k", rk.cpu().numpy(), erk)
    check_f32("rrms_v", rv.cpu().numpy(), erv)


def check_bwd(res, exact, sums=True):
    dH, dk, dv, dwh, dwv, dcw = res
    eH, ek, ev, ewh, ewv, ecw = exact
    check_bf16("dH", bf16_bits(dH), eH, floor="all")
    check_bf16("dk", bf16_bits(dk), ek, floor="all")
    check_bf16("dv", bf16_bits(dv), ev)
    if sums:
        check_f32_sum("drms_w_h", dwh.cpu().numpy(), ewh)
        check_f32_sum("drms_w_v", dwv.cpu().numpy(), ewv)
        check_f32_sum("dconv_w", dcw.cpu().numpy(), ecw)


# shapes span one-warp CTAs (d = 8, 64), ragged last column slices (d = 1032:
# 640 + 392 columns; d = 6152: 6 x 896 + 776), the largest d (8 CTAs of 1024
# columns), rows shorter than the conv (T = 1, 2) and rows cut into several
# token ranges with halos.  The backward runs d = 6152, 7168 and 8192 as
# groups of CTAs exchanging through global memory (M = 32, T = 64: 32 ranges
# on 21 groups, so groups take a second range), the others as clusters.
SMALL = [(1, 1, 8, 0), (2, 37, 64, 1), (3, 129, 512, 2), (1, 1000, 64, 3), (2, 300, 4096, 4),
         (1, 70, 7168, 5), (1, 5, 5120, 6), (2, 45, 1032, 7), (1, 40, 8192, 8), (3, 2, 264, 9),
         (1, 2500, 64, 10), (1, 40, 4200, 11), (2, 33, 6144, 12), (2, 45, 6152, 15),
         (32, 64, 7168, 16)]


@pytest.mark.parametrize("M,T,d,seed", SMALL)
def test_fwd_bwd_parity_small(M, T, d, seed):
    inp = gateconv_inputs(M, T, d, seed)
    dv = {k: v.to(DEV) for k, v in inp.items()}
    res = eg.gateconv_forward(dv["H"], dv["k"], dv["v"], dv["rms_w_h"], dv["rms_w_v"],
                              dv["conv_w"])
    exact = oracle_fwd(inp)
    check_fwd(res, exact)
    # backward fed from the GPU forward's saved tensors (both sides see them)
    Y, vhat, alpha, rh, rk, rv = res
    g = eg.gateconv_backward(dv["dY"], dv["H"], dv["k"], dv["v"], dv["rms_w_h"], dv["rms_w_v"],
                             dv["conv_w"], vhat, alpha, rh, rk, rv)
    ex = oracle.gateconv_bwd(f64(inp["dY"]), f64(inp["H"]), f64(inp["k"]), f64(inp["v"]),
                             f64(inp["rms_w_h"]), f64(inp["rms_w_v"]), f64(inp["conv_w"]),
                             f64(vhat), f64(alpha), f64(rh), f64(rk), f64(rv))
    check_bwd(g, ex)


def test_bwd_from_oracle_saved():
    M, T, d = 2, 200, 1024
    inp = gateconv_inputs(M, T, d, 12)
    Y, vh, a, rh, rk, rv = oracle_fwd(inp)
    vh_bits = oracle.round_bf16(vh)
    vh16 = torch.from_numpy(vh_bits.view(np.int16)).view(torch.bfloat16)
    sc = [torch.from_numpy(t.astype(np.float32)) for t in (a, rh, rk, rv)]
    dv = {k: v.to(DEV) for k, v in inp.items()}
    g = eg.gateconv_backward(dv["dY"], dv["H"], dv["k"], dv["v"], dv["rms_w_h"], dv["rms_w_v"],
                             dv["conv_w"], vh16.to(DEV), *(t.to(DEV) for t in sc))
    ex = oracle.gateconv_bwd(f64(inp["dY"]), f64(inp["H"]), f64(inp["k"]), f64(inp["v"]),
                             f64(inp["rms_w_h"]), f64(inp["rms_w_v"]), f64(inp["conv_w"]),
                             bf16_bits_to_f64(vh_bits), *(t.double().numpy() for t in sc))
    check_bwd(g, ex)


def test_zero_conv_gives_vhat_bitwise():
    inp = gateconv_inputs(2, 333, 2048, 13, device=DEV)
    res = eg.gateconv_forward(inp["H"], inp["k"], inp["v"], inp["rms_w_h"], inp["rms_w_v"],
                              torch.zeros_like(inp["conv_w"]))
    assert torch.equal(res[0].view(torch.int16), res[1].view(torch.int16))


def test_bwd_is_deterministic():
    inp = gateconv_inputs(2, 1024, 1024, 14, device=DEV)
    res = eg.gateconv_forward(inp["H"], inp["k"], inp["v"], inp["rms_w_h"], inp["rms_w_v"],
                              inp["conv_w"])
    args = (inp["dY"], inp["H"], inp["k"], inp["v"], inp["rms_w_h"], inp["rms_w_v"],
            inp["conv_w"], *res[1:])
    a = eg.gateconv_backward(*args)
    b = eg.gateconv_backward(*args)
    for x, y in zip(a, b):
        if x.dtype == torch.bfloat16:
            assert torch.equal(x.view(torch.int16), y.view(torch.int16))
        else:
            assert torch.equal(x, y)


def test_full_config_m4_t4096_d4096():
    """M=4, T=4096, d=4096: every element of every output against the oracle."""
    M, T, d = 4, 4096, 4096
    inp = gateconv_inputs(M, T, d, 21, device=DEV)
    res = eg.gateconv_forward(inp["H"], inp["k"], inp["v"], inp["rms_w_h"], inp["rms_w_v"],
                              inp["conv_w"])
    g = eg.gateconv_backward(inp["dY"], inp["H"], inp["k"], inp["v"], inp["rms_w_h"],
                             inp["rms_w_v"], inp["conv_w"], *res[1:])
    torch.cuda.synchronize()
    check_fwd(res, oracle_fwd(inp))
    ex = oracle.gateconv_bwd(f64(inp["dY"]), f64(inp["H"]), f64(inp["k"]), f64(inp["v"]),
                             f64(inp["rms_w_h"]), f64(inp["rms_w_v"]), f64(inp["conv_w"]),
                             *(f64(t) for t in res[1:]))
    check_bwd(g, ex)


def test_full_config_m8_t8192_d7168():
    """M=8, T=8192, d=7168, H x10, v ~N(0, 0.1).  The fp32 weight gradients,
    summed by the GPU over all 65,536 tokens, against the oracle's sum: the
    oracle runs each batch row m whole (1, 8192, 7168), fed that row's slice of
    the GPU forward's saved tensors, and the eight per-row results are added in
    fp64 (a weight gradient is a plain sum over tokens, and no token's term
    depends on another batch row, so this split is exact).  dH, dk, dv and the
    forward outputs of sampled token windows against the oracle run on the
    window plus a 3-token halo on each side (enough for every dependency of the
    conv and its transpose); the weight gradients are also bitwise
    reproducible run to run."""
    M, T, d = 8, 8192, 7168
    inp = gateconv_inputs(M, T, d, 22, device=DEV, h_scale=10.0, v_std=0.1 ** 0.5)
    res = eg.gateconv_forward(inp["H"], inp["k"], inp["v"], inp["rms_w_h"], inp["rms_w_v"],
                              inp["conv_w"])
    args = (inp["dY"], inp["H"], inp["k"], inp["v"], inp["rms_w_h"], inp["rms_w_v"],
            inp["conv_w"], *res[1:])
    g = eg.gateconv_backward(*args)
    g2 = eg.gateconv_backward(*args)
    torch.cuda.synchronize()
    for x, y in zip(g[3:], g2[3:]):
        assert torch.equal(x, y)
    del g2
    weights = [f64(inp[k]) for k in ("rms_w_h", "rms_w_v", "conv_w")]
    ewh = np.zeros(d)
    ewv = np.zeros(d)
    ecw = np.zeros((4, d))
    for m in range(M):
        row = lambda t: f64(t[m:m + 1])
        eb = oracle.gateconv_bwd(row(inp["dY"]), row(inp["H"]), row(inp["k"]), row(inp["v"]),
                                 *weights, *(row(t) for t in res[1:]))
        ewh += eb[3]
        ewv += eb[4]
        ecw += eb[5]
        if m in (0, M - 1):
            # every element of dH, dk, dv of two whole batch rows
            for name, got, e in (("dH", g[0], eb[0]), ("dk", g[1], eb[1]), ("dv", g[2], eb[2])):
                check_bf16(name, bf16_bits(got[m:m + 1]), e, floor="all" if name != "dv" else "row")
        del eb
    check_f32_sum("drms_w_h", g[3].cpu().numpy(), ewh)
    check_f32_sum("drms_w_v", g[4].cpu().numpy(), ewv)
    check_f32_sum("dconv_w", g[5].cpu().numpy(), ecw)
    windows = [(0, 0, 24), (3, 1000, 1040), (7, T - 40, T), (5, 4095, 4130)]
    for m, a, b in windows:
        lo, hi = max(0, a - 3), min(T, b + 3)
        sl = lambda t: t[m:m + 1, lo:hi].contiguous()
        sub = {k: sl(inp[k]) for k in ("H", "k", "v", "dY")}
        sub.update({k: inp[k] for k in ("rms_w_h", "rms_w_v", "conv_w")})
        ef = oracle_fwd(sub)
        o0, o1 = a - lo, b - lo
        Y, vhat, alpha, rh, rk, rv = (t[m:m + 1, a:b] for t in res)
        check_bf16("Y", bf16_bits(Y), ef[0][:, o0:o1])
        check_bf16("vhat", bf16_bits(vhat), ef[1][:, o0:o1])
        for name, got, e in (("alpha", alpha, ef[2]), ("rrms_h", rh, ef[3]),
                             ("rrms_k", rk, ef[4]), ("rrms_v", rv, ef[5])):
            check_f32(name, got.cpu().numpy(), e[:, o0:o1])
        eb = oracle.gateconv_bwd(f64(sub["dY"]), f64(sub["H"]), f64(sub["k"]), f64(sub["v"]),
                                 f64(inp["rms_w_h"]), f64(inp["rms_w_v"]), f64(inp["conv_w"]),
                                 *(f64(sl(t)) for t in res[1:]))
        for name, got, e in (("dH", g[0], eb[0]), ("dk", g[1], eb[1]), ("dv", g[2], eb[2])):
            check_bf16(name, bf16_bits(got[m:m + 1, a:b]), e[:, o0:o1],
                       floor="all" if name != "dv" else "row")


def test_bwd_group_mode_graph_replays_match_eager():
    """The backward at d = 7168 runs as cooperative groups that exchange row
    sums through records in the workspace, which every call clears before its
    kernels.  Captured in a CUDA graph (the clearing with it) and replayed
    twice, it gives the eager call's outputs bit for bit; M = 32, T = 64 has
    more token ranges than groups, so groups take ranges in turn."""
    M, T, d = 32, 64, 7168
    inp = gateconv_inputs(M, T, d, 17, device=DEV)
    res = eg.gateconv_forward(inp["H"], inp["k"], inp["v"], inp["rms_w_h"], inp["rms_w_v"],
                              inp["conv_w"])
    args = (inp["dY"], inp["H"], inp["k"], inp["v"], inp["rms_w_h"], inp["rms_w_v"],
            inp["conv_w"], *res[1:])
    eager = eg.gateconv_backward(*args)
    outs = [torch.empty_like(t) for t in eager]
    ws = torch.empty(eg.engram_gateconv_bwd_workspace_size(M, T, d), device=DEV, dtype=torch.uint8)
    eg.engram_gateconv_bwd(*args, *outs, ws)   # set-up outside the capture
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            eg.engram_gateconv_bwd(*args, *outs, ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        for t in outs:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for x, y in zip(outs, eager):
            if x.dtype == torch.bfloat16:
                assert torch.equal(x.view(torch.int16), y.view(torch.int16))
            else:
                assert torch.equal(x, y)
    assert eg.engram_device_error() == 0


def test_bwd_group_geometry():
    """At d = 7168 the backward's CTAs of a token row work as cooperative
    groups of 7 (1024 columns each) on at least 140 SMs, where clusters of 8
    packed onto 120, and the groups take the M = 8, T = 8192 batch's token
    ranges in turn."""
    m8 = eg.engram_launch_info(3, 8, 8192, 7168)
    assert m8["cluster"] == 7 and m8["cluster"] * m8["resident"] >= 140
    assert m8["clusters"] > m8["resident"]


def test_launch_geometry():
    """C CTAs per row with ceil(d/1024) <= C <= 8 (forward: ceil(d/2048) <= C
    for its 512-thread CTAs); forward CTAs of at most 512 threads (4 columns
    each), every CTA's column slice non-empty; backward CTAs of 512 threads
    (two warp groups of 256 over a slice of at most 1024 columns); at least one
    cluster per row."""
    for (M, T, d) in ((4, 4096, 4096), (8, 8192, 7168), (2, 45, 1032), (1, 40, 8192), (1, 5, 64)):
        for op in (2, 3):
            info = eg.engram_launch_info(op, M, T, d)
            C = info["cluster"]
            assert -(-d // (2048 if op == 2 else 1024)) <= C <= 8
            if op == 2:
                assert info["threads"] % 32 == 0 and info["threads"] <= 512
                assert info["threads"] <= 256 or C == -(-d // 2048)
                assert 4 * info["threads"] * C >= d > 4 * info["threads"] * (C - 1)
            else:
                assert info["threads"] == 512
            assert info["clusters"] >= M and info["resident"] >= 1
    with pytest.raises(eg.EngramError):
        eg.engram_launch_info(2, 1, 4, 8200)
