"""GPU parity of the saved-state gate against the fp64 oracle (through the C ABI).

Workloads: bf16 X and KV ~N(0,1) (optionally scaled per token by
LogUniform(1e-2, 1e2)), fused weight 1 + 0.1 N(0,1), boolean masks, eps 1e-20
(cuDNN Frontend "Engram saved-state gate"; tile-kernels engram gate tests).
Tolerances are in tests/tolerance.py.
"""
import numpy as np
import pytest
import torch

import engram_memory_gating_gb300 as eg
import oracle
from engram_memory_gating_gb300.inputs import bf16_bits, gate_inputs
from tolerance import bf16_bits_to_f64, check_bf16, check_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 5120


def f64(t):
    if t.dtype == torch.bfloat16:
        return bf16_bits_to_f64(bf16_bits(t)).reshape(tuple(t.shape))
    return t.detach().double().cpu().numpy()


def to_dev(inp):
    return {k: v.to(DEV) for k, v in inp.items()}


def oracle_fwd(inp):
    mask = inp["mask"].cpu().numpy().astype(np.uint8)
    return oracle.gate_fwd(f64(inp["x"]), f64(inp["kv"]), f64(inp["weight"]), mask)


def check_fwd(out, saved, inp, exact_out, exact_saved):
    check_bf16("out", bf16_bits(out), exact_out)
    if saved is not None:
        s = saved.cpu().numpy().astype(np.float64)
        check_f32("saved.gate", s[..., 0], exact_saved[..., 0])
        check_f32("saved.dot", s[..., 1], exact_saved[..., 1])
        check_f32("saved.rstd_X", s[..., 2], exact_saved[..., 2])
        check_f32("saved.rstd_key", s[..., 3], exact_saved[..., 3])
    # false mask: out == X bit for bit
    m = ~inp["mask"].cpu()
    if m.any():
        assert torch.equal(out.cpu()[m].view(torch.int16), inp["x"].cpu()[m].view(torch.int16))


@pytest.fixture(autouse=True)
def no_device_error():
    yield
    assert eg.engram_device_error() == 0


@pytest.mark.parametrize("N,mask,seed", [(1, "all", 0), (3, "bern0.5", 1), (64, "all", 0),
                                         (77, "bern0.9", 2), (301, "bern0.5", 3)])
def test_fwd_parity_small(N, mask, seed):
    inp = gate_inputs(N, seed, mask=mask, with_grad=False)
    d = to_dev(inp)
    out, saved = eg.gate_forward(d["x"], d["kv"], d["weight"], d["mask"])
    exact_out, exact_saved = oracle_fwd(inp)
    check_fwd(out, saved, inp, exact_out, exact_saved)


def test_fwd_scale_sweep_and_no_mask_pointer():
    inp = gate_inputs(257, 5, mask="all", sigma="loguniform", with_grad=False)
    d = to_dev(inp)
    out = torch.empty_like(d["x"])
    saved = torch.empty((257, 4, 4), device=DEV, dtype=torch.float32)
    eg.engram_gate_fwd(d["x"], d["kv"], d["weight"], None, out, saved)
    exact_out, exact_saved = oracle_fwd(inp)
    check_fwd(out, saved, inp, exact_out, exact_saved)


def test_fwd_save_null_is_bit_identical():
    inp = to_dev(gate_inputs(130, 7, mask="bern0.5", with_grad=False))
    out1, _ = eg.gate_forward(inp["x"], inp["kv"], inp["weight"], inp["mask"], save=True)
    out2, s2 = eg.gate_forward(inp["x"], inp["kv"], inp["weight"], inp["mask"], save=False)
    assert s2 is None
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_fwd_all_masked_copies_x():
    inp = to_dev(gate_inputs(96, 8, mask="none", with_grad=False))
    out, saved = eg.gate_forward(inp["x"], inp["kv"], inp["weight"], inp["mask"])
    assert torch.equal(out.view(torch.int16), inp["x"].view(torch.int16))
    assert torch.all(saved[..., 0] == 0)


def test_fwd_edge_rows():
    # zero rows (rstd = 1/sqrt(eps), dot = 0, gate = 1/2), constant rows,
    # key equal to X, huge and tiny scales, a zero weight stream
    inp = gate_inputs(8, 9, mask="all", with_grad=False)
    x, kv, w = inp["x"].clone(), inp["kv"].clone(), inp["weight"].clone()
    x[0] = 0
    kv[1, :4 * D] = 0
    x[2] = 3.0
    kv[2, :4 * D] = -0.5
    for s in range(4):
        kv[3, s * D:(s + 1) * D] = x[3, s]
    x[4] *= 1e3
    kv[5] *= 1e-3
    w[1] = 0
    inp = {"x": x, "kv": kv, "weight": w, "mask": inp["mask"]}
    d = to_dev(inp)
    out, saved = eg.gate_forward(d["x"], d["kv"], d["weight"], d["mask"])
    exact_out, exact_saved = oracle_fwd(inp)
    check_fwd(out, saved, inp, exact_out, exact_saved)
    s = saved.cpu()
    assert torch.all(s[0, :, 1] == 0) and torch.all(s[0, :, 0] == 0.5)
    assert torch.all(s[:, 1, 0] == 0.5)


def test_fwd_graph_capture_matches_eager():
    inp = to_dev(gate_inputs(200, 10, mask="bern0.5", with_grad=False))
    out_e, saved_e = eg.gate_forward(inp["x"], inp["kv"], inp["weight"], inp["mask"])
    out = torch.empty_like(out_e)
    saved = torch.empty_like(saved_e)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            eg.engram_gate_fwd(inp["x"], inp["kv"], inp["weight"], inp["mask"], out, saved,
                               stream=s)
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out_e.view(torch.int16))
    assert torch.equal(saved, saved_e)


@pytest.mark.parametrize("N", [4096, 32768, 32769, 65536, 262144])
def test_fwd_full_size_sweep_graph(N):
    """Full-size forward sweep: per-token sigma ~ LogUniform(1e-2, 1e2), mask
    Bernoulli(0.5), CUDA-graph captured execute.  Sampled tokens are checked
    against the oracle; the masked identity is checked on every token.  The
    sizes give the persistent grid's quads whole and ragged last rounds of
    rows (32768, 32769) and rows far more than the grid (262144)."""
    inp = gate_inputs(N, 100 + N % 97, device=DEV, mask="bern0.5", sigma="loguniform",
                      with_grad=False)
    out = torch.empty_like(inp["x"])
    saved = torch.empty((N, 4, 4), device=DEV, dtype=torch.float32)
    eg.engram_gate_fwd(inp["x"], inp["kv"], inp["weight"], inp["mask"], out, saved)  # set-up
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            eg.engram_gate_fwd(inp["x"], inp["kv"], inp["weight"], inp["mask"], out, saved,
                               stream=s)
    torch.cuda.current_stream().wait_stream(s)
    out.fill_(0)
    saved.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    m = ~inp["mask"]
    assert torch.equal(out[m].view(torch.int16), inp["x"][m].view(torch.int16))
    assert torch.all(saved[m][:, :, 0] == 0)
    gen = torch.Generator().manual_seed(N)
    idx = torch.randperm(N, generator=gen)[:192]
    idx = torch.cat([idx, torch.tensor([0, 1, N - 2, N - 1])]).unique().to(DEV)
    sub = {"x": inp["x"][idx].cpu(), "kv": inp["kv"][idx].cpu(),
           "weight": inp["weight"].cpu(), "mask": inp["mask"][idx].cpu()}
    exact_out, exact_saved = oracle_fwd(sub)
    check_fwd(out[idx], saved[idx], sub, exact_out, exact_saved)


# ----------------------------------------------------------------- backward

def oracle_bwd(inp, saved64):
    return oracle.gate_bwd(f64(inp["x"]), f64(inp["kv"]), f64(inp["weight"]), saved64,
                           f64(inp["grad_out"]))


def check_bwd(gx, gkv, gw, exact):
    ex_gx, ex_gkv, ex_gw = exact
    N = gx.shape[0]
    check_bf16("grad_x", bf16_bits(gx), ex_gx)
    gkv_bits = bf16_bits(gkv).reshape(N, 5, D)
    check_bf16("grad_key", gkv_bits[:, :4], ex_gkv.reshape(N, 5, D)[:, :4])
    check_bf16("grad_v", gkv_bits[:, 4], ex_gkv.reshape(N, 5, D)[:, 4])
    check_f32("grad_weight", gw.cpu().numpy(), ex_gw)


@pytest.mark.parametrize("N,mask,seed", [(64, "all", 0), (128, "bern0.9", 1),
                                         (320, "bern0.5", 2)])
def test_bwd_parity_from_oracle_saved(N, mask, seed):
    inp = gate_inputs(N, seed, mask=mask)
    _, saved64 = oracle_fwd(inp)
    saved32 = torch.from_numpy(saved64.astype(np.float32))
    d = to_dev(inp)
    gx, gkv, gw = eg.gate_backward(d["x"], d["kv"], d["weight"], saved32.to(DEV), d["grad_out"])
    check_bwd(gx, gkv, gw, oracle_bwd(inp, saved32.double().numpy()))


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_fwd_bwd_full_batch_8192(seed):
    """N = 8192 (the cuDNN page's backward maximum), mask Bernoulli(0.9): the GPU forward's
    saved state feeds the GPU backward; every element is compared."""
    N = 8192
    inp = gate_inputs(N, seed, device=DEV, mask="bern0.9")
    out, saved = eg.gate_forward(inp["x"], inp["kv"], inp["weight"], inp["mask"])
    gx, gkv, gw = eg.gate_backward(inp["x"], inp["kv"], inp["weight"], saved, inp["grad_out"])
    torch.cuda.synchronize()
    host = {k: v.cpu() for k, v in inp.items()}
    exact_out, exact_saved = oracle_fwd(host)
    check_fwd(out, saved, host, exact_out, exact_saved)
    del exact_out
    exact = oracle_bwd(host, saved.double().cpu().numpy())
    check_bwd(gx, gkv, gw, exact)
    m = ~host["mask"]
    assert torch.equal(gx.cpu()[m].view(torch.int16), host["grad_out"][m].view(torch.int16))
    assert torch.all(gkv.cpu()[m][:, :4 * D].float() == 0)


@pytest.mark.parametrize("N,kernels", [(3776, 3), (3840, 2)])
def test_bwd_either_side_of_the_one_pass_threshold(N, kernels):
    """The backward takes the one-pass kernel from 42 clusters on (the
    workspace of N = 3840 holds 42: token ranges of 91 and 92 tokens) and the
    three kernels below (N = 3776 holds 41).  Both against the oracle, every
    element, mask Bernoulli(0.9)."""
    assert eg.engram_launch_info(1, N)["kernels"] == kernels
    inp = gate_inputs(N, 9, device=DEV, mask="bern0.9")
    _, saved = eg.gate_forward(inp["x"], inp["kv"], inp["weight"], inp["mask"])
    gx, gkv, gw = eg.gate_backward(inp["x"], inp["kv"], inp["weight"], saved, inp["grad_out"])
    torch.cuda.synchronize()
    host = {k: v.cpu() for k, v in inp.items()}
    check_bwd(gx, gkv, gw, oracle_bwd(host, saved.double().cpu().numpy()))


def test_bwd_long_batch():
    """N = 65,728 (1,027 blocks of 64: an odd count, so three-block token
    groups and a one-block last group), past the cuDNN page's 8192 cap.  The
    GPU forward's saved state feeds the backward; grad_x and grad_kv are
    compared element by element on a sample of tokens (the first and last
    block and 256 random tokens) against the oracle run on those tokens, and
    grad_weight against the oracle's sum over every token, formed as the fp64
    sum of the oracle's grad_weight over 4096-token chunks (grad_weight is a
    plain sum over tokens)."""
    N = 65728
    inp = gate_inputs(N, 5, device=DEV, mask="bern0.9")
    _, saved = eg.gate_forward(inp["x"], inp["kv"], inp["weight"], inp["mask"])
    gx, gkv, gw = eg.gate_backward(inp["x"], inp["kv"], inp["weight"], saved, inp["grad_out"])
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    pick = np.unique(np.concatenate([np.arange(64), np.arange(N - 64, N),
                                     rng.choice(N, 256, replace=False)]))
    idx = torch.from_numpy(pick).to(DEV)
    w64 = f64(inp["weight"])
    sub = {k: inp[k].index_select(0, idx).cpu() for k in ("x", "kv", "grad_out")}
    sv = saved.index_select(0, idx).double().cpu().numpy()
    ex, ekv, _ = oracle.gate_bwd(f64(sub["x"]), f64(sub["kv"]), w64, sv, f64(sub["grad_out"]))
    check_bf16("grad_x", bf16_bits(gx.index_select(0, idx)), ex)
    gkv_bits = bf16_bits(gkv.index_select(0, idx)).reshape(len(pick), 5, D)
    check_bf16("grad_key", gkv_bits[:, :4], ekv.reshape(len(pick), 5, D)[:, :4])
    check_bf16("grad_v", gkv_bits[:, 4], ekv.reshape(len(pick), 5, D)[:, 4])
    ew = np.zeros((4, D))
    for c0 in range(0, N, 4096):
        sl = slice(c0, min(N, c0 + 4096))
        _, _, ewc = oracle.gate_bwd(f64(inp["x"][sl]), f64(inp["kv"][sl]), w64,
                                    saved[sl].double().cpu().numpy(), f64(inp["grad_out"][sl]))
        ew += ewc
    check_f32("grad_weight", gw.cpu().numpy(), ew)


@pytest.mark.parametrize("N", [1024, 8192])
def test_bwd_is_deterministic(N):
    inp = gate_inputs(N, 4, device=DEV, mask="bern0.9")
    _, saved = eg.gate_forward(inp["x"], inp["kv"], inp["weight"], inp["mask"])
    r1 = eg.gate_backward(inp["x"], inp["kv"], inp["weight"], saved, inp["grad_out"])
    r2 = eg.gate_backward(inp["x"], inp["kv"], inp["weight"], saved, inp["grad_out"])
    for a, b in zip(r1, r2):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b)


@pytest.mark.parametrize("N", [256, 8192])
def test_bwd_graph_capture_matches_eager(N):
    """The backward captured in a CUDA graph and replayed twice (outputs
    cleared in between) gives the eager call's bits."""
    inp = to_dev(gate_inputs(N, 11, mask="bern0.5"))
    _, saved = eg.gate_forward(inp["x"], inp["kv"], inp["weight"], inp["mask"])
    ref = eg.gate_backward(inp["x"], inp["kv"], inp["weight"], saved, inp["grad_out"])
    gx, gkv, gw = torch.empty_like(ref[0]), torch.empty_like(ref[1]), torch.empty_like(ref[2])
    ws = torch.empty(eg.engram_gate_bwd_workspace_size(N), device=DEV, dtype=torch.uint8)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            eg.engram_gate_bwd(inp["x"], inp["kv"], inp["weight"], saved, inp["grad_out"], gx,
                               gkv, gw, ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        gx.zero_(), gkv.zero_(), gw.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(gx.view(torch.int16), ref[0].view(torch.int16))
        assert torch.equal(gkv.view(torch.int16), ref[1].view(torch.int16))
        assert torch.equal(gw, ref[2])


def test_launch_geometry():
    # forward: one warp per (token, stream) row, persistent CTAs
    fwd = eg.engram_launch_info(0, 65536)
    assert fwd["cluster"] == 1 and fwd["threads"] % 32 == 0 and fwd["clusters"] >= 1
    assert eg.engram_launch_info(0, 1)["clusters"] == 1
    # the grid is sized so that the last round of rows leaves under one CTA idle
    f8 = eg.engram_launch_info(0, 8192)
    warps, rows = 8 * f8["clusters"], 4 * 8192
    rpw = -(-rows // warps)
    assert warps * rpw - rows < 8 * rpw
    # backward.  Large N: the one-pass kernel (two kernels a call), clusters of
    # two CTAs (a column half each), each cluster's grad_weight pair (4 x 5120
    # fp32 hi and bf16 lo words) within the workspace, no more clusters than
    # run at once.  Otherwise: token rows split across column slices, at
    # most one group per two 64-token blocks, groups of at most 256 tokens
    # (their scalars are staged in shared memory).
    for N in (64, 128, 192, 3776, 3840, 4096, 8192, 11520, 65536, 65728, 1 << 20):
        b = eg.engram_launch_info(1, N)
        if b["kernels"] == 2:
            assert b["cluster"] == 2 and b["threads"] >= 640 and b["threads"] % 32 == 0
            assert 1 <= b["clusters"] <= b["resident"]
            assert b["clusters"] * 4 * 5120 * (4 + 2) <= eg.engram_gate_bwd_workspace_size(N)
        else:
            assert b["kernels"] == 3
            assert b["cluster"] >= 2 and 5120 % (8 * b["cluster"]) == 0
            groups = b["clusters"]
            assert -(-N // groups) <= 256
            assert N // 64 < 2 or 2 * groups <= N // 64
    # the full batch takes the one-pass kernel on this device, small batches not
    assert eg.engram_launch_info(1, 8192)["kernels"] == 2
    assert eg.engram_launch_info(1, 1024)["kernels"] == 3


def test_chained_steps_without_host_sync_match_synchronised_ones():
    """Three forward + backward steps in which each step's grad_x is the next
    step's X and its out the next step's grad_out, enqueued back to back on one
    stream with nothing between the calls.  The gate kernels are launched with
    programmatic stream serialisation, so each may be scheduled while its
    predecessor finishes; this checks that every kernel still reads only
    completed data, against the same chain with a device synchronisation after
    every call (no overlap at all).  The kernels are deterministic, so the two
    chains must agree bit for bit.  N = 3584 runs the three-kernel backward
    (its elementwise kernel in token mode), N = 8192 the one-pass backward."""
    for N in (256, 3584, 8192):
        _chain_check(N)


def _chain_check(N):
    inp = to_dev(gate_inputs(N, 21, mask="bern0.9"))
    ws = torch.empty(eg.engram_gate_bwd_workspace_size(N), device=DEV, dtype=torch.uint8)

    def run(sync):
        x, gout = inp["x"].clone(), inp["grad_out"].clone()
        results = []
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(3):
                out = torch.empty_like(x)
                saved = torch.empty((N, 4, 4), device=DEV)
                gx, gkv = torch.empty_like(x), torch.empty_like(inp["kv"])
                gw = torch.empty_like(inp["weight"])
                eg.engram_gate_fwd(x, inp["kv"], inp["weight"], inp["mask"], out, saved, stream=s)
                if sync:
                    torch.cuda.synchronize()
                eg.engram_gate_bwd(x, inp["kv"], inp["weight"], saved, gout, gx, gkv, gw, ws, stream=s)
                if sync:
                    torch.cuda.synchronize()
                results.append((out, saved, gx, gkv, gw))
                x, gout = gx, out
        torch.cuda.synchronize()
        return results

    want = run(True)
    got = run(False)
    for step_w, step_g in zip(want, got):
        for a, b in zip(step_w, step_g):
            if a.dtype == torch.bfloat16:
                assert torch.equal(a.view(torch.int16), b.view(torch.int16))
            else:
                assert torch.equal(a, b)
