"""GPU parity of the GateConv decode step (TileOPs "Engram Operators", Decode
section, EngramDecodeFwdOp) against the fp64 oracle, through the C ABI.
Inputs: e, h, cache ~N(0,1) bf16, W_K, W_V ~N(0, 1/d_mem) bf16, norm weights
1 + 0.1 N(0,1), conv_w ~N(0, 0.25)."""
import numpy as np
import pytest
import torch

import engram_memory_gating_gb300 as eg
import oracle
from engram_memory_gating_gb300.inputs import bf16_bits, decode_inputs
from tolerance import bf16_bits_to_f64, check_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def no_device_error():
    yield
    assert eg.engram_device_error() == 0


def f64(t):
    if t.dtype == torch.bfloat16:
        return bf16_bits_to_f64(bf16_bits(t)).reshape(tuple(t.shape))
    return t.detach().double().cpu().numpy()


def step(inp, max_len, dil):
    d = {k: v.cuda() for k, v in inp.items()}
    y, ns = eg.decode_forward(d["e"], d["h"], d["conv_state"], d["W_K"], d["W_V"], d["rms_w_h"],
                              d["rms_w_v"], d["conv_w"], max_len, dil)
    torch.cuda.synchronize()
    return y, ns


def check_step(inp, y, ns, max_len, dil):
    ey, ens = oracle.decode_fwd(*(f64(inp[k]) for k in ("e", "h", "conv_state", "W_K", "W_V", "rms_w_h",
                                                        "rms_w_v", "conv_w")), max_len=max_len, dilation=dil)
    check_bf16("y", bf16_bits(y), ey)
    got = f64(ns)
    # shifted rows are copies (bit-exact); the new row is this token's u, rounded once
    assert np.array_equal(got[:, :-1], ens[:, :-1])
    check_bf16("new row", bf16_bits(ns[:, -1]), ens[:, -1])


@pytest.mark.parametrize("B,dmem,d,L,max_len,w,dil", [
    (1, 64, 64, 0, 4, 4, 1), (3, 256, 512, 5, 8, 4, 2), (8, 1024, 4096, 9, 12, 4, 3),
    (17, 512, 1024, 12, 12, 4, 3), (2, 1000, 2048, 16, 16, 3, 5), (4, 8192, 256, 3, 4, 4, 1),
    (5, 96, 128, 2, 40, 7, 6)])
def test_decode_parity(B, dmem, d, L, max_len, w, dil):
    inp = decode_inputs(B, dmem, d, L, w, seed=B * 7 + L)
    y, ns = step(inp, max_len, dil)
    check_step(inp, y, ns, max_len, dil)


def test_decode_chain_of_steps():
    """Eight steps, each fed the previous step's new cache (empty at first)."""
    B, dmem, d, max_len, w, dil = 2, 256, 512, 9, 4, 3
    inp = decode_inputs(B, dmem, d, 0, w, seed=5)
    g = torch.Generator().manual_seed(6)
    for t in range(8):
        inp["e"] = torch.randn((B, dmem), generator=g).to(torch.bfloat16)
        inp["h"] = torch.randn((B, d), generator=g).to(torch.bfloat16)
        y, ns = step(inp, max_len, dil)
        check_step(inp, y, ns, max_len, dil)
        inp["conv_state"] = ns.cpu()


def test_decode_is_deterministic_and_graph_capturable():
    B, dmem, d, L, max_len, w, dil = 8, 1024, 4096, 12, 16, 4, 3
    inp = {k: v.cuda() for k, v in decode_inputs(B, dmem, d, L, w, seed=9).items()}
    y, ns = torch.empty_like(inp["h"]), torch.empty((B, max_len, d), device="cuda", dtype=torch.bfloat16)
    ws = torch.empty(eg.engram_decode_workspace_size(B, dmem, d), device="cuda", dtype=torch.uint8)
    args = (inp["e"], inp["h"], inp["conv_state"], inp["W_K"], inp["W_V"], inp["rms_w_h"], inp["rms_w_v"],
            inp["conv_w"], y, ns, ws, dil)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        eg.engram_decode_fwd(*args, stream=s)
        torch.cuda.synchronize()
        ref = (y.clone(), ns.clone())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            eg.engram_decode_fwd(*args, stream=s)
    y.zero_()
    ns.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), ref[0].view(torch.int16))
    assert torch.equal(ns.view(torch.int16), ref[1].view(torch.int16))


def test_decode_chain_on_device_without_host_sync():
    """Eight decode steps on one stream, each reading the cache the previous
    step wrote (two buffers used in turn) and sharing one workspace, enqueued
    back to back.  Each step's projection is launched with programmatic stream
    serialisation behind the previous step's row kernel, so it may be scheduled
    early; this checks that it waits for that kernel before it reads the cache
    or overwrites the workspace, against the same chain synchronised after
    every step (bit-exact: the kernels are deterministic)."""
    B, dmem, d, max_len, w, dil = 4, 512, 1024, 8, 4, 3
    inp = {k: v.cuda() for k, v in decode_inputs(B, dmem, d, max_len, w, seed=11).items()}
    g = torch.Generator().manual_seed(12)
    es = [torch.randn((B, dmem), generator=g).to(torch.bfloat16).cuda() for _ in range(8)]
    hs = [torch.randn((B, d), generator=g).to(torch.bfloat16).cuda() for _ in range(8)]
    ws = torch.empty(eg.engram_decode_workspace_size(B, dmem, d), device="cuda", dtype=torch.uint8)

    def run(sync):
        caches = [inp["conv_state"].clone(), torch.empty((B, max_len, d), device="cuda", dtype=torch.bfloat16)]
        ys = []
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for t in range(8):
                y = torch.empty((B, d), device="cuda", dtype=torch.bfloat16)
                eg.engram_decode_fwd(es[t], hs[t], caches[t & 1], inp["W_K"], inp["W_V"], inp["rms_w_h"],
                                     inp["rms_w_v"], inp["conv_w"], y, caches[(t + 1) & 1], ws, dil, stream=s)
                if sync:
                    torch.cuda.synchronize()
                ys.append(y)
        torch.cuda.synchronize()
        return ys, caches[0]

    want_y, want_cache = run(True)
    got_y, got_cache = run(False)
    for a, b in zip(want_y, got_y):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(want_cache.view(torch.int16), got_cache.view(torch.int16))
