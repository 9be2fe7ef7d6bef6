"""The saved-state gate backward for callers that cannot allocate.

engram_gate_bwd_noalloc runs the same backward as engram_gate_bwd, with its
workspace taken from a fixed array inside the library instead of a buffer the
caller allocates (for callers inside a framework that owns all device memory,
or on a fixed memory budget).  Checked through the C
ABI: two calls in a row give the same bits as the workspace entry point (the
same deterministic kernels run, only the workspace's address differs, so any
difference would mean a misplaced workspace slot), they change the device's
free memory by nothing, and a size beyond the array's limit is refused before
any work is enqueued.
This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import engram_memory_gating_gb300 as eg
from engram_memory_gating_gb300.inputs import gate_inputs

MAX_N = 2048


@pytest.mark.gpu
def test_gate_bwd_noalloc_matches_workspace_entry_point_twice():
    lib = eg.load()
    for N, seed in ((MAX_N, 41), (576, 42)):
        inp = gate_inputs(N, seed, device="cuda", mask="bern0.9")
        _, saved = eg.gate_forward(inp["x"], inp["kv"], inp["weight"], inp["mask"])
        ref = eg.gate_backward(inp["x"], inp["kv"], inp["weight"], saved, inp["grad_out"])
        torch.cuda.synchronize()
        free_before = None
        for call in range(2):
            gx, gkv, gw = (torch.full_like(ref[0], 7.0), torch.full_like(ref[1], 7.0),
                           torch.full_like(ref[2], 7.0))
            torch.cuda.synchronize()
            if call == 1:
                free_before = torch.cuda.mem_get_info()[0]
            st = lib.engram_gate_bwd_noalloc(
                ctypes.c_void_p(inp["x"].data_ptr()), ctypes.c_void_p(inp["kv"].data_ptr()),
                ctypes.c_void_p(inp["weight"].data_ptr()), ctypes.c_void_p(saved.data_ptr()),
                ctypes.c_void_p(inp["grad_out"].data_ptr()), ctypes.c_void_p(gx.data_ptr()),
                ctypes.c_void_p(gkv.data_ptr()), ctypes.c_void_p(gw.data_ptr()), N,
                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
            assert st == 0
            torch.cuda.synchronize()
            if call == 1:
                assert torch.cuda.mem_get_info()[0] == free_before
            assert torch.equal(gx.view(torch.int16), ref[0].view(torch.int16))
            assert torch.equal(gkv.view(torch.int16), ref[1].view(torch.int16))
            assert torch.equal(gw.view(torch.int32), ref[2].view(torch.int32))
    assert eg.engram_device_error() == 0


@pytest.mark.gpu
def test_gate_bwd_noalloc_refuses_sizes_beyond_its_array():
    lib = eg.load()
    N = MAX_N + 64
    inp = gate_inputs(64, 43, device="cuda")
    # sizes are checked before any pointer is used: nothing is enqueued
    st = lib.engram_gate_bwd_noalloc(*(ctypes.c_void_p(inp["x"].data_ptr()),) * 8, N, None)
    assert st == 3
    assert lib.engram_gate_bwd_noalloc(*(ctypes.c_void_p(inp["x"].data_ptr()),) * 8, 100,
                                       None) == 3
