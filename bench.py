#!/usr/bin/env python
"""Benchmark of the Engram gate on GB300 through the C ABI (libengram.so).

Workload (one step): saved-state gate forward + backward, N = 8192 tokens
(the backward's maximum), S = 4 streams, d = 5120, bf16 X/KV ~N(0,1), fused
fp32 weight 1 + 0.1 N(0,1), mask ~Bernoulli(0.9), grad_out ~N(0,1), eps
1e-20, seed 1.  Inputs stay resident in HBM; one step reads and writes
1.85 GB, larger than the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  `value` is tokens/s over all ranks (replicas:
every rank runs the full workload on its own GPU, no collective on the data
path).  `--impl reference` times the fp64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

N_TOK, S, D = 8192, 4, 5120
FWD_BYTES_PER_TOKEN = 4 * D * 2 + 5 * D * 2 + 1 + 4 * D * 2 + 64      # 133,185
BWD_BYTES_PER_TOKEN = 4 * D * 2 + 5 * D * 2 + 64 + 4 * D * 2 + 4 * D * 2 + 5 * D * 2  # 225,344
FWD_FIXED = 4 * D * 4                 # weight
BWD_FIXED = 2 * 4 * D * 4             # weight + grad_weight
METRIC = "Engram gate fwd+bwd tokens/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
NOMINAL_GBS = 8000.0  # GB300's nominal HBM3e bandwidth (~8 TB/s), the second denominator
WORKLOAD = ("saved-state gate fwd+bwd, N=8192, S=4, d=5120, bf16 X/KV ~N(0,1), "
            "weight 1+0.1N(0,1), mask~Bernoulli(0.9), grad_out ~N(0,1), eps 1e-20, seed 1")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def scaled_traffic(profile_md, sources, factor):
    """A committed summary's per-launch DRAM bytes for a smaller case of the
    same kernels, scaled to this launch by the units processed (the kernels'
    traffic grows in proportion to tokens or rows)."""
    t = profile_traffic(profile_md, sources)
    return None if t is None else int(round(t * factor))


def profile_traffic(profile_md, sources):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current kernel sources (the kernel's file and the headers it
    includes); else None."""
    path = os.path.join(ROOT, "profiles", profile_md)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not m or not t or m.group(1) != source_hash(sources):
        return None
    return int(t.group(1))


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append(parts)
            except ValueError:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        smax = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


def max_over_ranks(x: float, dist, device) -> float:
    """The largest x over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms * 1e-3)


def time_region(torch, fn, reps, stream):
    """Mean ms of fn() over reps, CUDA events on `stream`; fn's work (graph
    replays included) is issued on that same stream."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            fn()
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / reps


def graph_of(torch, fn, stream):
    fn()  # one-time per-device set-up happens outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            fn()
    torch.cuda.synchronize()
    return g


def op_entry(ms, nbytes, peak):
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 5), "algorithmic_bytes": int(nbytes), "GB_s": round(gbs, 1),
            "frac_of_measured_peak": round(gbs / peak, 4),
            "frac_of_nominal_peak": round(gbs / NOMINAL_GBS, 4)}


def extra_ops(torch, eg, inputs_mod, stream, peak):
    """Each hot-path op at its own configuration, CUDA-graph replayed, inputs
    larger than L2 (no flush needed)."""
    ops = {}
    s = stream
    # the smallest configuration: forward + backward of N = 64 tokens (mask all
    # true), one CUDA graph of both calls, latency per call pair
    N = 64
    inp = inputs_mod.gate_inputs(N, 0, device="cuda", mask="all")
    out = torch.empty_like(inp["x"])
    saved = torch.empty((N, 4, 4), device="cuda", dtype=torch.float32)
    gx, gkv, gw = torch.empty_like(inp["x"]), torch.empty_like(inp["kv"]), torch.empty_like(inp["weight"])
    ws = torch.empty(eg.engram_gate_bwd_workspace_size(N), device="cuda", dtype=torch.uint8)

    def small_step():
        eg.engram_gate_fwd(inp["x"], inp["kv"], inp["weight"], inp["mask"], out, saved, stream=s)
        eg.engram_gate_bwd(inp["x"], inp["kv"], inp["weight"], saved, inp["grad_out"], gx, gkv, gw, ws, stream=s)

    g = graph_of(torch, small_step, s)
    time_region(torch, g.replay, 20, s)
    ms = time_region(torch, g.replay, 200, s)
    ops["gate_step_N64"] = op_entry(ms, N * (FWD_BYTES_PER_TOKEN + BWD_BYTES_PER_TOKEN) + FWD_FIXED + BWD_FIXED, peak)
    ops["gate_step_N64"]["us"] = round(1000 * ms, 2)
    del inp, out, saved, gx, gkv, gw, ws, g
    # forward sweep, N in {4096, 65536, 262144}, per-token sigma ~ LogUniform(1e-2, 1e2),
    # mask Bernoulli(0.5), CUDA-graph replays
    for N in (4096, 65536, 262144):
        inp = inputs_mod.gate_inputs(N, 103, device="cuda", mask="bern0.5", sigma="loguniform",
                                     with_grad=False)
        out = torch.empty_like(inp["x"])
        saved = torch.empty((N, 4, 4), device="cuda", dtype=torch.float32)
        fn = lambda: eg.engram_gate_fwd(inp["x"], inp["kv"], inp["weight"], inp["mask"], out, saved,
                                        stream=s)
        g = graph_of(torch, fn, s)
        time_region(torch, g.replay, 3, s)
        ms = time_region(torch, g.replay, 10 if N > 4096 else 40, s)
        ops[f"gate_fwd_N{N}"] = op_entry(ms, N * FWD_BYTES_PER_TOKEN + FWD_FIXED, peak)
        if N != 262144:
            del inp, out, saved, g
            torch.cuda.empty_cache()
    csrc = "engram_memory_gating_gb300/csrc/"
    hdrs = [csrc + "common.cuh", csrc + "engram_internal.h"]
    ops["gate_fwd_N262144"]["traffic"] = scaled_traffic(
        "gate_fwd_n36864.md", [csrc + "gate_fwd.cu"] + hdrs, N / 36864)
    ops["gate_fwd_N262144"]["traffic_from"] = "N = 36,864 capture of the same kernel and input recipe, x 262144/36864"
    del inp, out, saved, g
    torch.cuda.empty_cache()
    # backward past the 8192-token cap: N = 65536, mask Bernoulli(0.9)
    N = 65536
    inp = inputs_mod.gate_inputs(N, 104, device="cuda", mask="bern0.9")
    out = torch.empty_like(inp["x"])
    saved = torch.empty((N, 4, 4), device="cuda", dtype=torch.float32)
    eg.engram_gate_fwd(inp["x"], inp["kv"], inp["weight"], inp["mask"], out, saved, stream=s)
    del out
    gx, gkv, gw = torch.empty_like(inp["x"]), torch.empty_like(inp["kv"]), torch.empty_like(inp["weight"])
    ws = torch.empty(eg.engram_gate_bwd_workspace_size(N), device="cuda", dtype=torch.uint8)
    fn = lambda: eg.engram_gate_bwd(inp["x"], inp["kv"], inp["weight"], saved, inp["grad_out"], gx, gkv,
                                    gw, ws, stream=s)
    g = graph_of(torch, fn, s)
    time_region(torch, g.replay, 3, s)
    ms = time_region(torch, g.replay, 10, s)
    ops["gate_bwd_N65536"] = op_entry(ms, N * BWD_BYTES_PER_TOKEN + BWD_FIXED, peak)
    ops["gate_bwd_N65536"]["traffic"] = scaled_traffic(
        "gate_bwd_n16384.md", [csrc + "gate_bwd.cu", csrc + "gate_bwd_fused.cu"] + hdrs, N / 16384)
    ops["gate_bwd_N65536"]["traffic_from"] = "N = 16,384 capture of the same kernels and input recipe, x 4"
    del inp, saved, gx, gkv, gw, ws, g
    torch.cuda.empty_cache()
    # separate-tensor gate (tile-kernels layout), N = 8192, H = 4096
    N, H = 8192, 4096
    inp = inputs_mod.gate_inputs(N, 105, device="cuda", d=H)
    k = inp["kv"][:, :4 * H].reshape(N, 4, H).contiguous()
    v = inp["kv"][:, 4 * H:].contiguous()
    del inp["kv"]
    out = torch.empty_like(inp["x"])
    sv = [torch.empty((N, 4), device="cuda") for _ in range(4)]
    gx, gk, gv = torch.empty_like(inp["x"]), torch.empty_like(k), torch.empty_like(v)
    gwp = torch.empty(((N + 63) // 64, 4, H), device="cuda")
    ws = torch.empty(eg.engram_gate_sep_bwd_workspace_size(N), device="cuda", dtype=torch.uint8)
    f = lambda: eg.engram_gate_sep_fwd(inp["x"], k, v, inp["weight"], out, *sv, stream=s)
    b = lambda: eg.engram_gate_sep_bwd(inp["grad_out"], inp["x"], k, v, inp["weight"], *sv, gx, gk, gv,
                                       gwp, ws, stream=s)
    gf, gb = graph_of(torch, f, s), graph_of(torch, b, s)
    time_region(torch, lambda: (gf.replay(), gb.replay()), 3, s)
    ops["gate_sep_fwd_N8192_H4096"] = op_entry(time_region(torch, gf.replay, 10, s),
                                               N * (26 * H + 64) + 16 * H, peak)
    ops["gate_sep_bwd_N8192_H4096"] = op_entry(time_region(torch, gb.replay, 10, s),
                                               N * (44 * H + 64) + 16 * H + (N // 64) * 16 * H, peak)
    ops["gate_sep_fwd_N8192_H4096"]["traffic"] = profile_traffic(
        "gate_sep_fwd_n8192_h4096.md", [csrc + "gate_fwd.cu"] + hdrs)
    ops["gate_sep_bwd_N8192_H4096"]["traffic"] = profile_traffic(
        "gate_sep_bwd_n8192_h4096.md", [csrc + "gate_bwd.cu"] + hdrs)
    del inp, k, v, out, sv, gx, gk, gv, gwp, ws, gf, gb
    torch.cuda.empty_cache()
    # GateConv decode step, B = 8, d_mem = 1024, d = 4096, full cache of 16, w = 4, dilation 3,
    # with the L2 flushed before every step (the weights would otherwise stay resident).
    # Device time: one graph of 20 x (flush, step) minus one of 20 flushes, so that the
    # graph's own launch latency is spread over 20 steps; the latency of a single replay
    # (event to event around one graph of one step, launch included) is reported beside it.
    B, dm, d, L, w, dil = 8, 1024, 4096, 16, 4, 3
    di = inputs_mod.decode_inputs(B, dm, d, L, w, seed=107, device="cuda")
    y = torch.empty_like(di["h"])
    ns = torch.empty((B, L, d), device="cuda", dtype=torch.bfloat16)
    ws = torch.empty(eg.engram_decode_workspace_size(B, dm, d), device="cuda", dtype=torch.uint8)
    f = lambda: eg.engram_decode_fwd(di["e"], di["h"], di["conv_state"], di["W_K"], di["W_V"],
                                     di["rms_w_h"], di["rms_w_v"], di["conv_w"], y, ns, ws, dil, stream=s)
    flush = torch.ones(64 << 20, device="cuda", dtype=torch.float32)  # 256 MB, read: L2 keeps clean lines
    reps = 20

    def flushed_steps(with_step):
        def body():
            for _ in range(reps):
                flush.sum()
                if with_step:
                    f()
        return graph_of(torch, body, s)

    g_steps, g_flush = flushed_steps(True), flushed_steps(False)
    t_steps = sorted(time_region(torch, g_steps.replay, 1, s) for _ in range(5))[2]
    t_flush = sorted(time_region(torch, g_flush.replay, 1, s) for _ in range(5))[2]
    dev_ms = max(t_steps - t_flush, 0.0) / reps
    gd = graph_of(torch, f, s)
    total = 0.0
    with torch.cuda.stream(s):
        for r in range(reps + 3):
            flush.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            gd.replay()
            e1.record(s)
            e1.synchronize()
            if r >= 3:
                total += e0.elapsed_time(e1)
    nbytes = 2 * dm * d * 2 + B * dm * 2 + B * d * 2 + B * L * d * 2 + d * 4 * (2 + w) + B * d * 2 + B * L * d * 2
    ops["decode_B8_dmem1024_d4096"] = op_entry(dev_ms, nbytes, peak)
    ops["decode_B8_dmem1024_d4096"]["us"] = round(1000 * dev_ms, 2)
    ops["decode_B8_dmem1024_d4096"]["us_single_replay"] = round(1000 * total / reps, 2)
    csrc = "engram_memory_gating_gb300/csrc/"
    ops["decode_B8_dmem1024_d4096"]["traffic"] = profile_traffic(
        "decode_b8_dmem1024_d4096.md", [csrc + "decode.cu", csrc + "common.cuh", csrc + "engram_internal.h"])
    del di, y, ns, ws, gd, g_steps, g_flush, flush
    torch.cuda.empty_cache()
    # GateConv, two configurations
    for (M, T, d, hs, vs, name) in ((4, 4096, 4096, 1.0, 1.0, "gateconv_M4_T4096_d4096"),
                                    (8, 8192, 7168, 10.0, 0.1 ** 0.5, "gateconv_M8_T8192_d7168")):
        ci = inputs_mod.gateconv_inputs(M, T, d, 31, device="cuda", h_scale=hs, v_std=vs)
        res = [torch.empty_like(ci["H"]), torch.empty_like(ci["H"])] + \
            [torch.empty((M, T), device="cuda", dtype=torch.float32) for _ in range(4)]
        grads = [torch.empty_like(ci["H"]) for _ in range(3)] + \
            [torch.empty(d, device="cuda"), torch.empty(d, device="cuda"),
             torch.empty((4, d), device="cuda")]
        ws = torch.empty(eg.engram_gateconv_bwd_workspace_size(M, T, d), device="cuda",
                         dtype=torch.uint8)
        f = lambda: eg.engram_gateconv_fwd(ci["H"], ci["k"], ci["v"], ci["rms_w_h"],
                                           ci["rms_w_v"], ci["conv_w"], *res, stream=s)
        b = lambda: eg.engram_gateconv_bwd(ci["dY"], ci["H"], ci["k"], ci["v"], ci["rms_w_h"],
                                           ci["rms_w_v"], ci["conv_w"], *res[1:], *grads, ws,
                                           stream=s)
        gf, gb = graph_of(torch, f, s), graph_of(torch, b, s)
        time_region(torch, lambda: (gf.replay(), gb.replay()), 3, s)
        tok = M * T
        ops[name + "_fwd"] = op_entry(time_region(torch, gf.replay, 10, s),
                                      tok * (10 * d + 16) + 24 * d, peak)
        ops[name + "_bwd"] = op_entry(time_region(torch, gb.replay, 10, s),
                                      tok * (16 * d + 16) + 48 * d, peak)
        # DRAM bytes per launch from the committed ncu summaries (M8: the
        # M = 1 capture of the same kernels, scaled by the rows)
        csrc = "engram_memory_gating_gb300/csrc/"
        common = [csrc + "gateconv_xch.cuh", csrc + "common.cuh", csrc + "engram_internal.h"]
        tag, factor = ("m4_t4096_d4096", 1.0) if M == 4 else ("m1_t8192_d7168", float(M))
        ops[name + "_fwd"]["traffic"] = scaled_traffic(
            f"gateconv_fwd_{tag}.md", [csrc + "gateconv_fwd.cu"] + common, factor)
        ops[name + "_bwd"]["traffic"] = scaled_traffic(
            f"gateconv_bwd_{tag}.md", [csrc + "gateconv_bwd.cu"] + common, factor)
        if M != 4:
            ops[name + "_fwd"]["traffic_from"] = ops[name + "_bwd"]["traffic_from"] = \
                f"M = 1 capture of the same kernels, x {M}"
        del ci, res, grads, ws, gf, gb
        torch.cuda.empty_cache()
    return ops


def cpu_baseline(seconds=10.0):
    """The fp64 oracle (as it stands) on the N=8192 workload, fwd + bwd,
    repeated until about `seconds` of CPU work have run."""
    import oracle
    from engram_memory_gating_gb300.inputs import gate_inputs
    oracle.build()
    inp = gate_inputs(N_TOK, 1, mask="bern0.9")
    x, kv, w, m, g = f64_inputs(inp)
    reps, el = 0, 0.0
    while el < seconds and reps < 200:
        t0 = time.perf_counter()
        _, saved = oracle.gate_fwd(x, kv, w, m)
        oracle.gate_bwd(x, kv, w, saved, g)
        el += time.perf_counter() - t0
        reps += 1
    return {"value": round(reps * N_TOK / el, 2), "unit": "tokens/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{reps} x the full N=8192 workload (fwd+bwd, fp64), {el:.1f} s"}


def f64_inputs(inp):
    """bf16 / fp32 host tensors -> exact float64 arrays (plus the mask bytes)."""
    f = lambda t: t.double().numpy()
    return (f(inp["x"]), f(inp["kv"]), f(inp["weight"]),
            inp["mask"].numpy().astype("uint8"), f(inp["grad_out"]))


def run_config(world):
    """The workload description both arms print (identical, so that the two
    lines can be compared key for key)."""
    return {"workload": WORKLOAD, "N": N_TOK, "S": S, "d": D,
            "l2": "inputs larger than L2 (1.85 GB read+written per step); no flush",
            "parallelism": f"replicas x{world}"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    from engram_memory_gating_gb300.inputs import gate_inputs
    oracle.build()
    # per-token cost from a 64-token probe; the full-size arrays no longer fit
    # in the host caches and run about 2.7x slower per token, hence the margin
    inp = gate_inputs(64, 1, mask="bern0.9")
    x, kv, w, m, g = f64_inputs(inp)
    t0 = time.perf_counter()
    _, saved = oracle.gate_fwd(x, kv, w, m)
    oracle.gate_bwd(x, kv, w, saved, g)
    per_tok = 3.0 * (time.perf_counter() - t0) / 64
    budget = 150.0 / max(1, args.steps + args.warmup)
    n = int(max(64, min(N_TOK, budget / max(per_tok, 1e-9))))
    n = n // 64 * 64
    if n > 64:
        x, kv, w, m, g = f64_inputs(gate_inputs(n, 1, mask="bern0.9"))

    def step(n):
        _, saved = oracle.gate_fwd(x[:n], kv[:n], w, m[:n])
        oracle.gate_bwd(x[:n], kv[:n], w, saved, g[:n])

    for _ in range(args.warmup):
        step(n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(n)
    el = time.perf_counter() - t0
    value = args.steps * n / el
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": run_config(world),
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s",
                             "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{n} tokens of the workload per step"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


GC_WORKLOADS = {"m4": (4, 4096, 4096, 1.0, 1.0), "m8": (8, 8192, 7168, 10.0, 0.1 ** 0.5),
                "m1": (1, 8192, 7168, 10.0, 0.1 ** 0.5)}


def run_single_op(args):
    """One entry point alone, `warmup` + `steps` plain calls on one stream, for
    profiler captures: the gate at --n tokens (default the step's 8192) with the
    step's input recipe, or the forward sweep's with --sweep-inputs; the
    separate-tensor gate at --n tokens and hidden size --h (default 4096; the
    quad kernel for 4096 <= H <= 5120, one warp per row otherwise); GateConv at --gc-workload
    (m4: M=4, T=4096, d=4096; m8: M=8, T=8192, d=7168; m1: M=1, T=8192,
    d=7168); decode at B = 8, d_mem = 1024, d = 4096, a full cache of 16, w = 4,
    dilation 3 (back to back, weights L2-warm).  Prints the mean event-timed
    call.  Launches per call: gate_fwd 1, gate_bwd 2 (the one-pass kernel and
    the merge) or 3 (coefficients, elementwise, merge), gate_sep_fwd 1,
    gate_sep_bwd 2, gateconv_fwd 1, gateconv_bwd 4, decode 2."""
    import torch
    import engram_memory_gating_gb300 as eg
    from engram_memory_gating_gb300 import inputs as inputs_mod
    s = torch.cuda.Stream()
    if args.op.startswith("gate_sep_"):
        N, H = args.n, args.h
        inp = inputs_mod.gate_inputs(N, 105, device="cuda", d=H)
        k = inp["kv"][:, :4 * H].reshape(N, 4, H).contiguous()
        v = inp["kv"][:, 4 * H:].contiguous()
        del inp["kv"]
        out = torch.empty_like(inp["x"])
        sv = [torch.empty((N, 4), device="cuda") for _ in range(4)]
        eg.engram_gate_sep_fwd(inp["x"], k, v, inp["weight"], out, *sv, stream=s)
        gx, gk, gv = torch.empty_like(inp["x"]), torch.empty_like(k), torch.empty_like(v)
        gwp = torch.empty(((N + 63) // 64, 4, H), device="cuda")
        ws = torch.empty(eg.engram_gate_sep_bwd_workspace_size(N), device="cuda", dtype=torch.uint8)
        if args.op == "gate_sep_fwd":
            fn = lambda: eg.engram_gate_sep_fwd(inp["x"], k, v, inp["weight"], out, *sv, stream=s)
        else:
            fn = lambda: eg.engram_gate_sep_bwd(inp["grad_out"], inp["x"], k, v, inp["weight"], *sv, gx, gk,
                                                gv, gwp, ws, stream=s)
    elif args.op.startswith("gate_"):
        N = args.n
        if args.sweep_inputs:
            inp = inputs_mod.gate_inputs(N, 103, device="cuda", mask="bern0.5", sigma="loguniform")
        else:
            inp = inputs_mod.gate_inputs(N, 1, device="cuda", mask="bern0.9")
        out, saved = eg.gate_forward(inp["x"], inp["kv"], inp["weight"], inp["mask"])
        gx, gkv, gw = (torch.empty_like(inp["x"]), torch.empty_like(inp["kv"]),
                       torch.empty_like(inp["weight"]))
        ws = torch.empty(eg.engram_gate_bwd_workspace_size(N), device="cuda", dtype=torch.uint8)
        if args.op == "gate_fwd":
            fn = lambda: eg.engram_gate_fwd(inp["x"], inp["kv"], inp["weight"], inp["mask"], out,
                                            saved, stream=s)
        else:
            fn = lambda: eg.engram_gate_bwd(inp["x"], inp["kv"], inp["weight"], saved,
                                            inp["grad_out"], gx, gkv, gw, ws, stream=s)
    elif args.op == "decode":
        B, dm, d, L, w, dil = 8, 1024, 4096, 16, 4, 3
        di = inputs_mod.decode_inputs(B, dm, d, L, w, seed=107, device="cuda")
        y = torch.empty_like(di["h"])
        ns = torch.empty((B, L, d), device="cuda", dtype=torch.bfloat16)
        ws = torch.empty(eg.engram_decode_workspace_size(B, dm, d), device="cuda", dtype=torch.uint8)
        fn = lambda: eg.engram_decode_fwd(di["e"], di["h"], di["conv_state"], di["W_K"], di["W_V"],
                                          di["rms_w_h"], di["rms_w_v"], di["conv_w"], y, ns, ws, dil, stream=s)
    else:
        M, T, d, hs, vs = GC_WORKLOADS[args.gc_workload]
        ci = inputs_mod.gateconv_inputs(M, T, d, 31, device="cuda", h_scale=hs, v_std=vs)
        res = eg.gateconv_forward(ci["H"], ci["k"], ci["v"], ci["rms_w_h"], ci["rms_w_v"], ci["conv_w"])
        grads = [torch.empty_like(ci["H"]) for _ in range(3)] + \
            [torch.empty(d, device="cuda"), torch.empty(d, device="cuda"), torch.empty((4, d), device="cuda")]
        ws = torch.empty(eg.engram_gateconv_bwd_workspace_size(M, T, d), device="cuda", dtype=torch.uint8)
        if args.op == "gateconv_fwd":
            fn = lambda: eg.engram_gateconv_fwd(ci["H"], ci["k"], ci["v"], ci["rms_w_h"], ci["rms_w_v"],
                                                ci["conv_w"], *res, stream=s)
        else:
            fn = lambda: eg.engram_gateconv_bwd(ci["dY"], ci["H"], ci["k"], ci["v"], ci["rms_w_h"],
                                                ci["rms_w_v"], ci["conv_w"], *res[1:], *grads, ws, stream=s)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            fn()
        ms = time_region(torch, fn, max(1, args.steps), s)
    assert eg.engram_device_error() == 0
    print(json.dumps({"op": args.op, "ms": round(ms, 5)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the per-op sweep")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU baseline")
    ap.add_argument("--op", choices=["step", "gate_fwd", "gate_bwd", "gate_sep_fwd", "gate_sep_bwd", "gateconv_fwd",
                                     "gateconv_bwd", "decode"],
                    default="step", help="time one entry point alone (profiler captures)")
    ap.add_argument("--gc-workload", choices=sorted(GC_WORKLOADS), default="m4")
    ap.add_argument("--n", type=int, default=N_TOK, help="tokens of the gate ops (--op)")
    ap.add_argument("--h", type=int, default=4096, help="hidden size of the separate-tensor ops (--op)")
    ap.add_argument("--sweep-inputs", action="store_true",
                    help="--op gate_*: the forward sweep's inputs (LogUniform row scales, mask Bernoulli(0.5))")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.op != "step":
        run_single_op(args)
        return
    args.warmup = max(args.warmup, 3)

    import torch
    import engram_memory_gating_gb300 as eg
    from engram_memory_gating_gb300 import inputs as inputs_mod

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    eg.load()
    peak, peak_kind = peaks()
    stream = torch.cuda.Stream()

    inp = inputs_mod.gate_inputs(N_TOK, 1, device="cuda", mask="bern0.9")
    x, kv, w, mask, gout = inp["x"], inp["kv"], inp["weight"], inp["mask"], inp["grad_out"]
    out = torch.empty_like(x)
    saved = torch.empty((N_TOK, S, 4), device="cuda", dtype=torch.float32)
    gx, gkv, gw = torch.empty_like(x), torch.empty_like(kv), torch.empty_like(w)
    ws = torch.empty(eg.engram_gate_bwd_workspace_size(N_TOK), device="cuda", dtype=torch.uint8)

    def fwd():
        eg.engram_gate_fwd(x, kv, w, mask, out, saved, stream=stream)

    def bwd():
        eg.engram_gate_bwd(x, kv, w, saved, gout, gx, gkv, gw, ws, stream=stream)

    torch.cuda.synchronize()
    for _ in range(args.warmup):
        fwd()
        bwd()
    K = args.steps
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    # the timed steps, back to back: no event between two kernels, which
    # would end the overlap of one kernel's tail with the next one's launch
    with Clocks(local) as clk:
        t_start.record(stream)
        for i in range(K):
            fwd()
            bwd()
        t_end.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = t_start.elapsed_time(t_end) / K
    # forward / backward split (for the per-kernel rooflines): the same steps
    # again with an event around each entry point
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for i in range(K):
        evs[i][0].record(stream)
        fwd()
        evs[i][1].record(stream)
        bwd()
        evs[i][2].record(stream)
    torch.cuda.synchronize()
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    ms = max_over_ranks(ms, dist, "cuda")
    value = job_throughput(N_TOK, world, ms)
    step_bytes = N_TOK * (FWD_BYTES_PER_TOKEN + BWD_BYTES_PER_TOKEN) + FWD_FIXED + BWD_FIXED
    fwd_bytes = N_TOK * FWD_BYTES_PER_TOKEN + FWD_FIXED
    bwd_bytes = N_TOK * BWD_BYTES_PER_TOKEN + BWD_FIXED
    bwd_gbs = bwd_bytes / (bwd_ms * 1e-3) / 1e9
    fwd_gbs = fwd_bytes / (fwd_ms * 1e-3) / 1e9
    csrc = "engram_memory_gating_gb300/csrc/"
    hdrs = [csrc + "common.cuh", csrc + "engram_internal.h"]
    traffic = profile_traffic("gate_bwd_n8192.md", [csrc + "gate_bwd.cu", csrc + "gate_bwd_fused.cu"] + hdrs)
    traffic_fwd = profile_traffic("gate_fwd_n8192.md", [csrc + "gate_fwd.cu"] + hdrs)

    # ---- end to end through the public API with host buffers (pinned).  Every
    # step copies all of its inputs host -> device and all of its outputs
    # device -> host.  Three streams and two device buffer sets pipeline the
    # steps: step i + 1's inputs go in and step i - 1's outputs come out while
    # step i computes (the link carries both directions at once).
    h = {k: v.cpu().pin_memory() for k, v in inp.items()}
    ho = {"out": torch.empty_like(h["x"]).pin_memory(),
          "saved": torch.empty((N_TOK, S, 4), dtype=torch.float32).pin_memory(),
          "gx": torch.empty_like(h["x"]).pin_memory(), "gkv": torch.empty_like(h["kv"]).pin_memory(),
          "gw": torch.empty_like(h["weight"]).pin_memory()}
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = sum(t.numel() * t.element_size() for t in ho.values())
    sets = []
    for _ in range(2):
        di = {k: torch.empty_like(v, device="cuda") for k, v in h.items()}
        do = {"out": torch.empty_like(di["x"]), "saved": torch.empty((N_TOK, S, 4), device="cuda"),
              "gx": torch.empty_like(di["x"]), "gkv": torch.empty_like(di["kv"]),
              "gw": torch.empty_like(di["weight"])}
        sets.append((di, do))
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "done", "out")}

    def e2e_step(i):
        b = i & 1
        di, do = sets[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev["done"][b])          # step i - 2 has consumed these inputs
            for k in ("x", "kv", "weight", "mask", "grad_out"):
                di[k].copy_(h[k], non_blocking=True)
            ev["in"][b].record(s_in)
        stream.wait_event(ev["in"][b])
        if i >= 2:
            stream.wait_event(ev["out"][b])             # step i - 2's outputs have left
        eg.engram_gate_fwd(di["x"], di["kv"], di["weight"], di["mask"], do["out"], do["saved"],
                           stream=stream)
        eg.engram_gate_bwd(di["x"], di["kv"], di["weight"], do["saved"], di["grad_out"], do["gx"],
                           do["gkv"], do["gw"], ws, stream=stream)
        ev["done"][b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["done"][b])
            for k in ("out", "saved", "gx", "gkv", "gw"):
                ho[k].copy_(do[k], non_blocking=True)
            ev["out"][b].record(s_out)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    Ke = max(6, min(50, K // 20))
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0.record(s_in)
    for i in range(Ke):
        e2e_step(i)
    s_in.wait_stream(s_out)
    t1.record(s_in)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(t0.elapsed_time(t1) / Ke, dist, "cuda")
    del sets

    launch = {"fwd": eg.engram_launch_info(0, N_TOK), "bwd": eg.engram_launch_info(1, N_TOK)}
    ops = None
    if not args.no_extra and rank == 0:
        ops = {"gate_fwd_N8192": op_entry(fwd_ms, fwd_bytes, peak),
               "gate_bwd_N8192": op_entry(bwd_ms, bwd_bytes, peak)}
        del h, ho
        ops.update(extra_ops(torch, eg, inputs_mod, stream, peak))
    err = eg.engram_device_error()
    if dist:
        dist.barrier()
    if rank != 0:
        return
    cpu = None if (args.no_cpu or world > 1) else cpu_baseline()
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": run_config(world),
        "launch": launch,
        "hbm_GB_s": round(step_bytes / (ms * 1e-3) / 1e9, 1),
        "roofline": {"kernel": ("engram_gate_bwd (gate_bwd_fused_kernel + wreduce_kernel), N=8192"
                                if launch["bwd"]["kernels"] == 2 else
                                "engram_gate_bwd (gate_bwd_coef_kernel + gate_bwd_main_kernel + wreduce_kernel), N=8192"),
                     "bound": "hbm", "achieved": round(bwd_gbs, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(bwd_gbs / peak, 4),
                     "peak_nominal": NOMINAL_GBS, "frac_nominal": round(bwd_gbs / NOMINAL_GBS, 4),
                     "traffic": traffic},
        "roofline_fwd": {"kernel": "engram_gate_fwd (gate_fwd_quad_kernel<true>), N=8192", "bound": "hbm",
                         "achieved": round(fwd_gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(fwd_gbs / peak, 4), "peak_nominal": NOMINAL_GBS,
                         "frac_nominal": round(fwd_gbs / NOMINAL_GBS, 4), "traffic": traffic_fwd},
        "cpu_baseline": cpu,
        "e2e": {"value": round(job_throughput(N_TOK, world, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4)},
        # kernels per step as the library reports them for this N: the forward,
        # and the backward's (one pass + grad_weight merge, or coefficients,
        # elementwise and merge)
        "gpu_launches": (launch["fwd"]["kernels"] + launch["bwd"]["kernels"]) * K,
        "clocks": clk.summary(),
        "device_error_flags": err,
    }
    if ops is not None:
        line["ops"] = ops
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
