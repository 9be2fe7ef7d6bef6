"""Seeded synthetic inputs for the Engram gate and GateConv workloads.

This module only draws random tensors; it holds none of the gate's
arithmetic.  Tests feed the same tensors (as bf16 bit patterns / fp32 values
copied to the host) to the CPU oracle and to the CUDA path, and ``bench.py``
uses it for the timed workloads.

Distributions follow the workloads the pages benchmark (cuDNN Frontend
"Engram saved-state gate"; tile-kernels engram gate tests; TileOPs GateConv):
bf16 activations ~N(0,1), fused fp32 weight 1 + 0.1*N(0,1), boolean token
mask, bf16 upstream gradient ~N(0,1).  ``sigma="loguniform"`` scales each
token's X and KV rows by one factor drawn from LogUniform(1e-2, 1e2).
"""
from __future__ import annotations

import math

import torch

S_STREAMS = 4
D_GATE = 5120


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn_bf16(shape, g, device, scale=None) -> torch.Tensor:
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if scale is not None:
        t.mul_(scale)
    return t.to(torch.bfloat16)


def gate_inputs(N: int, seed: int = 0, *, device="cpu", mask: str = "all",
                sigma: str | None = None, d: int = D_GATE, S: int = S_STREAMS,
                with_grad: bool = True) -> dict:
    """Inputs of the four-stream saved-state gate.

    Returns a dict with x (N,S,d) bf16, kv (N,(S+1)d) bf16, weight (S,d) fp32,
    mask (N,) bool and, if requested, grad_out (N,S,d) bf16.
    mask: "all" (all true), "bern0.9", "bern0.5", "none" (all false).
    """
    dev = torch.device(device)
    g = _gen(dev, seed)
    scale_x = scale_kv = None
    if sigma == "loguniform":
        u = torch.rand((N, 1, 1), generator=g, device=dev, dtype=torch.float32)
        lo, hi = math.log(1e-2), math.log(1e2)
        sig = torch.exp(lo + (hi - lo) * u)
        scale_x = sig
        scale_kv = sig.view(N, 1)
    elif sigma is not None:
        raise ValueError(sigma)
    x = _randn_bf16((N, S, d), g, dev, scale_x)
    kv = _randn_bf16((N, (S + 1) * d), g, dev, scale_kv)
    weight = (1.0 + 0.1 * torch.randn((S, d), generator=g, device=dev,
                                      dtype=torch.float32)).contiguous()
    if mask == "all":
        m = torch.ones(N, dtype=torch.bool, device=dev)
    elif mask == "none":
        m = torch.zeros(N, dtype=torch.bool, device=dev)
    elif mask.startswith("bern"):
        p = float(mask[4:])
        m = torch.rand(N, generator=g, device=dev) < p
    else:
        raise ValueError(mask)
    out = {"x": x, "kv": kv, "weight": weight, "mask": m}
    if with_grad:
        out["grad_out"] = _randn_bf16((N, S, d), g, dev)
    return out


def gateconv_inputs(M: int, T: int, d: int, seed: int = 0, *, device="cpu",
                    h_scale: float = 1.0, v_std: float = 1.0,
                    conv_var: float = 0.25, with_grad: bool = True) -> dict:
    """Inputs of GateConv: H, k, v (M,T,d) bf16; rms_w_h, rms_w_v (d,) fp32
    = 1 + 0.1*N(0,1); conv_w (4,d) fp32 ~ N(0, conv_var) (variance);
    dY (M,T,d) bf16 ~ N(0,1)."""
    dev = torch.device(device)
    g = _gen(dev, seed)
    H = _randn_bf16((M, T, d), g, dev, h_scale if h_scale != 1.0 else None)
    k = _randn_bf16((M, T, d), g, dev)
    v = _randn_bf16((M, T, d), g, dev, v_std if v_std != 1.0 else None)
    wh = (1.0 + 0.1 * torch.randn(d, generator=g, device=dev)).contiguous()
    wv = (1.0 + 0.1 * torch.randn(d, generator=g, device=dev)).contiguous()
    cw = (math.sqrt(conv_var) * torch.randn((4, d), generator=g, device=dev)).contiguous()
    out = {"H": H, "k": k, "v": v, "rms_w_h": wh, "rms_w_v": wv, "conv_w": cw}
    if with_grad:
        out["dY"] = _randn_bf16((M, T, d), g, dev)
    return out


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
