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


def _formula(shape, a: float, b: float, c: float, scale: float = 1.0) -> torch.Tensor:
    """Deterministic, generator-free values scale * sin(a*i + b*j + c) over the
    flattened index i and the leading index j: the same on every machine."""
    n = 1
    for s in shape:
        n *= s
    i = torch.arange(n, dtype=torch.float64)
    j = torch.div(i, n // shape[0], rounding_mode="floor")
    return (scale * torch.sin(a * i + b * j + c)).reshape(shape)


def gate_inputs_formula(N: int = 64) -> dict:
    """Small gate inputs defined by formulas (no random generator), for the
    stored fixtures: x, kv, grad_out bf16, weight fp32, mask [1, 0, 1, ...]."""
    x = _formula((N, S_STREAMS, D_GATE), 0.37, 1.3, 0.1, 2.0).to(torch.bfloat16)
    kv = _formula((N, (S_STREAMS + 1) * D_GATE), 0.23, 0.7, 0.5, 1.5).to(torch.bfloat16)
    w = (1.0 + 0.1 * _formula((S_STREAMS, D_GATE), 0.11, 0.9, 0.3)).to(torch.float32)
    mask = torch.tensor([n % 2 == 0 or n % 3 == 2 for n in range(N)], dtype=torch.bool)
    g = _formula((N, S_STREAMS, D_GATE), 0.53, 0.4, 0.2).to(torch.bfloat16)
    return {"x": x, "kv": kv, "weight": w.contiguous(), "mask": mask, "grad_out": g}


def gateconv_inputs_formula(M: int = 2, T: int = 7, d: int = 16) -> dict:
    """Small GateConv inputs defined by formulas (no random generator)."""
    H = _formula((M, T, d), 0.31, 0.8, 0.2, 1.5).to(torch.bfloat16)
    k = _formula((M, T, d), 0.17, 0.6, 0.9).to(torch.bfloat16)
    v = _formula((M, T, d), 0.29, 1.1, 0.4).to(torch.bfloat16)
    wh = (1.0 + 0.1 * _formula((d,), 0.7, 0.0, 0.1)).to(torch.float32)
    wv = (1.0 + 0.1 * _formula((d,), 0.45, 0.0, 0.6)).to(torch.float32)
    cw = (0.5 * _formula((4, d), 0.13, 1.7, 0.3)).to(torch.float32)
    dY = _formula((M, T, d), 0.41, 0.5, 0.7).to(torch.bfloat16)
    return {"H": H, "k": k, "v": v, "rms_w_h": wh.contiguous(), "rms_w_v": wv.contiguous(),
            "conv_w": cw.contiguous(), "dY": dY}


def decode_inputs(B: int, d_mem: int, d: int, L: int, w: int = 4, seed: int = 0, *,
                  device="cpu") -> dict:
    """Inputs of one GateConv decode step: e (B,d_mem), h (B,d), conv_state
    (B,L,d) bf16 ~N(0,1); W_K, W_V (d_mem,d) bf16 ~N(0, 1/d_mem) (so k, v are
    of unit scale); rms_w_h, rms_w_v = 1 + 0.1 N(0,1); conv_w (w,d) ~N(0, 0.25)."""
    dev = torch.device(device)
    g = _gen(dev, seed)
    e = _randn_bf16((B, d_mem), g, dev)
    h = _randn_bf16((B, d), g, dev)
    st = _randn_bf16((B, L, d), g, dev)
    WK = _randn_bf16((d_mem, d), g, dev, 1.0 / math.sqrt(d_mem))
    WV = _randn_bf16((d_mem, d), g, dev, 1.0 / math.sqrt(d_mem))
    wh = (1.0 + 0.1 * torch.randn(d, generator=g, device=dev)).contiguous()
    wv = (1.0 + 0.1 * torch.randn(d, generator=g, device=dev)).contiguous()
    cw = (0.5 * torch.randn((w, d), generator=g, device=dev)).contiguous()
    return {"e": e, "h": h, "conv_state": st, "W_K": WK, "W_V": WV, "rms_w_h": wh, "rms_w_v": wv,
            "conv_w": cw}
