"""Writes the stored oracle fixtures of tests/golden/ (oracle_*.json).

Inputs come from the formula generators of engram_memory_gating_gb300.inputs
(no random generator, so every machine builds the same tensors); every stored
value is computed by the fp64 oracle (oracle/) and nothing else.  The fixtures
freeze the oracle's results: a later change to the oracle's arithmetic that
moves them must say which passage of the pages justifies it.

    python tests/golden/make_golden.py
"""
from __future__ import annotations

import hashlib
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from engram_memory_gating_gb300.inputs import (  # noqa: E402
    bf16_bits, gate_inputs_formula, gateconv_inputs_formula)

N_SAMPLE = 64


def f64(t):
    if str(t.dtype) == "torch.bfloat16":
        b = bf16_bits(t).astype(np.uint32) << 16
        return b.view(np.float32).astype(np.float64).reshape(tuple(t.shape))
    return t.detach().double().numpy()


def digest(tensors) -> str:
    h = hashlib.sha256()
    for t in tensors:
        h.update(t.detach().contiguous().view(-1).view(dtype=__import__("torch").uint8).numpy().tobytes())
    return h.hexdigest()[:32]


def sample_idx(size: int) -> list[int]:
    """Fixed, spread-out flat indices of a tensor (prime stride)."""
    return sorted({(k * 7919 + 13) % size for k in range(N_SAMPLE)})


def floats(a) -> list[float]:
    return [float(x) for x in np.asarray(a, dtype=np.float64).reshape(-1)]


def bits(a) -> list[int]:
    return [int(x) for x in np.asarray(a).reshape(-1)]


def gate_fixture() -> dict:
    inp = gate_inputs_formula(64)
    x, kv, w, g = (f64(inp[k]) for k in ("x", "kv", "weight", "grad_out"))
    m = inp["mask"].numpy().astype(np.uint8)
    out, saved = oracle.gate_fwd(x, kv, w, m)
    gx, gkv, gw = oracle.gate_bwd(x, kv, w, saved, g)
    fx = {"inputs": "gate_inputs_formula(64)",
          "inputs_sha256": digest([inp[k] for k in ("x", "kv", "weight", "mask", "grad_out")]),
          "saved": floats(saved)}
    for name, arr, kind in (("out", out, "bf16"), ("grad_x", gx, "bf16"), ("grad_kv", gkv, "bf16"),
                            ("grad_weight", gw, "f64")):
        idx = sample_idx(arr.size)
        flat = np.asarray(arr).reshape(-1)
        vals = bits(oracle.round_bf16(flat[idx])) if kind == "bf16" else floats(flat[idx])
        fx[name] = {"index": idx, "bf16_bits" if kind == "bf16" else "value": vals}
        if kind == "bf16":
            fx[name]["exact"] = floats(flat[idx])
    return fx


def gateconv_fixture() -> dict:
    inp = gateconv_inputs_formula(2, 7, 16)
    H, k, v, wh, wv, cw, dY = (f64(inp[n]) for n in ("H", "k", "v", "rms_w_h", "rms_w_v", "conv_w", "dY"))
    Y, vhat, alpha, rh, rk, rv = oracle.gateconv_fwd(H, k, v, wh, wv, cw)
    vhat_bits = oracle.round_bf16(vhat)
    vh16 = (vhat_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    sc = [np.asarray(t, dtype=np.float32).astype(np.float64) for t in (alpha, rh, rk, rv)]
    dH, dk, dv, dwh, dwv, dcw = oracle.gateconv_bwd(dY, H, k, v, wh, wv, cw, vh16, *sc)
    fx = {"inputs": "gateconv_inputs_formula(2, 7, 16)",
          "inputs_sha256": digest([inp[n] for n in ("H", "k", "v", "rms_w_h", "rms_w_v", "conv_w", "dY")]),
          "note": "backward fed with the forward's outputs rounded as stored (vhat bf16, scalars fp32)"}
    for name, arr in (("Y", Y), ("vhat", vhat), ("dH", dH), ("dk", dk), ("dv", dv)):
        fx[name] = {"exact": floats(arr), "bf16_bits": bits(oracle.round_bf16(np.asarray(arr).reshape(-1)))}
    for name, arr in (("alpha", alpha), ("rrms_h", rh), ("rrms_k", rk), ("rrms_v", rv),
                      ("drms_w_h", dwh), ("drms_w_v", dwv), ("dconv_w", dcw)):
        fx[name] = floats(arr)
    return fx


def main():
    oracle.build()
    for name, fx in (("oracle_gate_n64.json", gate_fixture()), ("oracle_gateconv_m2_t7_d16.json", gateconv_fixture())):
        fx["written_by"] = "tests/golden/make_golden.py (oracle only)"
        with open(os.path.join(HERE, name), "w") as f:
            # one key per line, each value compact
            f.write("{\n" + ",\n".join(f"{json.dumps(k)}: {json.dumps(fx[k], separators=(',', ':'))}"
                                        for k in sorted(fx)) + "\n}\n")
        print("wrote", name)


if __name__ == "__main__":
    main()
