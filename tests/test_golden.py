"""Stored fixtures of tests/golden/.

closed_forms.json holds values derived by hand from the definitions (each
entry states its derivation); the oracle must reproduce them.  The oracle_*
fixtures were written by tests/golden/make_golden.py from the oracle alone on
formula-defined inputs: on the CPU they guard the oracle against unintended
changes, and on the GPU the CUDA path is checked against them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from engram_memory_gating_gb300.inputs import (bf16_bits, gate_inputs_formula,
                                               gateconv_inputs_formula)
from tolerance import BF16_REL, F32_ABS, F32_REL, ROW_FLOOR, bf16_bits_to_f64

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def f64(t):
    if t.dtype == torch.bfloat16:
        return bf16_bits_to_f64(bf16_bits(t)).reshape(tuple(t.shape))
    return t.detach().double().cpu().numpy()


def _gm():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(GOLDEN, "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


# ---------------------------------------------------------------- closed forms

def _gate_case(d, k_sign=1.0, w_val=1.0):
    x = np.ones((1, 1, d))
    kv = np.concatenate([k_sign * np.ones((1, d)), np.ones((1, d))], axis=1)
    w = np.full((1, d), w_val)
    return oracle.gate_fwd(x, kv, w)


@pytest.mark.parametrize("name,d,k_sign,w_val", [
    ("gate_zero_weight", 16, 1.0, 0.0),
    ("gate_key_equals_x_d16", 16, 1.0, 1.0),
    ("gate_key_minus_x_d16", 16, -1.0, 1.0),
    ("gate_key_equals_x_d64", 64, 1.0, 1.0),
    ("gate_clamp", 16, 1.0, 2.5e-8),
])
def test_gate_closed_forms(name, d, k_sign, w_val):
    cf = load("closed_forms.json")[name]
    _, saved = _gate_case(d, k_sign, w_val)
    assert saved[0, 0, 0] == pytest.approx(cf["gate"], rel=1e-14, abs=1e-300)
    assert saved[0, 0, 1] == pytest.approx(cf["dot"], rel=1e-12, abs=1e-300)


def test_gateconv_closed_forms():
    cf = load("closed_forms.json")
    d = 16
    H = np.ones((1, 2, d))
    v = np.linspace(-1.0, 1.0, 2 * d).reshape(1, 2, d)
    ones = np.ones(d)
    cw = np.zeros((4, d))
    Y, vhat, alpha, rh, rk, rv = oracle.gateconv_fwd(H, H.copy(), v, ones, ones, cw)
    c = cf["gateconv_h_equals_k_d16"]
    assert np.allclose(alpha, c["alpha"], rtol=1e-14)
    assert np.allclose(rh, c["rrms_h"], rtol=1e-14)
    assert cf["gateconv_zero_conv"]["Y_equals_vhat"] and np.array_equal(Y, vhat)


# ---------------------------------------------------- oracle regression (CPU)

def test_formula_inputs_are_stable():
    gm = _gm()
    g = gate_inputs_formula(64)
    c = gateconv_inputs_formula(2, 7, 16)
    assert gm.digest([g[k] for k in ("x", "kv", "weight", "mask", "grad_out")]) == \
        load("oracle_gate_n64.json")["inputs_sha256"]
    assert gm.digest([c[k] for k in ("H", "k", "v", "rms_w_h", "rms_w_v", "conv_w", "dY")]) == \
        load("oracle_gateconv_m2_t7_d16.json")["inputs_sha256"]


def test_oracle_reproduces_stored_gate_fixture():
    fx = load("oracle_gate_n64.json")
    now = _gm().gate_fixture()
    assert np.allclose(now["saved"], fx["saved"], rtol=1e-13, atol=0)
    for name in ("out", "grad_x", "grad_kv"):
        assert now[name]["index"] == fx[name]["index"]
        assert now[name]["bf16_bits"] == fx[name]["bf16_bits"]
        assert np.allclose(now[name]["exact"], fx[name]["exact"], rtol=1e-12, atol=1e-300)
    assert np.allclose(now["grad_weight"]["value"], fx["grad_weight"]["value"], rtol=1e-12, atol=1e-300)


def test_oracle_reproduces_stored_gateconv_fixture():
    fx = load("oracle_gateconv_m2_t7_d16.json")
    now = _gm().gateconv_fixture()
    for name in ("Y", "vhat", "dH", "dk", "dv"):
        assert now[name]["bf16_bits"] == fx[name]["bf16_bits"]
        assert np.allclose(now[name]["exact"], fx[name]["exact"], rtol=1e-12, atol=1e-300)
    for name in ("alpha", "rrms_h", "rrms_k", "rrms_v", "drms_w_h", "drms_w_v", "dconv_w"):
        assert np.allclose(now[name], fx[name], rtol=1e-12, atol=1e-300)


# ------------------------------------------------- CUDA path vs fixtures (GPU)

def _near(got, exact, floor):
    got, exact = np.asarray(got, dtype=np.float64), np.asarray(exact, dtype=np.float64)
    return np.abs(got - exact) <= BF16_REL * np.abs(exact) + floor


@pytest.mark.gpu
def test_cuda_gate_matches_stored_fixture():
    import engram_memory_gating_gb300 as eg
    fx = load("oracle_gate_n64.json")
    inp = {k: v.cuda() for k, v in gate_inputs_formula(64).items()}
    out, saved = eg.gate_forward(inp["x"], inp["kv"], inp["weight"], inp["mask"])
    gx, gkv, gw = eg.gate_backward(inp["x"], inp["kv"], inp["weight"], saved, inp["grad_out"])
    torch.cuda.synchronize()
    s = saved.cpu().double().numpy().reshape(-1)
    e = np.asarray(fx["saved"])
    assert np.all(np.abs(s - e) <= F32_REL * np.abs(e) + F32_ABS)
    for name, t in (("out", out), ("grad_x", gx), ("grad_kv", gkv)):
        got = f64(t).reshape(-1)[fx[name]["index"]]
        ex = np.asarray(fx[name]["exact"])
        floor = ROW_FLOOR * math.sqrt(float(np.mean(ex * ex)))
        assert _near(got, ex, floor).all(), name
    got = gw.cpu().double().numpy().reshape(-1)[fx["grad_weight"]["index"]]
    ex = np.asarray(fx["grad_weight"]["value"])
    assert np.all(np.abs(got - ex) <= F32_REL * np.abs(ex) + F32_ABS)


@pytest.mark.gpu
def test_cuda_gateconv_matches_stored_fixture():
    import engram_memory_gating_gb300 as eg
    fx = load("oracle_gateconv_m2_t7_d16.json")
    c = {k: v.cuda() for k, v in gateconv_inputs_formula(2, 7, 16).items()}
    res = eg.gateconv_forward(c["H"], c["k"], c["v"], c["rms_w_h"], c["rms_w_v"], c["conv_w"])
    g = eg.gateconv_backward(c["dY"], c["H"], c["k"], c["v"], c["rms_w_h"], c["rms_w_v"], c["conv_w"],
                             *res[1:])
    torch.cuda.synchronize()
    for name, t in (("Y", res[0]), ("vhat", res[1]), ("dH", g[0]), ("dk", g[1]), ("dv", g[2])):
        ex = np.asarray(fx[name]["exact"]).reshape(2, 7, 16)
        floor = ROW_FLOOR * np.sqrt(np.mean(ex * ex, axis=-1, keepdims=True))
        assert _near(f64(t), ex, floor).all(), name
    for name, t in (("alpha", res[2]), ("rrms_h", res[3]), ("rrms_k", res[4]), ("rrms_v", res[5])):
        e = np.asarray(fx[name]).reshape(2, 7)
        assert np.all(np.abs(t.cpu().double().numpy() - e) <= F32_REL * np.abs(e) + F32_ABS), name
    for name, t in (("drms_w_h", g[3]), ("drms_w_v", g[4]), ("dconv_w", g[5])):
        e = np.asarray(fx[name]).reshape(tuple(t.shape))
        scale = max(1.0, float(np.max(np.abs(e))))
        assert np.all(np.abs(t.cpu().double().numpy() - e) <= F32_REL * np.abs(e) + F32_ABS * scale), name
