"""Pins for the saved-state gate oracle (forward and backward).

What the pages fix (cuDNN Frontend "Engram saved-state gate"; tile-kernels
engram gate tests) and what the mathematics fixes, checked without re-typing
the oracle's formula:
  * closed forms: zero weight, key equal / opposite to X, constant rows,
    all-zero rows, the 1e-6 clamp of the signed square root;
  * invariants: per-row scale invariance of dot and gate, stream permutation
    equivariance, the masked token identity, grad_v as the sum of the four
    shared-value contributions;
  * brute force: central finite differences of the fp64 forward against the
    analytic backward, for every element of X, KV and weight, and the
    product rule for the two q/k weights whose product is the fused weight.
"""
import math

import numpy as np
import pytest

import oracle

EPS = oracle.GATE_EPS
CLAMP = oracle.GATE_CLAMP


def sig(z):
    return 1.0 / (1.0 + math.exp(-z))


def rand_case(rng, N, S, d, w_scale=0.1):
    x = rng.standard_normal((N, S, d))
    kv = rng.standard_normal((N, (S + 1) * d))
    w = 1.0 + w_scale * rng.standard_normal((S, d))
    return x, kv, w


# ----------------------------------------------------------------- closed forms

def test_zero_weight_gives_half_gate():
    rng = np.random.default_rng(0)
    x, kv, _ = rand_case(rng, 3, 4, 32)
    w = np.zeros((4, 32))
    out, saved = oracle.gate_fwd(x, kv, w)
    assert np.all(saved[..., 1] == 0.0)
    assert np.all(saved[..., 0] == 0.5)
    v = kv[:, 4 * 32:]
    assert np.allclose(out, x + 0.5 * v[:, None, :], rtol=0, atol=1e-15)


@pytest.mark.parametrize("d", [4, 16, 64])
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_key_equal_to_x_gives_sigmoid_sqrt_d(d, sign):
    # k = +-x, w = 1: dot = +-sum xh^2 = +-d*m/(m+eps) with m = mean x^2, so the
    # gate is sigmoid(+-sqrt(d)) up to the eps term (1e-20 here).
    rng = np.random.default_rng(d)
    N, S = 2, 4
    x = rng.standard_normal((N, S, d))
    kv = rng.standard_normal((N, (S + 1) * d))
    for s in range(S):
        kv[:, s * d:(s + 1) * d] = sign * x[:, s, :]
    w = np.ones((S, d))
    _, saved = oracle.gate_fwd(x, kv, w)
    assert np.allclose(saved[..., 1], sign * d, rtol=1e-13, atol=0)
    assert np.allclose(saved[..., 0], sig(sign * math.sqrt(d)), rtol=1e-13, atol=0)
    if d == 16 and sign > 0:
        # sigmoid(4) written out
        assert abs(saved[0, 0, 0] - 0.9820137900379085) < 1e-15


def test_constant_row_rstd():
    # mean of c^2 over d is c^2, so rstd = 1/sqrt(c^2 + eps): a sum instead of
    # a mean, or eps outside the root, would change this.
    d = 24
    x = np.full((1, 4, d), 3.0)
    kv = np.full((1, 5 * d), -0.5)
    w = np.ones((4, d))
    _, saved = oracle.gate_fwd(x, kv, w)
    assert np.allclose(saved[0, :, 2], 1.0 / math.sqrt(9.0 + EPS), rtol=1e-15)
    assert np.allclose(saved[0, :, 3], 1.0 / math.sqrt(0.25 + EPS), rtol=1e-15)
    # xh = 1, kh = -1 everywhere, so dot = -d
    assert np.allclose(saved[0, :, 1], -d, rtol=1e-14)


def test_zero_row():
    d = 16
    x = np.zeros((1, 4, d))
    kv = np.random.default_rng(1).standard_normal((1, 5 * d))
    w = np.ones((4, d))
    out, saved = oracle.gate_fwd(x, kv, w)
    assert np.allclose(saved[0, :, 2], 1e10, rtol=1e-12)   # 1/sqrt(eps)
    assert np.all(saved[0, :, 1] == 0.0)
    assert np.all(saved[0, :, 0] == 0.5)                   # sign(0) = 0 -> sigmoid(0)
    assert np.allclose(out[0], 0.5 * kv[0, 4 * d:][None, :], rtol=0, atol=0)


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_clamp_of_signed_sqrt(sign):
    # |dot| below 1e-6: the signed root is sign(dot)*sqrt(1e-6) = +-1e-3
    d = 16
    rng = np.random.default_rng(3)
    x = rng.standard_normal((1, 4, d))
    kv = rng.standard_normal((1, 5 * d))
    for s in range(4):
        kv[0, s * d:(s + 1) * d] = sign * x[0, s]
    w = np.full((4, d), 1e-8)                      # dot = +-1.6e-7
    _, saved = oracle.gate_fwd(x, kv, w)
    assert np.allclose(saved[0, :, 1], sign * 1.6e-7, rtol=1e-12)
    assert np.allclose(saved[0, :, 0], sig(sign * 1e-3), rtol=1e-15)
    # just above the clamp the root is taken of |dot| itself
    w = np.full((4, d), 1e-5)                      # dot = +-1.6e-4
    _, saved = oracle.gate_fwd(x, kv, w)
    assert np.allclose(saved[0, :, 0], sig(sign * math.sqrt(1.6e-4)), rtol=1e-12)


# ------------------------------------------------------------------- invariants

@pytest.mark.parametrize("c", [1e-3, 0.5, 7.0, 1e3])
def test_scale_invariance(c):
    rng = np.random.default_rng(11)
    x, kv, w = rand_case(rng, 4, 4, 32)
    _, s0 = oracle.gate_fwd(x, kv, w)
    x2 = x.copy()
    kv2 = kv.copy()
    x2[1, 2] *= c
    kv2[3, 0:32] *= c
    kv2[2, 96:128] *= 1.0 / c
    _, s1 = oracle.gate_fwd(x2, kv2, w)
    assert np.allclose(s1[..., :2], s0[..., :2], rtol=1e-12, atol=0)


def test_stream_permutation_equivariance():
    rng = np.random.default_rng(12)
    N, S, d = 3, 4, 16
    x, kv, w = rand_case(rng, N, S, d)
    g = rng.standard_normal((N, S, d))
    perm = [2, 0, 3, 1]
    xp = x[:, perm]
    kvp = kv.copy()
    for new, old in enumerate(perm):
        kvp[:, new * d:(new + 1) * d] = kv[:, old * d:(old + 1) * d]
    wp = w[perm]
    gp = g[:, perm]
    out, saved = oracle.gate_fwd(x, kv, w)
    outp, savedp = oracle.gate_fwd(xp, kvp, wp)
    assert np.array_equal(outp, out[:, perm])
    assert np.array_equal(savedp, saved[:, perm])
    gx, gkv, gw = oracle.gate_bwd(x, kv, w, saved, g)
    gxp, gkvp, gwp = oracle.gate_bwd(xp, kvp, wp, savedp, gp)
    assert np.allclose(gxp, gx[:, perm], rtol=1e-14, atol=1e-14)
    for new, old in enumerate(perm):
        assert np.allclose(gkvp[:, new * d:(new + 1) * d], gkv[:, old * d:(old + 1) * d],
                           rtol=1e-14, atol=1e-14)
    # the shared value's gradient does not depend on the stream order
    assert np.allclose(gkvp[:, S * d:], gkv[:, S * d:], rtol=1e-13, atol=1e-14)
    assert np.allclose(gwp, gw[perm], rtol=1e-13, atol=1e-14)


def test_mask_false_identity():
    rng = np.random.default_rng(13)
    N, S, d = 4, 4, 32
    x, kv, w = rand_case(rng, N, S, d)
    x = oracle.bf16_to_f64(oracle.round_bf16(x))
    mask = np.array([1, 0, 1, 0], dtype=np.uint8)
    out, saved = oracle.gate_fwd(x, kv, w, mask)
    _, saved_on = oracle.gate_fwd(x, kv, w, None)
    # out == X bit-exactly after the one bf16 rounding
    assert np.array_equal(oracle.round_bf16(out[1]), oracle.round_bf16(x[1]))
    assert np.array_equal(oracle.round_bf16(out[3]), oracle.round_bf16(x[3]))
    assert np.all(saved[[1, 3], :, 0] == 0.0)
    assert np.array_equal(saved[..., 1:], saved_on[..., 1:])
    assert np.array_equal(saved[[0, 2]], saved_on[[0, 2]])
    g = rng.standard_normal((N, S, d))
    gx, gkv, gw = oracle.gate_bwd(x, kv, w, saved, g)
    assert np.array_equal(gx[[1, 3]], g[[1, 3]])
    assert np.all(gkv[[1, 3], :S * d] == 0.0)
    # no v or weight contribution from masked tokens
    keep = np.array([1, 0, 1, 0], dtype=bool)
    gx2, gkv2, gw2 = oracle.gate_bwd(x[keep], kv[keep], w, saved[keep], g[keep])
    assert np.all(gkv[[1, 3], S * d:] == 0.0)
    assert np.allclose(gw, gw2, rtol=1e-14, atol=1e-15)


def test_grad_v_is_sum_of_stream_contributions():
    rng = np.random.default_rng(14)
    N, S, d = 5, 4, 16
    x, kv, w = rand_case(rng, N, S, d)
    g = rng.standard_normal((N, S, d))
    _, saved = oracle.gate_fwd(x, kv, w)
    _, gkv, _ = oracle.gate_bwd(x, kv, w, saved, g)
    expect = np.einsum("ns,nsd->nd", saved[..., 0], g)
    assert np.allclose(gkv[:, S * d:], expect, rtol=1e-14, atol=1e-14)


# ------------------------------------------------------ finite differences (fp64)

def _loss(x, kv, w, g):
    out, _ = oracle.gate_fwd(x, kv, w)
    return float(np.sum(out * g))


def _fd_check(f, theta, analytic, rel=1e-6):
    flat = theta.reshape(-1)
    an = analytic.reshape(-1)
    scale = np.max(np.abs(an))
    worst = 0.0
    for i in range(flat.size):
        # fourth-order central stencil: truncation O(h^4), round-off ~1e-11
        h = 1e-4 * max(1.0, abs(flat[i]))
        old = flat[i]
        vals = []
        for k in (2, 1, -1, -2):
            flat[i] = old + k * h
            vals.append(f())
        flat[i] = old
        fd = (-vals[0] + 8 * vals[1] - 8 * vals[2] + vals[3]) / (12 * h)
        err = abs(fd - an[i]) / max(abs(an[i]), 1e-3 * scale)
        worst = max(worst, err)
    assert worst < rel, worst


def _safe_case(seed, N, S, d):
    # keep |dot| away from the 1e-6 clamp, where the derivative jumps
    rng = np.random.default_rng(seed)
    while True:
        x, kv, w = rand_case(rng, N, S, d, w_scale=0.3)
        _, saved = oracle.gate_fwd(x, kv, w)
        if np.min(np.abs(saved[..., 1])) > 1e-2 and np.max(np.abs(saved[..., 1])) < 30:
            return rng, x, kv, w


@pytest.mark.parametrize("d,N,S", [(8, 5, 4), (16, 4, 4), (32, 3, 4), (64, 3, 4), (16, 3, 2)])
def test_backward_matches_finite_differences(d, N, S):
    rng, x, kv, w = _safe_case(100 + d + S, N, S, d)
    g = rng.standard_normal((N, S, d))
    _, saved = oracle.gate_fwd(x, kv, w)
    gx, gkv, gw = oracle.gate_bwd(x, kv, w, saved, g)
    _fd_check(lambda: _loss(x, kv, w, g), x, gx)
    _fd_check(lambda: _loss(x, kv, w, g), kv, gkv)
    _fd_check(lambda: _loss(x, kv, w, g), w, gw)


def test_product_rule_for_the_two_norm_weights():
    # weight = wh * we (fused fp32 product of the q/k norm weights); the
    # caller's grads are grad_wh = grad_w * we and grad_we = grad_w * wh
    rng, x, kv, _ = _safe_case(5, 4, 4, 16)
    wh = 1.0 + 0.3 * rng.standard_normal((4, 16))
    we = 1.0 + 0.3 * rng.standard_normal((4, 16))
    g = rng.standard_normal((4, 4, 16))
    _, saved = oracle.gate_fwd(x, kv, wh * we)
    _, _, gw = oracle.gate_bwd(x, kv, wh * we, saved, g)
    _fd_check(lambda: _loss(x, kv, wh * we, g), wh, gw * we)
    _fd_check(lambda: _loss(x, kv, wh * we, g), we, gw * wh)


def test_clamped_region_has_zero_gate_derivative():
    # below the clamp the signed root is constant, so X and the key only act
    # through out = X + gate*v with a frozen gate
    d = 16
    rng = np.random.default_rng(21)
    x = rng.standard_normal((1, 4, d))
    kv = rng.standard_normal((1, 5 * d))
    for s in range(4):
        kv[0, s * d:(s + 1) * d] = x[0, s]
    w = np.full((4, d), 1e-8)
    g = rng.standard_normal((1, 4, d))
    _, saved = oracle.gate_fwd(x, kv, w)
    gx, gkv, gw = oracle.gate_bwd(x, kv, w, saved, g)
    assert np.array_equal(gx, g)
    assert np.all(gkv[:, :4 * d] == 0.0)
    assert np.all(gw == 0.0)


def test_saturated_gate_keeps_its_derivative_through_fp32_saved_state():
    # a key close to X at d = 64 gives dot ~ 60, sq ~ 7.8, 1 - gate ~ 4e-4.
    # An fp32 saved gate keeps 1 - gate only to ~1e-4 relative; the backward
    # evaluates sigmoid'(sq) from the saved dot, so fp32 and fp64 saved state
    # give the same gradients to fp32 precision of dot and rstd.
    d = 64
    rng = np.random.default_rng(31)
    x = rng.standard_normal((3, 4, d))
    kv = rng.standard_normal((3, 5 * d))
    for s in range(4):
        kv[:, s * d:(s + 1) * d] = x[:, s] + 0.3 * rng.standard_normal((3, d))
    w = 1.0 + 0.1 * rng.standard_normal((4, d))
    g = rng.standard_normal((3, 4, d))
    _, saved = oracle.gate_fwd(x, kv, w)
    assert np.all(saved[..., 1] > 40)
    saved32 = saved.astype(np.float32).astype(np.float64)
    lost = np.abs((1.0 - saved32[..., 0]) / (1.0 - saved[..., 0]) - 1.0)
    assert np.max(lost) > 1e-5   # fp32 lost those bits
    r64 = oracle.gate_bwd(x, kv, w, saved, g)
    r32 = oracle.gate_bwd(x, kv, w, saved32, g)
    # compared on the scale of each tensor (the gate path of grad_x is
    # grad_x - grad_out); the old 1 - gate form would be off by `lost`
    pairs = [(r64[0] - g, r32[0] - g), (r64[1][:, :4 * d], r32[1][:, :4 * d]),
             (r64[1][:, 4 * d:], r32[1][:, 4 * d:]), (r64[2], r32[2])]
    for a, b in pairs:
        assert np.max(np.abs(a - b)) <= 2e-6 * np.max(np.abs(a))


def test_fused_weight_is_the_exact_product():
    # products of bf16 values are exact in fp64; compare with rational arithmetic
    from fractions import Fraction
    rng = np.random.default_rng(31)
    wh = oracle.bf16_to_f64(oracle.round_bf16(rng.standard_normal(64)))
    we = oracle.bf16_to_f64(oracle.round_bf16(3.0 * rng.standard_normal(64)))
    got = oracle.fused_weight(wh, we)
    for a, b, c in zip(wh, we, got):
        assert Fraction(c) == Fraction(a) * Fraction(b)


def test_fused_weight_bwd_sums_blocks_and_applies_the_product_rule():
    # per-block partials of the gate's grad_w, summed and pushed through
    # w = wh * we, give the derivatives of the loss in wh and we (differences)
    rng, x, kv, _ = _safe_case(6, 6, 4, 16)
    wh = 1.0 + 0.3 * rng.standard_normal((4, 16))
    we = 1.0 + 0.3 * rng.standard_normal((4, 16))
    g = rng.standard_normal((6, 4, 16))
    w = oracle.fused_weight(wh, we)
    _, saved = oracle.gate_fwd(x, kv, w)
    parts = np.stack([oracle.gate_bwd(x[b:b + 2], kv[b:b + 2], w, saved[b:b + 2], g[b:b + 2])[2]
                      for b in range(0, 6, 2)])
    gw, gwh, gwe = oracle.fused_weight_bwd(parts, wh, we)
    _, _, gw_all = oracle.gate_bwd(x, kv, w, saved, g)
    assert np.allclose(gw, gw_all, rtol=1e-13, atol=1e-15)
    _fd_check(lambda: _loss(x, kv, oracle.fused_weight(wh, we), g), wh, gwh)
    _fd_check(lambda: _loss(x, kv, oracle.fused_weight(wh, we), g), we, gwe)
