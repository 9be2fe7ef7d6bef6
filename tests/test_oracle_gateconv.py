"""Pins for the GateConv oracle (TileOPs "Engram Operators", GateConv section).

The page gives the stage order (RMSNorm gating -> causal depthwise conv1d,
4 taps -> SiLU + residual), the shapes and the saved tensors, but no
formula.  Checked here:
  * closed forms: zero conv weights (Y = vhat), an identity tap on the
    current token (Y = SiLU(u) + vhat), a pure 3-token delay, zero value
    (Y = 0 and no gradient into H or k), H = k (alpha = sigmoid(sqrt(d)));
  * invariants: causality along the sequence, independence of batch rows;
  * brute force: fourth-order central finite differences of the fp64
    forward against the analytic backward for every input and weight;
  * the conv against the standard causal depthwise conv1d (torch's grouped
    Conv1d with left padding, written independently of the oracle), which
    fixes the tap order and the causal zero padding.
The gate formula (a plain sigmoid of the normalised dot scaled by 1/sqrt(d),
one weight shared by H and k) is a reading of the page, not printed by it:
for that choice parity is unpinned.
"""
import math

import numpy as np
import pytest

import oracle

EPS = oracle.GATECONV_EPS


def silu(c):
    return c / (1.0 + np.exp(-c))


def rand_case(rng, M, T, d):
    H = rng.standard_normal((M, T, d))
    k = rng.standard_normal((M, T, d))
    v = rng.standard_normal((M, T, d))
    wh = 1.0 + 0.1 * rng.standard_normal(d)
    wv = 1.0 + 0.1 * rng.standard_normal(d)
    cw = 0.5 * rng.standard_normal((4, d))
    return H, k, v, wh, wv, cw


def test_zero_conv_gives_gated_value():
    rng = np.random.default_rng(0)
    H, k, v, wh, wv, _ = rand_case(rng, 2, 7, 16)
    cw = np.zeros((4, 16))
    Y, vhat, alpha, *_ = oracle.gateconv_fwd(H, k, v, wh, wv, cw)
    assert np.array_equal(Y, vhat)
    assert np.allclose(vhat, alpha[..., None] * v, rtol=1e-15, atol=0)


def test_current_token_tap_and_delay_tap():
    rng = np.random.default_rng(1)
    M, T, d = 2, 9, 16
    H, k, v, wh, wv, _ = rand_case(rng, M, T, d)
    cw = np.zeros((4, d))
    cw[3] = 1.0
    Y, vhat, alpha, rh, rk, rv = oracle.gateconv_fwd(H, k, v, wh, wv, cw)
    u = vhat * rv[..., None] * wv
    assert np.allclose(Y, silu(u) + vhat, rtol=1e-14, atol=1e-15)
    # tap 0 reads the token three steps back; the first three see zero padding
    cw = np.zeros((4, d))
    cw[0] = 1.0
    Y0, vhat0, *_ = oracle.gateconv_fwd(H, k, v, wh, wv, cw)
    assert np.allclose(Y0[:, 3:], silu(u[:, :-3]) + vhat0[:, 3:], rtol=1e-14, atol=1e-15)
    assert np.array_equal(Y0[:, :3], vhat0[:, :3])


def test_rms_of_gated_value():
    # u = vhat * rrms_v * wv has mean square mean(wv^2 vh^2)/(mean vh^2 + eps);
    # with wv = 1 it is 1 - eps/(mean vh^2 + eps)
    rng = np.random.default_rng(2)
    H, k, v, wh, _, cw = rand_case(rng, 1, 4, 32)
    wv = np.ones(32)
    Y, vhat, alpha, rh, rk, rv = oracle.gateconv_fwd(H, k, v, wh, wv, cw)
    m = np.mean(vhat ** 2, axis=-1)
    assert np.allclose(rv, 1.0 / np.sqrt(m + EPS), rtol=1e-14)
    u = vhat * rv[..., None]
    assert np.allclose(np.mean(u ** 2, axis=-1), m / (m + EPS), rtol=1e-13)


@pytest.mark.parametrize("d", [16, 64])
def test_h_equal_k_gives_sigmoid_sqrt_d(d):
    rng = np.random.default_rng(d)
    H, _, v, _, wv, cw = rand_case(rng, 1, 3, d)
    wh = np.ones(d)
    Y, vhat, alpha, rh, rk, rv = oracle.gateconv_fwd(H, H.copy(), v, wh, wv, cw)
    m = np.mean(H ** 2, axis=-1)
    z = math.sqrt(d) * m / (m + EPS)
    assert np.allclose(alpha, 1.0 / (1.0 + np.exp(-z)), rtol=1e-14)
    assert np.allclose(rh, 1.0 / np.sqrt(m + EPS), rtol=1e-14)
    # H = -k flips the gate
    _, _, alpha2, *_ = oracle.gateconv_fwd(H, -H, v, wh, wv, cw)
    assert np.allclose(alpha2, 1.0 / (1.0 + np.exp(z)), rtol=1e-14)


def test_zero_value():
    rng = np.random.default_rng(3)
    M, T, d = 2, 5, 16
    H, k, _, wh, wv, cw = rand_case(rng, M, T, d)
    v = np.zeros((M, T, d))
    Y, vhat, alpha, rh, rk, rv = oracle.gateconv_fwd(H, k, v, wh, wv, cw)
    assert np.all(Y == 0.0) and np.all(vhat == 0.0)
    assert np.allclose(rv, 1.0 / math.sqrt(EPS), rtol=1e-14)
    dY = rng.standard_normal((M, T, d))
    dH, dk, dv, dwh, dwv, dcw = oracle.gateconv_bwd(dY, H, k, v, wh, wv, cw, vhat, alpha,
                                                    rh, rk, rv)
    assert np.all(dH == 0.0) and np.all(dk == 0.0) and np.all(dwh == 0.0)
    # u = 0 so c = 0 and SiLU'(0) = 1/2: dc = dY/2; du_t = sum_j cw_j dc_{t+3-j};
    # uh = 0 leaves only the scale path of the norm: dvhat = dY + rrms_v*wv*du
    dc = 0.5 * dY
    du = np.zeros_like(dY)
    for j in range(4):
        lag = 3 - j
        du[:, :T - lag] += cw[j] * dc[:, lag:]
    expect = alpha[..., None] * (dY + rv[..., None] * wv * du)
    assert np.allclose(dv, expect, rtol=1e-13, atol=1e-12)


def test_causality_and_row_independence():
    rng = np.random.default_rng(4)
    M, T, d = 3, 10, 8
    H, k, v, wh, wv, cw = rand_case(rng, M, T, d)
    base = oracle.gateconv_fwd(H, k, v, wh, wv, cw)
    for arr in (H, k, v):
        a2 = arr.copy()
        a2[1, 6] += 0.7
        args = [H, k, v]
        args[[H is arr, k is arr, v is arr].index(True)] = a2
        out = oracle.gateconv_fwd(*args, wh, wv, cw)
        for b, o in zip(base, out):
            assert np.array_equal(b[1, :6], o[1, :6])   # earlier tokens untouched
            assert np.array_equal(b[0], o[0])           # other rows untouched
            assert np.array_equal(b[2], o[2])
        # the change reaches at most three tokens ahead through the conv
        assert np.array_equal(base[0][1, 10:], out[0][1, 10:])


def _fd_check(f, theta, analytic, rel=1e-6):
    flat = theta.reshape(-1)
    an = analytic.reshape(-1)
    scale = np.max(np.abs(an))
    worst = 0.0
    for i in range(flat.size):
        h = 1e-4 * max(1.0, abs(flat[i]))
        old = flat[i]
        vals = []
        for kk in (2, 1, -1, -2):
            flat[i] = old + kk * h
            vals.append(f())
        flat[i] = old
        fd = (-vals[0] + 8 * vals[1] - 8 * vals[2] + vals[3]) / (12 * h)
        worst = max(worst, abs(fd - an[i]) / max(abs(an[i]), 1e-3 * scale))
    assert worst < rel, worst


@pytest.mark.parametrize("M,T,d", [(1, 6, 8), (2, 5, 16), (1, 4, 32)])
def test_backward_matches_finite_differences(M, T, d):
    rng = np.random.default_rng(50 + d)
    H, k, v, wh, wv, cw = rand_case(rng, M, T, d)
    dY = rng.standard_normal((M, T, d))

    def loss():
        Y, *_ = oracle.gateconv_fwd(H, k, v, wh, wv, cw)
        return float(np.sum(Y * dY))

    Y, vhat, alpha, rh, rk, rv = oracle.gateconv_fwd(H, k, v, wh, wv, cw)
    dH, dk, dv, dwh, dwv, dcw = oracle.gateconv_bwd(dY, H, k, v, wh, wv, cw, vhat, alpha,
                                                    rh, rk, rv)
    for theta, an in ((H, dH), (k, dk), (v, dv), (wh, dwh), (wv, dwv), (cw, dcw)):
        _fd_check(loss, theta, an)


@pytest.mark.parametrize("M,T,d,seed", [(2, 11, 16, 31), (1, 3, 8, 32), (3, 40, 24, 33)])
def test_conv_is_the_standard_causal_depthwise_conv1d(M, T, d, seed):
    """The page names the op's middle stage a causal depthwise conv1d with
    (4, d) weights.  The standard form of that layer is PyTorch's grouped
    Conv1d (groups = d, one 4-tap filter per channel, no bias) applied with
    3 zeros of left padding and the output cut to the first T positions, i.e.
    a cross-correlation in which tap j multiplies the input 3 - j steps back
    (tap 3 the current token).  Here torch's fp64 conv1d, an implementation
    written independently of the oracle, recomputes Y = SiLU(conv(u)) + vhat
    from the oracle's own u = vhat rrms_v w_v, so the tap order, the causal
    padding and the per-row reset are pinned to that convention."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(seed)
    H, k, v, wh, wv, cw = rand_case(rng, M, T, d)
    Y, vhat, alpha, rh, rk, rv = oracle.gateconv_fwd(H, k, v, wh, wv, cw)
    u = torch.from_numpy(vhat * rv[..., None] * wv)                 # (M, T, d)
    x = u.permute(0, 2, 1)                                           # (M, d, T)
    x = torch.nn.functional.pad(x, (3, 0))                           # causal left padding
    w = torch.from_numpy(cw.T.copy()).unsqueeze(1)                  # (d, 1, 4): tap j at index j
    c = torch.nn.functional.conv1d(x, w, groups=d)[..., :T]          # (M, d, T)
    c = c.permute(0, 2, 1).numpy()
    assert np.allclose(Y, silu(c) + vhat, rtol=1e-13, atol=1e-14)
