"""Pins for the GateConv decode oracle (TileOPs "Engram Operators", Decode
section, EngramDecodeFwdOp).  The page gives the interface only; the readings
are the GateConv ones.  Pinned here without re-typing the formula:
  * chaining decode steps from an empty cache reproduces the GateConv forward
    oracle (written separately, pinned by its own tests) token by token;
  * a conv with dilation delta equals the dense conv whose taps sit every
    delta positions (zeros between);
  * a single nonzero tap reads exactly the cached token at its lag (or the
    current token, or zero beyond the cache);
  * the cache update is a one-token shift of the left-padded cache;
  * the dilated taps against the standard causal conv1d (torch's grouped
    Conv1d with dilation and left padding, written independently of the
    oracle), which fixes the tap order at every dilation.
"""
import numpy as np
import pytest

import oracle


def sig(z):
    return 1.0 / (1.0 + np.exp(-z))


def weights(rng, d, w):
    return (1.0 + 0.1 * rng.standard_normal(d), 1.0 + 0.1 * rng.standard_normal(d),
            0.5 * rng.standard_normal((w, d)))


@pytest.mark.parametrize("T,d", [(7, 16), (5, 64)])
def test_decode_steps_reproduce_gateconv_forward(T, d):
    rng = np.random.default_rng(T)
    H = rng.standard_normal((1, T, d))
    k = rng.standard_normal((1, T, d))
    v = rng.standard_normal((1, T, d))
    wh, wv, cw = weights(rng, d, 4)
    Y, *_ = oracle.gateconv_fwd(H, k, v, wh, wv, cw)
    # e = [k, v] with W_K = [I; 0], W_V = [0; I] projects to exactly k and v
    WK = np.concatenate([np.eye(d), np.zeros((d, d))])
    WV = np.concatenate([np.zeros((d, d)), np.eye(d)])
    state = np.zeros((1, 0, d))
    for t in range(T):
        e = np.concatenate([k[:, t], v[:, t]], axis=1)
        y, state = oracle.decode_fwd(e, H[:, t], state, WK, WV, wh, wv, cw, max_len=3, dilation=1)
        assert np.allclose(y, Y[:, t], rtol=1e-12, atol=1e-14)


def test_dilation_equals_dense_conv_with_zero_taps():
    rng = np.random.default_rng(3)
    B, dmem, d, w, dil, L = 2, 24, 16, 4, 3, 9
    e, h = rng.standard_normal((B, dmem)), rng.standard_normal((B, d))
    WK, WV = rng.standard_normal((dmem, d)), rng.standard_normal((dmem, d))
    wh, wv, cw = weights(rng, d, w)
    st = rng.standard_normal((B, L, d))
    dense = np.zeros(((w - 1) * dil + 1, d))
    dense[::dil] = cw
    y1, s1 = oracle.decode_fwd(e, h, st, WK, WV, wh, wv, cw, max_len=L, dilation=dil)
    y2, s2 = oracle.decode_fwd(e, h, st, WK, WV, wh, wv, dense, max_len=L, dilation=1)
    assert np.array_equal(y1, y2) and np.array_equal(s1, s2)


@pytest.mark.parametrize("L", [0, 2, 5, 8])
def test_single_tap_reads_the_lagged_token(L):
    rng = np.random.default_rng(10 + L)
    B, dmem, d, w, dil, max_len = 2, 12, 16, 4, 2, 8
    e, h = rng.standard_normal((B, dmem)), rng.standard_normal((B, d))
    WK, WV = rng.standard_normal((dmem, d)), rng.standard_normal((dmem, d))
    wh, wv, _ = weights(rng, d, w)
    st = rng.standard_normal((B, L, d))
    y0, s0 = oracle.decode_fwd(e, h, st, WK, WV, wh, wv, np.zeros((w, d)), max_len=max_len, dilation=dil)
    vhat = y0                      # zero taps: SiLU(0) = 0, y = vhat
    u_t = s0[:, -1]
    for j in range(w):
        cw = np.zeros((w, d))
        cw[j] = 0.7
        y, _ = oracle.decode_fwd(e, h, st, WK, WV, wh, wv, cw, max_len=max_len, dilation=dil)
        lag = (w - 1 - j) * dil
        src = u_t if lag == 0 else (st[:, L - lag] if lag <= L else np.zeros((B, d)))
        c = 0.7 * src
        assert np.allclose(y - vhat, c * sig(c), rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("L,max_len", [(0, 4), (3, 6), (6, 6)])
def test_cache_update_is_a_one_token_shift(L, max_len):
    rng = np.random.default_rng(L * 7 + max_len)
    B, dmem, d = 3, 8, 16
    e, h = rng.standard_normal((B, dmem)), rng.standard_normal((B, d))
    WK, WV = rng.standard_normal((dmem, d)), rng.standard_normal((dmem, d))
    wh, wv, cw = weights(rng, d, 4)
    st = rng.standard_normal((B, L, d))
    _, s = oracle.decode_fwd(e, h, st, WK, WV, wh, wv, cw, max_len=max_len, dilation=1)
    padded = np.concatenate([np.zeros((B, max_len - L, d)), st], axis=1)
    assert np.array_equal(s[:, :-1], padded[:, 1:])
    # the new last row is this token's conv input: rms 1 after w_v is divided out
    u = s[:, -1] / wv
    assert np.allclose(np.sqrt(np.mean(u * u, axis=1)), 1.0, rtol=1e-5)


@pytest.mark.parametrize("w,dil,L,max_len,seed", [(4, 1, 6, 8, 41), (4, 3, 12, 16, 42),
                                                  (3, 2, 2, 8, 43), (5, 4, 16, 16, 44)])
def test_dilated_tap_order_is_the_standard_causal_conv1d(w, dil, L, max_len, seed):
    """The page's decode step is a dilated depthwise conv over the cached conv
    inputs.  The standard causal form is PyTorch's grouped Conv1d with
    dilation delta and (w - 1) delta zeros of left padding: at the last
    position, tap j multiplies the input (w - 1 - j) delta steps back.  torch's
    fp64 conv1d, applied to the sequence [cache rows oldest first, this
    token's u], recomputes y = SiLU(c) + vhat from the oracle's own u (read
    back from the last row of the new cache), which pins the tap order, the
    dilation and the zero reads beyond the cache to that convention."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(seed)
    B, dmem, d = 2, 8, 16
    e = rng.standard_normal((B, dmem))
    h = rng.standard_normal((B, d))
    state = rng.standard_normal((B, L, d))
    WK = rng.standard_normal((dmem, d)) / np.sqrt(dmem)
    WV = rng.standard_normal((dmem, d)) / np.sqrt(dmem)
    wh, wv, cw = weights(rng, d, w)
    y, ns = oracle.decode_fwd(e, h, state, WK, WV, wh, wv, cw, max_len, dil)
    u = ns[:, -1]                                                   # this token's u
    k = e @ WK
    v = e @ WV
    rh = 1.0 / np.sqrt(np.mean(h * h, axis=1) + oracle.GATECONV_EPS)
    rk = 1.0 / np.sqrt(np.mean(k * k, axis=1) + oracle.GATECONV_EPS)
    alpha = sig(np.sum((h * rh[:, None] * wh) * (k * rk[:, None] * wh), axis=1) / np.sqrt(d))
    vhat = alpha[:, None] * v
    seq = np.concatenate([state, u[:, None]], axis=1)               # (B, L + 1, d)
    x = torch.from_numpy(seq).permute(0, 2, 1)                       # (B, d, L + 1)
    x = torch.nn.functional.pad(x, ((w - 1) * dil, 0))
    wt = torch.from_numpy(cw.T.copy()).unsqueeze(1)                 # (d, 1, w)
    c = torch.nn.functional.conv1d(x, wt, groups=d, dilation=dil)[..., -1].numpy()
    assert np.allclose(y, c / (1.0 + np.exp(-c)) + vhat, rtol=1e-12, atol=1e-13)
