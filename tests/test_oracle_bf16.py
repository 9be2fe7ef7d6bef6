"""Pins for the oracle's own bf16 conversion (round-to-nearest-even, one step).

bf16 is the top half of an IEEE binary32 word: 1 sign, 8 exponent and 7
stored mantissa bits.  The rounding is pinned against PyTorch's float32 ->
bfloat16 conversion (a library routine, exact for inputs that are float32
values) and against hand-worked ties, overflow, subnormal and NaN cases.
"""
import numpy as np
import pytest
import torch

import oracle


def test_widening_is_exact():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_round_matches_library_on_float32_values():
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(50000) * 1e30).astype(np.float32),
        (rng.standard_normal(50000) * 1e-38).astype(np.float32),   # subnormal range
        rng.integers(0, 1 << 32, 100000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    vals = vals[~np.isnan(vals)]
    got = oracle.round_bf16(vals.astype(np.float64))
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("value,bits", [
    (1.0, 0x3F80),
    (1.0 + 2.0 ** -8, 0x3F80),          # tie -> even (mantissa 0)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),      # tie -> even (mantissa 2)
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),  # just above the tie: fp64-only bits count
    (-2.5, 0xC020),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (2.0 ** -133, 0x0001),              # smallest bf16 subnormal
    (2.0 ** -134, 0x0000),              # tie between 0 and the smallest subnormal -> even
    (3 * 2.0 ** -134, 0x0002),          # tie between 1 and 2 quanta -> even (2)
    ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),    # largest finite bf16
    ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),    # tie above the largest finite -> inf
    ((2 - 2.0 ** -8 - 2.0 ** -30) * 2.0 ** 127, 0x7F7F),  # just below that tie
    (float("inf"), 0x7F80),
    (float("-inf"), 0xFF80),
])
def test_round_hand_cases(value, bits):
    assert int(oracle.round_bf16([value])[0]) == bits


def test_round_single_step_differs_from_double_rounding():
    # 1 + 2^-8 + 2^-30 is above the bf16 tie; rounding it first to fp32 gives
    # exactly the tie (ties-to-even -> 1.0).  The oracle rounds once.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert int(oracle.round_bf16([v])[0]) == 0x3F81
    assert torch.tensor(np.float32(v)).to(torch.bfloat16).view(torch.int16).item() == 0x3F80


def test_nan_keeps_sign():
    got = oracle.round_bf16([float("nan"), -float("nan")])
    assert (got[0] & 0x7F80) == 0x7F80 and (got[0] & 0x7F) != 0 and got[0] >> 15 == 0
    assert (got[1] & 0x7F80) == 0x7F80 and (got[1] & 0x7F) != 0 and got[1] >> 15 == 1
