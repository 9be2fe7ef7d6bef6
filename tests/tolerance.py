"""Comparison rules between the CUDA path and the fp64 oracle.

bf16 tensors (out, grad_x, grad_kv, Y, vhat, dH, dk, dv):
    |gpu - exact| <= 2^-7 |exact| + 2^-16 rms(row of exact)
  2^-7 = 7.8e-3 is "within one bf16 ulp" (the ulp of a bf16 value is at most
  2^-7 of it).  The second term is the near-zero allowance: a value formed in
  fp32 from terms of the row's magnitude that cancel cannot be resolved below
  about 2^-23 of those terms; 2^-16 of the row's RMS leaves a 100x margin and
  is still far below one ulp of any typical element.  A row whose exact
  values are all zero must match exactly.
GateConv's dH and dk take the near-zero allowance from the rms over the whole
compared slice instead of the token's row.  Both are the token's scalar dz
times per-element terms, and dz = dalpha alpha (1 - alpha) with dalpha =
sum_i dvhat_i v_i, which the kernel forms in fp32 as a difference of row sums
(the RMSNorm of vhat makes them cancel).  The rounding error of dz therefore
scales with those sums, i.e. with the dz of a typical token, not with the
token's own dz: a token whose dalpha happens to cancel to 1e-4 of its terms
has a row 1e4 times below the others with a relative error of a few percent
and an absolute error of a few 2^-23 of the typical row.  2^-16 of the slice's
rms bounds that with a wide margin and stays 2^-8 below one ulp of any typical
element.
fp32 tensors (saved gate/dot/rstd, grad_weight, alpha, rrms_*):
    |gpu - exact| <= 1e-4 |exact| + 1e-6
fp32 weight gradients of GateConv, summed over up to 65536 tokens:
    |gpu - exact| <= 1e-4 |exact| + 1e-6 max(1, max|exact|)
  (the near-zero allowance scales with the magnitude of the summed vector,
  because fp32 partial sums of that magnitude carry rounding of that order).
Every check records its worst diff/tol ratio per name in WORST, with the
number of elements that only the near-zero term kept inside the bound.
"""
from __future__ import annotations

import numpy as np

# Worst |gpu - exact| / tol seen per checked name in this process (1.0 = at
# the tolerance).  The test session prints it at the end, so a run shows how
# close each output family comes to its bound and whether the near-zero
# allowances are ever what keeps an element inside it.
WORST: dict = {}


def _record(name, diff, tol, floor_only=None):
    if diff.size == 0:
        return 0.0
    r = diff / np.maximum(tol, 1e-300)
    worst = float(np.max(r))
    prev = WORST.get(name)
    # elements inside the bound only thanks to the near-zero allowance
    floor_hits = int(np.count_nonzero(floor_only)) if floor_only is not None else 0
    if prev is None:
        WORST[name] = [worst, floor_hits, int(diff.size)]
    else:
        prev[0] = max(prev[0], worst)
        prev[1] += floor_hits
        prev[2] += int(diff.size)
    return worst

BF16_REL = 2.0 ** -7
ROW_FLOOR = 2.0 ** -16
F32_REL = 1e-4
F32_ABS = 1e-6


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits).view(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _report(name, got, exact, tol, bad):
    idx = np.argwhere(bad)[:5]
    lines = [f"{name}: {int(bad.sum())} of {bad.size} elements out of tolerance"]
    for i in idx:
        t = tuple(int(v) for v in i)
        lines.append(f"  at {t}: got {got[t]!r} exact {exact[t]!r} tol {tol[t]!r}")
    return "\n".join(lines)


def check_bf16(name, got_bits, exact, row_axis=-1, floor="row"):
    """floor="row": near-zero allowance from the rms of each row (token);
    floor="all": from the rms of the whole compared array (see the module
    docstring: GateConv's dH and dk)."""
    got = bf16_bits_to_f64(got_bits).reshape(exact.shape)
    if floor == "all":
        rms = np.sqrt(np.mean(exact * exact)) if exact.size else 0.0
    else:
        rms = np.sqrt(np.mean(exact * exact, axis=row_axis, keepdims=True))
    rel_tol = BF16_REL * np.abs(exact)
    tol = rel_tol + ROW_FLOOR * rms
    diff = np.abs(got - exact)
    bad = ~(diff <= tol)
    assert not bad.any(), _report(name, got, exact, tol, bad)
    return _record(name, diff, tol, diff > rel_tol)


def check_f32(name, got, exact, rel=F32_REL, abs_=F32_ABS):
    got = np.asarray(got, dtype=np.float64).reshape(exact.shape)
    rel_tol = rel * np.abs(exact)
    tol = rel_tol + abs_
    diff = np.abs(got - exact)
    bad = ~(diff <= tol)
    assert not bad.any(), _report(name, got, exact, tol, bad)
    return _record(name, diff, tol, diff > rel_tol)


def check_f32_sum(name, got, exact):
    scale = max(1.0, float(np.max(np.abs(exact)))) if exact.size else 1.0
    r = check_f32(name, got, exact, F32_REL, F32_ABS * scale)
    # also recorded against the plain abs 1e-6 floor, to show whether the
    # magnitude-scaled floor is ever needed
    got64 = np.asarray(got, dtype=np.float64).reshape(exact.shape)
    diff = np.abs(got64 - exact)
    plain = F32_REL * np.abs(exact) + F32_ABS
    _record(name + " [plain 1e-6 floor]", diff, plain, diff > F32_REL * np.abs(exact))
    return r
