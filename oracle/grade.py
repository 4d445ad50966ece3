"""Comparing a BF16 result with the oracle.

Two measures are reported for every element:

* ``raw``: the distance in BF16 units in the last place between the two
  values (the number of representable BF16 values between them, signed
  zeros equal).
* ``graded``: |y - y_oracle| divided by the BF16 spacing at
  max(|y64|, 2**-8 * A), where y64 is the oracle's unrounded value and A its
  magnitude scale (sum of |terms|).  An implementation that accumulates in
  FP32 errs by about 2**-24 * sqrt(n) * A, so an element whose exact value
  nearly cancels (|y64| much smaller than A) cannot be expected within 2 raw
  ulp; the floor 2**-8 * A keeps the criterion a forward-error bound there.

Where the operator has an inner BF16 write boundary (the FFN hidden slice),
a correct FP32 evaluation may round an inner value the other way when the
exact value lies within the FP32 error bound of a rounding boundary; the
oracle's ``slack`` is the largest effect such flips can have on each output
and is subtracted from |y - y_oracle| before grading.  ``n_pass_by_slack``
counts the elements that are within tolerance only because of it.

The tolerance is ``graded <= 2`` for every element; raw violations are listed
with their condition number A / |y64|.  Normwise errors: max|dy| / max|y| and
relative L2, the measure used in section IV-B of the paper.
"""
from __future__ import annotations

import numpy as np

from .bf16 import encode, ulp


def _ordered(bits):
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def raw_ulps(y, y_ref) -> np.ndarray:
    """Distance in BF16 ulps between two arrays of BF16 values (float64)."""
    return np.abs(_ordered(encode(y)) - _ordered(encode(y_ref)))


def graded_ulps(y, y_ref, y64, A, slack=None) -> np.ndarray:
    scale = np.maximum(np.abs(np.asarray(y64)), np.ldexp(np.asarray(A, np.float64), -8))
    d = np.abs(np.asarray(y, np.float64) - np.asarray(y_ref, np.float64))
    if slack is not None:
        d = np.maximum(d - np.asarray(slack, np.float64), 0.0)
    return d / ulp(scale)


def _slack_used(y, ref, res) -> int:
    slack = getattr(res, "slack", None)
    if slack is None:
        return 0
    return int(np.count_nonzero((np.abs(y - ref) > 0) & (slack > 0)))


def _pass_by_slack(y, res, tol) -> int:
    """Elements within tolerance only because of the slack: graded above
    ``tol`` without it and at most ``tol`` with it."""
    slack = getattr(res, "slack", None)
    if slack is None:
        return 0
    with_s = graded_ulps(y, res.y, res.y64, res.A, slack)
    without = graded_ulps(y, res.y, res.y64, res.A)
    return int(np.count_nonzero((without > tol) & (with_s <= tol)))


def report(y, res, tol_ulps: float = 2.0) -> dict:
    """Compare BF16 values ``y`` (float64 array) with an oracle ``Result``."""
    y = np.asarray(y, np.float64)
    ref = res.y
    if y.shape != ref.shape:
        raise ValueError(f"shape mismatch {y.shape} vs {ref.shape}")
    finite = np.isfinite(y)
    g = graded_ulps(y, ref, res.y64, res.A, getattr(res, "slack", None))
    r = raw_ulps(np.where(finite, y, 0.0), ref)
    diff = np.abs(y - ref)
    denom = max(float(np.max(np.abs(ref))), 1e-300)
    l2 = float(np.linalg.norm((y - res.y64).ravel()) /
               max(float(np.linalg.norm(res.y64.ravel())), 1e-300))
    bad = np.argwhere(r > tol_ulps)
    cond = res.A / np.maximum(np.abs(res.y64), 1e-300)
    return {
        "n": int(y.size),
        "all_finite": bool(finite.all()),
        "max_graded_ulps": float(g.max()) if g.size else 0.0,
        "n_slack_used": _slack_used(y, ref, res),
        "n_pass_by_slack": _pass_by_slack(np.where(finite, y, 0.0), res, tol_ulps),
        "max_raw_ulps": int(r.max()) if r.size else 0,
        "n_raw_gt_tol": int(len(bad)),
        "n_differing": int(np.count_nonzero(r)),
        "raw_violations": [(tuple(int(v) for v in ij), int(r[tuple(ij)]),
                            float(cond[tuple(ij)])) for ij in bad[:20]],
        "max_rel_err": float(diff.max()) / denom if diff.size else 0.0,
        "rel_l2": l2,
        "pass": bool(finite.all() and (g.size == 0 or g.max() <= tol_ulps)),
    }
