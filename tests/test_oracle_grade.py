"""Pins of the oracle's comparator (oracle/grade.py), CPU only.

Every GPU parity test passes through ``grade.report``, so its pieces are
checked here against values worked by hand: the raw BF16 ulp distance
(signed zeros, sign changes, the subnormal/normal boundary, whole binades),
the graded distance with its 2^-8 * A floor (cases one step inside and one
step outside the 2-ulp tolerance, where a wrong floor exponent or a wrong
ulp would flip the verdict), the slack subtraction, and the normwise error
measures of section IV-B.
"""
import numpy as np
import pytest

from oracle import grade, ops

E = np.ldexp


def test_raw_ulps_hand_values():
    cases = [
        (0.0, -0.0, 0),                  # signed zeros are equal
        (1.0, 1.0078125, 1),             # 1 and 1 + 2^-7, its upper neighbour
        (1.0, 0.99609375, 1),            # 1 and 1 - 2^-8, its lower neighbour
        (2.0, 1.0, 128),                 # one binade holds 128 BF16 values
        (-1.0, 1.0, 2 * 0x3F80),         # across zero: both halves counted
        (E(1.0, -133), -E(1.0, -133), 2),  # the two smallest subnormals
        (E(127.0, -133), E(1.0, -126), 1),  # largest subnormal, smallest normal
        (0.0, E(1.0, -126), 128),        # 127 subnormals lie in between
        (-3.0, -3.5, 32),                # negative values: magnitude order
    ]
    for a, b, want in cases:
        assert int(grade.raw_ulps(np.array([a]), np.array([b]))[0]) == want, (a, b)
        assert int(grade.raw_ulps(np.array([b]), np.array([a]))[0]) == want, (b, a)


def test_graded_ulps_floor_decides_pass_and_fail():
    """|y64| = 2^-20 with A = 1: the floor 2^-8 * A sets the scale, whose
    BF16 spacing is 2^-15.  Offsets of 63/32 and 65/32 spacings fall on either
    side of the 2-ulp tolerance; with the floor taken at 2^-7 or 2^-9 A, or
    without it, the verdicts would change."""
    y64 = np.array([E(1.0, -20)])
    A = np.array([1.0])
    ref = y64.copy()
    inside = ref + E(63 / 32, -15)
    outside = ref + E(65 / 32, -15)
    assert grade.graded_ulps(inside, ref, y64, A)[0] == 63 / 32
    assert grade.graded_ulps(outside, ref, y64, A)[0] == 65 / 32
    # where |y64| is above the floor it sets the scale: ulp(3) = 2^-6
    g = grade.graded_ulps(np.array([3.0 + E(1.0, -5)]), np.array([3.0]), np.array([3.0]),
                          np.array([4.0]))
    assert g[0] == 2.0
    # no floor when A is small: the 2^-20 value's own spacing 2^-27 applies
    g = grade.graded_ulps(inside, ref, y64, np.array([E(1.0, -20)]))
    assert g[0] == 63 / 32 * 2 ** 12


def test_graded_ulps_spacing_at_a_binade_edge():
    # at exactly 1 the spacing is 2^-7 (the values above 1), just below it 2^-8
    one = grade.graded_ulps(np.array([1.0 + E(1.0, -7)]), np.array([1.0]), np.array([1.0]),
                            np.array([1.0]))
    below = grade.graded_ulps(np.array([0.99609375 + E(1.0, -8)]), np.array([0.99609375]),
                              np.array([0.9990234375]), np.array([1.0]))
    assert one[0] == 1.0 and below[0] == 1.0


def test_graded_ulps_slack_is_subtracted():
    y64 = np.array([E(1.0, -20)] * 3)
    A = np.ones(3)
    ref = y64.copy()
    y = ref + E(2.5, -15)
    slack = np.array([E(0.625, -15), E(0.375, -15), E(4.0, -15)])
    g = grade.graded_ulps(y, ref, y64, A, slack)
    assert list(g) == [1.875, 2.125, 0.0]
    assert grade.graded_ulps(y, ref, y64, A)[0] == 2.5


def test_report_counts_and_normwise_errors():
    """Four elements: exact, one spacing off, three spacings off with a slack
    that brings it to 1.875, and (second call) three spacings off without
    slack."""
    ref = np.array([[1.0, 2.0, 1.0, -1.0]])
    y64 = ref.copy()
    A = np.ones_like(ref)
    res = ops.Result(y=ref.copy(), y64=y64, A=A,
                     slack=np.array([[0.0, 0.0, E(1.125, -7), 0.0]]))
    y = np.array([[1.0, 2.0 + E(1.0, -6), 1.0 + E(3.0, -7), -1.0]])
    rep = grade.report(y, res)
    assert rep["pass"] and rep["n_pass_by_slack"] == 1
    assert rep["max_raw_ulps"] == 3 and rep["n_differing"] == 2 and rep["n_raw_gt_tol"] == 1
    assert rep["max_graded_ulps"] == 1.875
    # normwise: max|dy| / max|y| and the relative L2 against y64
    assert rep["max_rel_err"] == E(3.0, -7) / 2.0
    assert rep["rel_l2"] == pytest.approx(np.sqrt(E(1.0, -12) + E(9.0, -14)) / np.sqrt(7.0))
    y[0, 3] = -1.0 - E(3.0, -7)          # three spacings below -1, no slack there
    rep = grade.report(y, res)
    assert not rep["pass"] and rep["max_graded_ulps"] == 3.0
    res.slack = None
    rep = grade.report(np.array([[1.0, 2.0, 1.0 + E(3.0, -7), -1.0]]), res)
    assert not rep["pass"] and rep["n_pass_by_slack"] == 0
    # a non-finite output never passes
    rep = grade.report(np.array([[np.nan, 2.0, 1.0, -1.0]]), res)
    assert not rep["pass"] and not rep["all_finite"]
