"""Pins of the oracle's linear, FFN and attention (CPU only).

Each test checks the oracle against something other than itself: values
worked by hand (tests/golden), exact rational brute force, closed forms and
invariants of PSI section II-B (Eqs.(2)-(4)), and independent library
routines (torch CPU float64 linear, GELU and scaled-dot-product attention).
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import bf16, ops

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand_bf16(rng, shape, scale=1.0):
    return bf16.round_bf16(rng.standard_normal(shape) * scale)


# ----------------------------------------------------------------- linear --
def test_linear_hand_worked():
    g = json.load(open(os.path.join(GOLD, "linear_hand.json")))
    r = ops.linear(np.array(g["X"]), np.array(g["W"]), np.array(g["b"]))
    assert np.array_equal(r.y, np.array(g["Y"]))


def test_linear_exact_bruteforce_small_integers():
    """All sign patterns of a 2x3 @ 3x2 case with mantissa-sized entries,
    against the exact rational sum rounded once (section IV-B)."""
    base_x = np.array([[1.5, 0.75, 3.0], [0.1015625, 2.25, 0.5]])
    base_w = np.array([[0.375, 1.25, 0.0078125], [2.5, 0.5, 1.75]])
    b = np.array([0.0625, -1.0])
    for sx in itertools.product([1, -1], repeat=3):
        for sw in itertools.product([1, -1], repeat=3):
            X = base_x * np.array(sx)
            W = base_w * np.array(sw)
            r = ops.linear(X, W, b)
            for i in range(2):
                for j in range(2):
                    s = sum(Fraction(X[i, k]) * Fraction(W[j, k]) for k in range(3))
                    s += Fraction(b[j])
                    assert r.y[i, j] == bf16.round_fraction(s)


def test_linear_against_torch_fp64():
    rng = np.random.default_rng(0)
    X = _rand_bf16(rng, (13, 70))
    W = _rand_bf16(rng, (29, 70), 0.1)   # non-square: a transposed W fails
    b = _rand_bf16(rng, (29,), 0.02)
    R = _rand_bf16(rng, (13, 29))
    r = ops.linear(X, W, b, residual=R)
    ref = F.linear(torch.from_numpy(X), torch.from_numpy(W), torch.from_numpy(b)).numpy() + R
    assert np.allclose(r.y64, ref, rtol=0, atol=1e-12)
    assert np.array_equal(r.y, bf16.round_bf16(r.y64))


def test_linear_identity_and_single_term():
    rng = np.random.default_rng(1)
    x = _rand_bf16(rng, (5, 8))
    b = _rand_bf16(rng, (8,), 0.3)
    r = ops.linear(x, np.eye(8), b)
    assert np.array_equal(r.y, bf16.round_bf16(x + b))
    W = np.zeros((3, 8))
    W[1, 4] = 0.8125
    r = ops.linear(x, W, b[:3])
    assert np.array_equal(r.y[:, 1], bf16.round_bf16(x[:, 4] * 0.8125 + b[1]))
    assert np.array_equal(r.y[:, 0], np.full(5, b[0]))


def test_linear_exact_tie_resolution():
    """1 + 2^-8 + 2^-70: the float64 sum drops 2^-70 and lands on a tie; the
    exact sum lies above it and rounds up."""
    X = np.array([[1.0, 2.0**-8, 2.0**-70]])
    W = np.ones((1, 3))
    r = ops.linear(X, W, np.zeros(1))
    assert r.exact_fixed == 1 and r.y[0, 0] == 1.0 + 2.0**-7
    r2 = ops.linear(X, W, np.zeros(1), exact_ties=False)
    assert r2.y[0, 0] == 1.0   # what float64 alone would give


def test_linear_output_column_partition_bitwise():
    """Paging W by output rows (section II-A) is the same per-element sum."""
    rng = np.random.default_rng(2)
    X = _rand_bf16(rng, (9, 64))
    W = _rand_bf16(rng, (48, 64), 0.125)
    b = _rand_bf16(rng, (48,), 0.02)
    full = ops.linear(X, W, b).y
    parts = [ops.linear(X, W[p:p + 16], b[p:p + 16]).y for p in range(0, 48, 16)]
    assert np.array_equal(np.concatenate(parts, axis=1), full)


# -------------------------------------------------------------------- ffn --
def test_gelu_against_torch_and_identities():
    x = np.linspace(-12, 12, 4001)
    ref = F.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.allclose(ops.gelu_tanh(x), ref, rtol=1e-14, atol=1e-15)
    assert ops.gelu_tanh(0.0) == 0.0
    # phi(x) - phi(-x) = x for the tanh form
    assert np.allclose(ops.gelu_tanh(x) - ops.gelu_tanh(-x), x, rtol=0, atol=1e-14)


def test_ffn_hand_worked():
    g = json.load(open(os.path.join(GOLD, "ffn_hand.json")))
    r = ops.ffn(np.array(g["X"]), np.array(g["U"]), np.array(g["V"]),
                np.array(g["a"]), np.array(g["b"]))
    assert np.array_equal(r.H, np.array(g["H"]))
    assert np.array_equal(r.y, np.array(g["Y"]))


def test_ffn_against_torch_fp64():
    rng = np.random.default_rng(3)
    X = _rand_bf16(rng, (7, 40))
    U = _rand_bf16(rng, (96, 40), 1 / math.sqrt(40))
    V = _rand_bf16(rng, (24, 96), 1 / math.sqrt(96))
    a = _rand_bf16(rng, (96,), 0.02)
    b = _rand_bf16(rng, (24,), 0.02)
    r = ops.ffn(X, U, V, a, b)
    t = F.linear(torch.from_numpy(X), torch.from_numpy(U), torch.from_numpy(a))
    H = bf16.round_bf16(F.gelu(t, approximate="tanh").numpy())
    assert np.array_equal(r.H, H)
    y = F.linear(torch.from_numpy(H), torch.from_numpy(V), torch.from_numpy(b)).numpy()
    assert np.allclose(r.y64, y, rtol=0, atol=1e-12)


@pytest.mark.parametrize("nslices", [1, 2, 3, 6])
def test_ffn_hidden_partition_identity_exact(nslices):
    """Eq.(2): a complete disjoint hidden partition, exact down-projection
    sums, output bias once, equals the dense FFN rounded once."""
    rng = np.random.default_rng(4)
    X = _rand_bf16(rng, (2, 5))
    U = _rand_bf16(rng, (6, 5), 0.5)
    V = _rand_bf16(rng, (3, 6), 0.4)
    a = _rand_bf16(rng, (6,), 0.1)
    b = _rand_bf16(rng, (3,), 0.1)
    perm = rng.permutation(6)
    slices = [list(s) for s in np.array_split(perm, nslices)]
    y, H = ops.ffn_partitioned_exact(X, U, V, a, b, slices)
    dense = ops.ffn(X, U, V, a, b)
    assert np.array_equal(H, dense.H)
    assert np.array_equal(y, dense.y)


def test_ffn_pregelu_boundary_changes_result():
    """The paper's extra pre-GELU BF16 write (section III-A) is a declared
    boundary: with t = 257/256 + tiny, B(t) != t and the outputs differ."""
    X = np.array([[1.0, 2.0**-8, 2.0**-12]])
    U = np.array([[1.0, 1.0, 1.0]])
    V = np.array([[1.0]])
    z = np.zeros(1)
    r0 = ops.ffn(X, U, V, z, z)
    r1 = ops.ffn(X, U, V, z, z, pregelu_bf16=True)
    t = 1.0 + 2.0**-8 + 2.0**-12
    assert r0.H[0, 0] == bf16.round_bf16(ops.gelu_tanh(t))
    assert r1.H[0, 0] == bf16.round_bf16(ops.gelu_tanh(bf16.round_bf16(t)))
    assert r0.H[0, 0] != r1.H[0, 0]


# -------------------------------------------------------------- attention --
def test_attention_single_key_and_equal_keys():
    rng = np.random.default_rng(5)
    q = _rand_bf16(rng, (4, 16))
    k = _rand_bf16(rng, (1, 16))
    v = _rand_bf16(rng, (1, 16))
    r = ops.attention(q, k, v, 0.25)
    assert np.array_equal(r.y, np.repeat(v, 4, axis=0))
    K = np.repeat(k, 9, axis=0)
    V = np.repeat(v, 9, axis=0)
    r = ops.attention(q, K, V, 0.25)
    assert np.allclose(r.y64, np.repeat(v, 4, axis=0), rtol=1e-15, atol=0)


def test_attention_zero_query_is_mean():
    rng = np.random.default_rng(6)
    K = _rand_bf16(rng, (37, 8))
    V = _rand_bf16(rng, (37, 8))
    r = ops.attention(np.zeros((1, 8)), K, V, 1.0)
    assert np.allclose(r.y64[0], V.mean(axis=0), rtol=0, atol=1e-15)


def test_attention_two_keys_closed_form():
    q = np.array([[1.0, -2.0]])
    K = np.array([[0.5, 0.25], [-1.0, 1.5]])
    V = np.array([[3.0, -1.0], [0.5, 2.0]])
    alpha = 0.75
    s1, s2 = alpha * (0.5 - 0.5), alpha * (-1.0 - 3.0)
    w1 = 1.0 / (1.0 + math.exp(s2 - s1))
    want = w1 * V[0] + (1 - w1) * V[1]
    r = ops.attention(q, K, V, alpha)
    assert np.allclose(r.y64[0], want, rtol=1e-15, atol=1e-15)


def test_attention_against_torch_sdpa():
    rng = np.random.default_rng(8)
    Q = _rand_bf16(rng, (3, 50, 32))
    K = _rand_bf16(rng, (3, 70, 32))
    V = _rand_bf16(rng, (3, 70, 32))
    sc = 1 / math.sqrt(32)
    r = ops.attention_heads(Q, K, V, sc)
    ref = F.scaled_dot_product_attention(torch.from_numpy(Q), torch.from_numpy(K),
                                         torch.from_numpy(V), scale=sc).numpy()
    assert np.allclose(r.y64, ref, rtol=0, atol=1e-13)


def test_attention_key_permutation_invariant():
    rng = np.random.default_rng(9)
    Q = _rand_bf16(rng, (6, 16))
    K = _rand_bf16(rng, (40, 16))
    V = _rand_bf16(rng, (40, 16))
    p = rng.permutation(40)
    a = ops.attention(Q, K, V, 0.3).y64
    b = ops.attention(Q, K[p], V[p], 0.3).y64
    assert np.allclose(a, b, rtol=0, atol=1e-14)


@pytest.mark.parametrize("kb", [1, 3, 64, 256, 300])
def test_online_softmax_equals_dense(kb):
    """Eqs.(3)-(4): any complete key partition gives the dense result (within
    the float64 bound)."""
    rng = np.random.default_rng(10)
    Q = _rand_bf16(rng, (17, 24))
    K = _rand_bf16(rng, (300, 24))
    V = _rand_bf16(rng, (300, 24))
    sc = 1 / math.sqrt(24)
    dense = ops.attention(Q, K, V, sc)
    y, o64 = ops.attention_online(Q, K, V, sc, kb)
    assert np.allclose(o64, dense.y64, rtol=0, atol=1e-13)


def test_attention_rows_subset():
    rng = np.random.default_rng(11)
    Q = _rand_bf16(rng, (20, 8))
    K = _rand_bf16(rng, (30, 8))
    V = _rand_bf16(rng, (30, 8))
    full = ops.attention(Q, K, V, 0.5)
    sub = ops.attention(Q, K, V, 0.5, rows=[3, 17])
    assert np.array_equal(sub.y, full.y[[3, 17]])


def test_attention_needs_a_key():
    with pytest.raises(ValueError):
        ops.attention(np.zeros((1, 4)), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)


def test_ffn_hidden_rounding_slack():
    """A hidden pre-activation placed within 2^-26 of the value whose GELU is
    the midpoint between the BF16 neighbours 1 and 1 + 2^-7: an FP32
    evaluation may round H either way.  The output nearly cancels, so the
    other rounding moves y by ~60 graded ulps; the oracle's slack covers it,
    and without the slack the same output would fail."""
    from oracle import grade
    mid = 1.0 + 2.0 ** -8
    t = 1.1
    for _ in range(80):                    # Newton on phi(t) = mid, float64
        eps = 1e-7
        d = (ops.gelu_tanh(t + eps) - ops.gelu_tanh(t - eps)) / (2 * eps)
        t -= (float(ops.gelu_tanh(t)) - mid) / d
    u = []
    rest = t
    for _ in range(3):                     # t as a sum of three BF16 values
        u.append(float(bf16.round_bf16(rest)))
        rest -= u[-1]
    assert abs(rest) < 2.0 ** -26
    X = np.array([[1.0, 1.0, 1.0]])
    U = np.array([u, [2.0, 0.0, 0.0]])
    h2 = float(bf16.round_bf16(ops.gelu_tanh(2.0)))
    V = np.array([[1.0, float(bf16.round_bf16(-1.0 / h2))]])
    r = ops.ffn(X, U, V, np.zeros(2), np.zeros(1))
    h1 = r.H[0, 0]
    assert h1 in (1.0, 1.0078125)
    assert r.slack[0, 0] == 2.0 ** -7      # one BF16 ulp at 1, times |v| = 1
    other = 1.0078125 if h1 == 1.0 else 1.0
    y_alt = bf16.round_bf16(np.array([[other * V[0, 0] + r.H[0, 1] * V[0, 1]]]))
    assert grade.report(y_alt, r)["pass"]
    r.slack = None
    assert not grade.report(y_alt, r)["pass"]
    g = json.load(open(os.path.join(GOLD, "ffn_hand.json")))
    r0 = ops.ffn(np.array(g["X"]), np.array(g["U"]), np.array(g["V"]),
                 np.array(g["a"]), np.array(g["b"]))
    # t = 8 has an unambiguous rounding; t = 0 = 1 - 1 only a tiny one
    t0 = np.array(g["X"]) @ np.array(g["U"]).T
    jump = ops.hidden_rounding_jump(t0, np.abs(np.array(g["X"])) @ np.abs(np.array(g["U"])).T,
                                    r0.H)
    assert jump[0, 1] == 0 and jump[0, 0] < 2.0 ** -20


def test_ffn_slack_is_small_on_random_inputs():
    """The slack is a small correction: a fraction of a percent of the hidden
    values are ambiguous, and it never exceeds 2^-7 of the output scale."""
    rng = np.random.default_rng(12)
    X = _rand_bf16(rng, (16, 256))
    U = _rand_bf16(rng, (512, 256), 1 / 16)
    V = _rand_bf16(rng, (64, 512), 1 / math.sqrt(512))
    r = ops.ffn(X, U, V, np.zeros(512), np.zeros(64))
    t = X @ U.T
    At = np.abs(X) @ np.abs(U).T
    jump = ops.hidden_rounding_jump(t, At, r.H)
    assert np.count_nonzero(jump) < 0.02 * jump.size
    assert np.all(r.slack <= 2.0 ** -7 * r.A)


# ----------------------------------------------- baseline numerics variant --
def test_linear_bias_after_bf16_worked():
    """The rounding mechanism of section II-C Eq.(5) on a projection: the
    product 1 + 2^-9 rounds to 1 before the bias 2^-8 is added (baseline
    order, a tie that goes to even: 1), while adding the bias first gives
    1 + 3*2^-9, which rounds to 1 + 2^-7 (modified order)."""
    X = np.array([[1.0, 2.0 ** -9]])
    W = np.array([[1.0, 1.0]])
    b = np.array([2.0 ** -8])
    assert ops.linear(X, W, b, bias_after_bf16=True).y[0, 0] == 1.0
    assert ops.linear(X, W, b).y[0, 0] == 1.0 + 2.0 ** -7


def test_linear_bias_after_bf16_against_definition():
    rng = np.random.default_rng(21)
    X = _rand_bf16(rng, (9, 33))
    W = _rand_bf16(rng, (12, 33), 0.2)
    b = _rand_bf16(rng, (12,), 0.5)
    R = _rand_bf16(rng, (9, 12))
    r = ops.linear(X, W, b, residual=R, bias_after_bf16=True)
    p = F.linear(torch.from_numpy(X), torch.from_numpy(W)).numpy()
    want = bf16.round_bf16(bf16.round_bf16(p) + b + R)
    assert np.array_equal(r.y, want)


def test_ffn_bias_after_bf16_against_definition():
    rng = np.random.default_rng(22)
    X = _rand_bf16(rng, (5, 24))
    U = _rand_bf16(rng, (40, 24), 0.2)
    V = _rand_bf16(rng, (16, 40), 0.15)
    a = _rand_bf16(rng, (40,), 0.1)
    b = _rand_bf16(rng, (16,), 0.1)
    r = ops.ffn(X, U, V, a, b, pregelu_bf16=True, bias_after_bf16=True)
    t = bf16.round_bf16(bf16.round_bf16(X @ U.T) + a)
    H = bf16.round_bf16(F.gelu(torch.from_numpy(t), approximate="tanh").numpy())
    assert np.array_equal(r.H, H)
    assert np.array_equal(r.y, bf16.round_bf16(bf16.round_bf16(H @ V.T) + b))


def test_attention_bf16_weights_definition():
    """Numerator weights rounded to BF16 relative to the running max; with a
    single key block this is sum B(e^{s-m}) v / sum e^{s-m}."""
    rng = np.random.default_rng(23)
    Q = _rand_bf16(rng, (7, 16))
    K = _rand_bf16(rng, (50, 16))
    V = _rand_bf16(rng, (50, 16))
    sc = 0.25
    r = ops.attention_bf16_weights(Q, K, V, sc, key_block=50)
    S = sc * Q @ K.T
    P = np.exp(S - S.max(axis=1, keepdims=True))
    want = (bf16.round_bf16(P) @ V) / P.sum(axis=1, keepdims=True)
    assert np.allclose(r.y64, want, rtol=0, atol=1e-14)
    # one key: weight exactly 1
    r1 = ops.attention_bf16_weights(Q, K[:1], V[:1], sc, key_block=128)
    assert np.array_equal(r1.y, np.repeat(V[:1], 7, axis=0))
    # the BF16 weights move the result by about 2^-9 of its scale, the FP32
    # ones do not
    dense = ops.attention(Q, K, V, sc)
    d = np.abs(r.y64 - dense.y64).max() / np.abs(dense.y64).max()
    assert 1e-5 < d < 2.0 ** -6


def _bf16_weights_closed_form(Q, K, V, sc, kb, mp):
    """The numerator/denominator of the BF16-weights recurrence unrolled: a
    key j of block t gets the weight B(e^{s_j - m_t}) relative to the running
    max m_t after block t, and the later rescales multiply it by e^{m_t - M}
    (M the final max), so z = sum_j e^{m_t - M} B(e^{s_j - m_t}) v_j and
    l = sum_j e^{s_j - M}.  Scores are exact rationals, exponentials are
    taken at 60 significant digits, each weight is rounded to BF16 by the
    rational rounder of this file.  Returns o = z/l (mpf), whether every
    weight is at least 2^-40 (relative) away from a BF16 rounding boundary,
    and the outputs with the weights rounded against the final max instead."""
    def mpf(fr):
        return mp.mpf(fr.numerator) / fr.denominator

    def frac(x):
        sign, man, ex, _ = mp.mpf(x)._mpf_      # value = (-1)^sign * man * 2^ex
        return (-1) ** sign * Fraction(man) * Fraction(2) ** ex

    n, nk = Q.shape[0], K.shape[0]
    s = [[Fraction(sc) * sum(Fraction(float(Q[i, c])) * Fraction(float(K[j, c]))
                             for c in range(Q.shape[1])) for j in range(nk)] for i in range(n)]
    blocks = [range(t0, min(t0 + kb, nk)) for t0 in range(0, nk, kb)]
    o, o_final, clear = [], [], True
    eps = Fraction(1, 2 ** 40)
    for i in range(n):
        run, ms = None, []
        for blk in blocks:
            bm = max(s[i][j] for j in blk)
            run = bm if run is None else max(run, bm)
            ms.append(run)
        M = ms[-1]
        z = [mp.mpf(0)] * V.shape[1]
        zf = [mp.mpf(0)] * V.shape[1]
        den = mp.mpf(0)
        for t, blk in enumerate(blocks):
            resc = mp.exp(mpf(ms[t] - M))
            for j in blk:
                p = frac(mp.exp(mpf(s[i][j] - ms[t])))
                w = _round_rational(p)
                clear = clear and _round_rational(p * (1 - eps)) == _round_rational(p * (1 + eps))
                pf = mp.exp(mpf(s[i][j] - M))
                wf = _round_rational(frac(pf))
                den += pf
                for c in range(V.shape[1]):
                    z[c] += resc * w * float(V[j, c])
                    zf[c] += wf * float(V[j, c])
        o.append([zc / den for zc in z])
        o_final.append([zc / den for zc in zf])
    return o, clear, o_final, frac


def test_attention_bf16_weights_several_blocks_running_max_moves():
    """Four key blocks (the last one partial) whose scores grow from block to
    block in every row, so the running max moves at each block and every
    earlier block's weights are rescaled: the oracle's recurrence against
    the unrolled closed form evaluated independently in high precision.  The
    same inputs with the weights rounded against the final max give other
    BF16 outputs, so a recurrence that rounded against the wrong max, or
    skipped or inverted a rescale, fails here."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 60
    rng = np.random.default_rng(31)
    dh, kb, nk = 8, 5, 17
    u = np.full(dh, 0.5)
    Q = bf16.round_bf16(u + 0.25 * rng.standard_normal((4, dh)))
    K = bf16.round_bf16(0.5 * rng.standard_normal((nk, dh))
                        + np.repeat(np.arange(4), kb)[:nk, None] * 1.5 * u)
    V = _rand_bf16(rng, (nk, dh))
    sc = 0.5
    S = sc * Q @ K.T
    bmax = np.stack([S[:, t0:t0 + kb].max(axis=1) for t0 in range(0, nk, kb)], axis=1)
    assert np.all(np.diff(bmax, axis=1) > 0)       # the max moves at every block
    r = ops.attention_bf16_weights(Q, K, V, sc, key_block=kb)
    o, clear, o_final, frac = _bf16_weights_closed_form(Q, K, V, sc, kb, mp)
    assert clear                       # no weight within 2^-40 of a rounding boundary
    want64 = np.array([[float(x) for x in row] for row in o])
    assert np.allclose(r.y64, want64, rtol=1e-13, atol=0)
    want = np.array([[_round_rational(frac(x)) for x in row] for row in o])
    assert np.array_equal(r.y, want)
    assert np.all(r.slack == 0)        # no ambiguous weight, so no slack
    wrong = np.array([[_round_rational(frac(x)) for x in row] for row in o_final])
    assert not np.array_equal(wrong, want)


# ------------------------------------------------- RMSNorm and split RoPE --
def _round_rational(v: Fraction) -> float:
    """RNE to 8 significant bits of any rational (normal range), by exact
    integer arithmetic: v = n * 2^q with q the quantum's exponent."""
    if v == 0:
        return 0.0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1                        # now 2^e <= a < 2^(e+1)
    q = Fraction(2) ** (e - 7)
    n = a / q
    k = n.numerator // n.denominator
    rem = n - k
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and k % 2 == 1):
        k += 1
    return math.copysign(float(k * q), float(v))


def test_rmsnorm_hand_worked():
    g = json.load(open(os.path.join(GOLD, "rmsnorm_hand.json")))
    for c in g["cases"]:
        r = ops.rmsnorm(np.array([c["x"]]), np.array(c["gamma"]), c["eps"])
        want = [_round_rational(Fraction(n, c["y_den"])) for n in c["y_num"]]
        assert r.y[0].tolist() == want, c["note"]


def test_rmsnorm_against_torch_rms_norm():
    """torch's own RMSNorm in float64 (an independent library routine)."""
    rng = np.random.default_rng(31)
    X = _rand_bf16(rng, (17, 96), 3.0)
    gmm = _rand_bf16(rng, (96,))
    for eps in (0.0, 1e-6, 0.5):
        r = ops.rmsnorm(X, gmm, eps)
        t = F.rms_norm(torch.from_numpy(X), (96,), torch.from_numpy(gmm), eps).numpy()
        assert np.allclose(r.y64, t, rtol=1e-13, atol=0)


def test_rmsnorm_scale_invariance_and_unit_mean_square():
    """With eps = 0 the map is invariant under x -> 2^k x (exact in float64)
    and, with gamma = 1, the output's mean square is 1."""
    rng = np.random.default_rng(32)
    X = _rand_bf16(rng, (9, 64))
    ones = np.ones(64)
    r = ops.rmsnorm(X, ones, 0.0)
    for k in (-20, 3):
        assert np.array_equal(ops.rmsnorm(X * 2.0 ** k, ones, 0.0).y, r.y)
    assert np.allclose((r.y64 ** 2).mean(axis=1), 1.0, rtol=1e-14)


@pytest.mark.parametrize("tile", [1, 7, 64, 100, 256])
def test_rmsnorm_width_partition(tile):
    """Section II-B: partial sums of squares over any width partition give
    the one global denominator (equal within the float64 bound)."""
    rng = np.random.default_rng(33)
    X = _rand_bf16(rng, (11, 256))
    gmm = _rand_bf16(rng, (256,))
    full = ops.rmsnorm(X, gmm, 1e-6)
    part = ops.rmsnorm_partitioned(X, gmm, 1e-6, tile)
    assert np.allclose(part.y64, full.y64, rtol=1e-14, atol=0)


def test_rmsnorm_zero_row():
    r = ops.rmsnorm(np.zeros((2, 8)), np.ones(8), 1e-6)
    assert np.array_equal(r.y, np.zeros((2, 8)))


def _rope_table(n, half, seed):
    rng = np.random.default_rng(seed)
    th = rng.uniform(-np.pi, np.pi, (n, half))
    return np.cos(th).astype(np.float32).astype(np.float64), \
        np.sin(th).astype(np.float32).astype(np.float64)


def test_rope_split_against_complex_multiplication():
    """The pair (t_j, t_{j+dh/2}) as the complex number t_j + i t_{j+dh/2},
    multiplied by c + i s: an independent formulation of the rotation."""
    rng = np.random.default_rng(34)
    dh, H = 8, 3
    T = rng.standard_normal((5, dh * H + 8))
    c, s = _rope_table(5, dh // 2, 1)
    out = ops.rope_split(T, c, s, dh, dh * H)
    for h in range(H):
        z = torch.complex(torch.from_numpy(T[:, h * dh:h * dh + dh // 2]),
                          torch.from_numpy(T[:, h * dh + dh // 2:(h + 1) * dh]))
        w = z * torch.complex(torch.from_numpy(c), torch.from_numpy(s))
        assert np.allclose(out[:, h * dh:h * dh + dh // 2], w.real.numpy(), rtol=0, atol=1e-15)
        assert np.allclose(out[:, h * dh + dh // 2:(h + 1) * dh], w.imag.numpy(), rtol=0, atol=1e-15)
    assert np.array_equal(out[:, dh * H:], T[:, dh * H:])


def test_linear_rope_quarter_turn_is_a_row_permutation():
    """c = 0, s = 1 maps (a, b) to (-b, a): the rotated projection is the
    plain projection of W and b with each head's halves swapped and the
    first negated, rounded once (bitwise, exact ties included)."""
    rng = np.random.default_rng(35)
    dh, H, K = 8, 2, 40
    M = dh * H + 8
    X = _rand_bf16(rng, (6, K))
    W = _rand_bf16(rng, (M, K), 0.2)
    b = _rand_bf16(rng, (M,), 0.1)
    c, s = np.zeros((6, dh // 2)), np.ones((6, dh // 2))
    r = ops.linear_rope(X, W, b, c, s, dh, dh * H)
    perm = np.arange(M)
    sign = np.ones(M)
    for h in range(H):
        lo = np.arange(h * dh, h * dh + dh // 2)
        perm[lo], perm[lo + dh // 2] = lo + dh // 2, lo
        sign[lo] = -1.0
    ref = ops.linear(X, W[perm] * sign[:, None], b[perm] * sign)
    assert np.array_equal(r.y, ref.y)
    ident = ops.linear_rope(X, W, b, np.ones_like(c), np.zeros_like(s), dh, dh * H)
    assert np.array_equal(ident.y, ops.linear(X, W, b).y)


def test_linear_rope_preserves_pair_norms():
    """|rotated pair| = |pair| when c^2 + s^2 = 1 (within the table's FP32
    rounding): a wrong pairing or sign breaks it."""
    rng = np.random.default_rng(36)
    dh, H, K = 16, 2, 24
    X = _rand_bf16(rng, (7, K))
    W = _rand_bf16(rng, (dh * H, K), 0.2)
    b = np.zeros(dh * H)
    th = rng.uniform(-np.pi, np.pi, (7, dh // 2))
    r = ops.linear_rope(X, W, b, np.cos(th), np.sin(th), dh, dh * H)
    t = X @ W.T
    h = dh // 2
    for h0 in range(0, dh * H, dh):
        n_in = t[:, h0:h0 + h] ** 2 + t[:, h0 + h:h0 + dh] ** 2
        n_out = r.y64[:, h0:h0 + h] ** 2 + r.y64[:, h0 + h:h0 + dh] ** 2
        assert np.allclose(n_out, n_in, rtol=1e-13)


def test_linear_rope_bf16_first_variant():
    """The baseline materialisation rounds the projection before rotating:
    equal to rotating the oracle's own rounded linear output; for c = 1,
    s = 0 both variants equal the plain projection."""
    rng = np.random.default_rng(37)
    dh, K = 8, 32
    X = _rand_bf16(rng, (5, K))
    W = _rand_bf16(rng, (2 * dh, K), 0.3)
    b = _rand_bf16(rng, (2 * dh,), 0.1)
    c, s = _rope_table(5, dh // 2, 2)
    r = ops.linear_rope(X, W, b, c, s, dh, dh, rope_after_bf16=True)
    lin = ops.linear(X, W, b)
    assert np.array_equal(r.y, bf16.round_bf16(ops.rope_split(lin.y, c, s, dh, dh)))
    one = ops.linear_rope(X, W, b, np.ones_like(c), np.zeros_like(s), dh, dh,
                          rope_after_bf16=True)
    assert np.array_equal(one.y, lin.y)
