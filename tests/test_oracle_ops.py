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
