"""Dense float64 definitions of the paged operators, one BF16 rounding per
declared write boundary.

All array arguments are float64 arrays whose entries are BF16 values (decode
them with ``oracle.bf16.decode``).  Products of two BF16 values are exact in
float64; sums are float64 and carry the usual error bound
|fl(sum) - sum| <= gamma_n * sum|terms|, gamma_n = n*u/(1-n*u), u = 2**-53.
Where that bound straddles a BF16 rounding decision, ``linear`` and ``ffn``
recompute the element exactly with rational arithmetic and round that exact
sum a single time (the exact evaluation of section IV-B, Eq.(6)).

Each result carries ``y`` (BF16 values as float64), ``y64`` (the unrounded
float64 value) and ``A`` (the sum of the magnitudes of the terms, or for
attention the softmax-weighted mean of |v|), which the grading uses.
"""
from __future__ import annotations

from dataclasses import dataclass
from fractions import Fraction

import numpy as np

from .bf16 import round_bf16, round_fraction

U64 = 2.0 ** -53
GELU_K0 = np.sqrt(2.0 / np.pi)
GELU_K1 = 0.044715


@dataclass
class Result:
    y: np.ndarray     # B(value), float64
    y64: np.ndarray   # float64 value before the final rounding
    A: np.ndarray     # magnitude scale of the element (see module docstring)
    H: np.ndarray | None = None   # FFN hidden activations (BF16 values)
    exact_fixed: int = 0          # elements re-rounded from an exact sum
    slack: np.ndarray | None = None  # extra |dy| allowed by ambiguous BF16
                                     # roundings at an inner write boundary


def _gamma(n: int) -> float:
    return n * U64 / (1.0 - n * U64)


def _fix_ties(y, y64, A, nterms, exact_elem):
    """Re-round, from the exact sum, every element whose float64 value is
    within its error bound of a BF16 rounding boundary."""
    d = 2.0 * _gamma(nterms) * A
    amb = round_bf16(y64 - d) != round_bf16(y64 + d)
    idx = np.argwhere(amb)
    for ij in idx:
        t = tuple(ij)
        y[t] = round_fraction(exact_elem(t))
    return len(idx)


def gelu_tanh(x):
    """phi(x) = x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3))), float64.

    Section II-B names a tanh-based GELU without constants; this is the
    textbook tanh approximation of the Gaussian error linear unit.
    """
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(GELU_K0 * (x + GELU_K1 * x * x * x)))


def linear(X, W, b, residual=None, exact_ties=True, bias_after_bf16=False) -> Result:
    """y = B(X W^T + b [+ residual]).

    X [N x K], W [M x K] (out x in, as U in Eq.(2)), b [M], residual [N x M].
    The bias (and residual) join the float64 sum before the only BF16 write:
    the modified order of section III-A.  With ``bias_after_bf16`` (the
    paper's baseline variant) the product is rounded first:
    y = B(B(X W^T) + b [+ residual]).
    """
    X = np.asarray(X, np.float64)
    W = np.asarray(W, np.float64)
    b = np.asarray(b, np.float64)
    if bias_after_bf16:
        return _linear_bias_after(X, W, b, residual, exact_ties)
    y64 = X @ W.T + b[None, :]
    A = np.abs(X) @ np.abs(W).T + np.abs(b)[None, :]
    if residual is not None:
        residual = np.asarray(residual, np.float64)
        y64 = y64 + residual
        A = A + np.abs(residual)
    y = round_bf16(y64)
    fixed = 0
    if exact_ties:
        def exact(t):
            i, j = t
            s = sum(Fraction(float(X[i, k])) * Fraction(float(W[j, k]))
                    for k in range(X.shape[1]))
            s += Fraction(float(b[j]))
            if residual is not None:
                s += Fraction(float(residual[i, j]))
            return s
        fixed = _fix_ties(y, y64, A, X.shape[1] + 2, exact)
    return Result(y=y, y64=y64, A=A, exact_fixed=fixed)


def _round_exact(p64, A, X, W, exact_ties):
    """B(X W^T), re-rounding near-ties from the exact sum."""
    p = round_bf16(p64)
    if exact_ties:
        def exact(ij):
            i, j = ij
            return sum(Fraction(float(X[i, k])) * Fraction(float(W[j, k]))
                       for k in range(X.shape[1]))
        _fix_ties(p, p64, A, X.shape[1] + 1, exact)
    return p


def _linear_bias_after(X, W, b, residual, exact_ties):
    p64 = X @ W.T
    Ap = np.abs(X) @ np.abs(W).T
    p = _round_exact(p64, Ap, X, W, exact_ties)
    y64 = p + b[None, :]
    A = np.abs(p) + np.abs(b)[None, :]
    if residual is not None:
        residual = np.asarray(residual, np.float64)
        y64 = y64 + residual
        A = A + np.abs(residual)
    y = round_bf16(y64)
    # an FP32 product near a BF16 rounding boundary may round the other way
    d = T_REL * Ap
    jump = np.maximum(np.abs(round_bf16(p64 - d) - p), np.abs(round_bf16(p64 + d) - p))
    slack = np.maximum(np.abs(round_bf16(y64 + jump) - y), np.abs(round_bf16(y64 - jump) - y))
    return Result(y=y, y64=y64, A=A, slack=slack)


def ffn(X, U, V, a, b, residual=None, pregelu_bf16=False,
        exact_ties=True, bias_after_bf16=False) -> Result:
    """Dense FFN with the declared boundaries of Eq.(2):

        t   = X U^T + a                         (float64, exact ties)
        t   = B(t)            only if pregelu_bf16 (the paper's extra write)
        H   = B(phi(t))
        y   = B(H V^T + b [+ residual])

    X [N x d], U [h x d], V [r x h], a [h], b [r], residual [N x r].
    With ``bias_after_bf16`` (the baseline variant of section III-A) both
    products are rounded before their bias: t = B(X U^T) + a and
    y = B(B(H V^T) + b [+ residual]).
    """
    X = np.asarray(X, np.float64)
    U = np.asarray(U, np.float64)
    V = np.asarray(V, np.float64)
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if bias_after_bf16:
        p64 = X @ U.T
        Ap = np.abs(X) @ np.abs(U).T
        pr = _round_exact(p64, Ap, X, U, exact_ties)
        t = pr + a[None, :]
        At = Ap + np.abs(a)[None, :]
    else:
        p64 = None
        t = X @ U.T + a[None, :]
        At = np.abs(X) @ np.abs(U).T + np.abs(a)[None, :]
    t_exact = t
    if pregelu_bf16:
        tb = round_bf16(t)
        if exact_ties:
            def exact_t(ij):
                i, j = ij
                if bias_after_bf16:  # t = B(product) + a
                    return Fraction(float(pr[i, j])) + Fraction(float(a[j]))
                s = sum(Fraction(float(X[i, k])) * Fraction(float(U[j, k]))
                        for k in range(X.shape[1]))
                return s + Fraction(float(a[j]))
            _fix_ties(tb, t, At if not bias_after_bf16 else np.abs(t), 4 if bias_after_bf16
                      else X.shape[1] + 2, exact_t)
        t = tb
    H = round_bf16(gelu_tanh(t))
    if bias_after_bf16:
        # the pre-activation moves with the product's rounding
        d = T_REL * Ap
        lo_t = round_bf16(p64 - d) + a[None, :]
        hi_t = round_bf16(p64 + d) + a[None, :]
        jump = np.maximum(hidden_rounding_jump(lo_t, At, H, pregelu_bf16),
                          hidden_rounding_jump(hi_t, At, H, pregelu_bf16))
    else:
        jump = hidden_rounding_jump(t_exact, At, H, pregelu_bf16)
    slack = jump @ np.abs(V).T
    if bias_after_bf16:
        q64 = H @ V.T
        Aq = np.abs(H) @ np.abs(V).T
        q = _round_exact(q64, Aq, H, V, exact_ties)
        y64 = q + b[None, :]
        A = np.abs(q) + np.abs(b)[None, :]
        dq = T_REL * Aq + slack
        qj = np.maximum(np.abs(round_bf16(q64 - dq) - q), np.abs(round_bf16(q64 + dq) - q))
        if residual is not None:
            residual = np.asarray(residual, np.float64)
            y64 = y64 + residual
            A = A + np.abs(residual)
        y = round_bf16(y64)
        slack = np.maximum(np.abs(round_bf16(y64 + qj) - y), np.abs(round_bf16(y64 - qj) - y))
        return Result(y=y, y64=y64, A=A, H=H, slack=slack)
    y64 = H @ V.T + b[None, :]
    A = np.abs(H) @ np.abs(V).T + np.abs(b)[None, :]
    if residual is not None:
        residual = np.asarray(residual, np.float64)
        y64 = y64 + residual
        A = A + np.abs(residual)
    y = round_bf16(y64)
    fixed = 0
    if exact_ties:
        def exact(ij):
            i, j = ij
            s = sum(Fraction(float(H[i, k])) * Fraction(float(V[j, k]))
                    for k in range(H.shape[1]))
            s += Fraction(float(b[j]))
            if residual is not None:
                s += Fraction(float(residual[i, j]))
            return s
        fixed = _fix_ties(y, y64, A, H.shape[1] + 2, exact)
    return Result(y=y, y64=y64, A=A, H=H, exact_fixed=fixed, slack=slack)


# FP32 evaluation bound used to decide whether a BF16 rounding at the hidden
# write boundary is ambiguous: pre-activation error <= 2**-22 * sum|terms|
# (a few units of FP32 roundoff relative to the term magnitudes, far above
# the ~2**-24 / sqrt(K) typical relative error of a K-term FP32 dot
# product), GELU evaluated in FP32 to within 2**-21 * (|t| + |phi(t)|).
T_REL = 2.0 ** -22
PHI_REL = 2.0 ** -21


def hidden_rounding_jump(t, At, H, pregelu_bf16=False):
    """For each hidden element, how far B(phi(t')) can move from H when t'
    and phi are evaluated in FP32 instead of exactly (0 where the rounding is
    unambiguous).  Two correct evaluations of Eq.(2) with a BF16 write of H
    may differ there by this much; the output tolerance adds the effect of
    those differences on the down projection."""
    d = T_REL * At
    lo, hi = t - d, t + d
    if pregelu_bf16:
        lo, hi = round_bf16(lo), round_bf16(hi)
    cands = []
    for x in (lo, hi):
        p = gelu_tanh(x)
        e = PHI_REL * (np.abs(x) + np.abs(p))
        cands.append(round_bf16(p - e))
        cands.append(round_bf16(p + e))
    jump = np.zeros_like(H)
    for c in cands:
        jump = np.maximum(jump, np.abs(c - H))
    return jump


def ffn_partitioned_exact(X, U, V, a, b, slices):
    """Eq.(2) taken literally on a small case, in exact rationals.

    ``slices`` is a list of disjoint hidden-index lists covering 0..h-1.
    For each slice J: H_J = B(phi(X U_J^T + a_J)) (phi in float64 on the
    exact pre-activation, which is exact in float64 for small K), then the
    down-projection partials H_J V_:,J^T are summed exactly over J and the
    output bias is added once before a single rounding.  Python loops only:
    for tiny shapes.
    """
    X = np.asarray(X, np.float64)
    U = np.asarray(U, np.float64)
    V = np.asarray(V, np.float64)
    N, r = X.shape[0], V.shape[0]
    acc = [[Fraction(0)] * r for _ in range(N)]
    Hfull = np.zeros((N, U.shape[0]))
    for J in slices:
        for i in range(N):
            for j in J:
                t = sum(Fraction(float(X[i, k])) * Fraction(float(U[j, k]))
                        for k in range(X.shape[1])) + Fraction(float(a[j]))
                h = float(round_bf16(gelu_tanh(float(t))))
                Hfull[i, j] = h
                for o in range(r):
                    acc[i][o] += Fraction(h) * Fraction(float(V[o, j]))
    y = np.array([[round_fraction(acc[i][o] + Fraction(float(b[o])))
                   for o in range(r)] for i in range(N)])
    return y, Hfull


def attention(Q, K, V, scale, rows=None) -> Result:
    """Dense softmax attention for one head, Eq.(3) over the whole key set.

    Q [Nq x dh], K [Nk x dh], V [Nk x dh]; s_j = scale * q.k_j;
    o = sum_j e^{s_j - m} v_j / sum_j e^{s_j - m}, m = max_j s_j; O = B(o).
    ``rows`` selects a subset of query rows.  Unmasked, noncausal, no
    dropout, at least one key (the conditions stated under Eq.(4)).
    """
    Q = np.asarray(Q, np.float64)
    if rows is not None:
        Q = Q[np.asarray(rows)]
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    if K.shape[0] == 0:
        raise ValueError("attention needs at least one key")
    S = scale * (Q @ K.T)
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    l = P.sum(axis=1, keepdims=True)
    o64 = (P @ V) / l
    A = (P @ np.abs(V)) / l
    return Result(y=round_bf16(o64), y64=o64, A=A)


def attention_heads(Q, K, V, scale, rows=None, heads=None) -> Result:
    """``attention`` over a [heads x N x dh] layout; returns stacked results."""
    hs = range(Q.shape[0]) if heads is None else heads
    rs = [attention(Q[h], K[h], V[h], scale, rows) for h in hs]
    return Result(y=np.stack([r.y for r in rs]), y64=np.stack([r.y64 for r in rs]),
                  A=np.stack([r.A for r in rs]))


# relative error bound of an FP32-evaluated exponential weight (FP32 score,
# scaled exponent, hardware ex2): used to decide ambiguous BF16 roundings
P_REL = 2.0 ** -19


def attention_bf16_weights(Q, K, V, scale, key_block, rows=None) -> Result:
    """The baseline variant of section III-A: the online recurrence of
    Eqs.(3)-(4) over key blocks of ``key_block`` with the numerator's
    exponential weights rounded to BF16, z' = eta*z + sum B(e^{s_j-m'}) v_j,
    and the denominator l' = eta*l + sum e^{s_j-m'} in float64; O = B(z/l).
    The rounded weights depend on the running max, so the partition is the
    kernel's.  ``slack`` covers weights within P_REL of a rounding boundary."""
    Q = np.asarray(Q, np.float64)
    if rows is not None:
        Q = Q[np.asarray(rows)]
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    n = Q.shape[0]
    m = np.full((n, 1), -np.inf)
    l = np.zeros((n, 1))
    z = np.zeros((n, V.shape[1]))
    zs = np.zeros((n, V.shape[1]))
    za = np.zeros((n, V.shape[1]))
    for t0 in range(0, K.shape[0], key_block):
        s = scale * (Q @ K[t0:t0 + key_block].T)
        m_new = np.maximum(m, s.max(axis=1, keepdims=True))
        eta = np.exp(m - m_new)
        p = np.exp(s - m_new)
        pb = round_bf16(p)
        jump = np.maximum(np.abs(round_bf16(p * (1 - P_REL)) - pb),
                          np.abs(round_bf16(p * (1 + P_REL)) - pb))
        Vt = V[t0:t0 + key_block]
        l = eta * l + p.sum(axis=1, keepdims=True)
        z = eta * z + pb @ Vt
        zs = eta * zs + jump @ np.abs(Vt)
        za = eta * za + p @ np.abs(Vt)
        m = m_new
    o64 = z / l
    return Result(y=round_bf16(o64), y64=o64, A=za / l, slack=zs / l)


def attention_online(Q, K, V, scale, key_block):
    """The online-softmax recurrence of Eqs.(3)-(4), float64.

    Keys are visited in disjoint tiles T of ``key_block`` keys.  For each
    tile: m' = max(m, max_T s_j), eta = e^{m - m'}, l' = eta*l + sum_T
    e^{s_j - m'}, z' = eta*z + sum_T e^{s_j - m'} v_j.  Returns B(z/l) and
    z/l.
    """
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    n = Q.shape[0]
    m = np.full((n, 1), -np.inf)
    l = np.zeros((n, 1))
    z = np.zeros((n, V.shape[1]))
    for t0 in range(0, K.shape[0], key_block):
        s = scale * (Q @ K[t0:t0 + key_block].T)
        m_new = np.maximum(m, s.max(axis=1, keepdims=True))
        eta = np.exp(m - m_new)
        p = np.exp(s - m_new)
        l = eta * l + p.sum(axis=1, keepdims=True)
        z = eta * z + p @ V[t0:t0 + key_block]
        m = m_new
    o64 = z / l
    return round_bf16(o64), o64


def rmsnorm(X, gamma, eps) -> Result:
    """Full-row RMS normalisation of section II-B, one BF16 write:

        y_i = B(gamma_i * x_i / sqrt(s/d + eps)),   s = sum_i x_i^2

    over the whole row width d.  X [N x d], gamma [d] (BF16 values), eps a
    float.  ``A`` is |y| (one product per element)."""
    X = np.asarray(X, np.float64)
    g = np.asarray(gamma, np.float64)
    d = X.shape[1]
    s = (X * X).sum(axis=1, keepdims=True)
    den = np.sqrt(s / d + eps)
    y64 = g[None, :] * X / den
    return Result(y=round_bf16(y64), y64=y64, A=np.abs(y64))


def rmsnorm_partitioned(X, gamma, eps, tile) -> Result:
    """The partitioned form of section II-B: the row is cut into width tiles
    J of ``tile`` columns, each tile contributes its partial sum of squares,
    s = sum_J sum_{i in J} x_i^2 is formed once, and the same positive
    denominator normalises every tile."""
    X = np.asarray(X, np.float64)
    g = np.asarray(gamma, np.float64)
    N, d = X.shape
    parts = [(X[:, j0:j0 + tile] ** 2).sum(axis=1) for j0 in range(0, d, tile)]
    s = np.sum(parts, axis=0)[:, None]
    den = np.sqrt(s / d + eps)
    y64 = np.concatenate([g[None, j0:j0 + tile] * X[:, j0:j0 + tile] / den
                          for j0 in range(0, d, tile)], axis=1)
    return Result(y=round_bf16(y64), y64=y64, A=np.abs(y64))


def rope_split(T, cos, sin, dh, cols):
    """Split RoPE of section II-B on float64 values T [N x M]: in each head
    of ``dh`` columns among the first ``cols``, the pair (a, b) = (t_j,
    t_{j+dh/2}) becomes (c a - s b, s a + c b) with c = cos[n, j], s =
    sin[n, j] (table row n = token, index j < dh/2).  Columns from ``cols``
    on pass through.  Returns the rotated values."""
    T = np.asarray(T, np.float64)
    c = np.asarray(cos, np.float64)
    s = np.asarray(sin, np.float64)
    h = dh // 2
    out = T.copy()
    for h0 in range(0, cols, dh):
        a = T[:, h0:h0 + h]
        b = T[:, h0 + h:h0 + dh]
        out[:, h0:h0 + h] = c * a - s * b
        out[:, h0 + h:h0 + dh] = s * a + c * b
    return out


def linear_rope(X, W, b, cos, sin, dh, cols, rope_after_bf16=False,
                exact_ties=True) -> Result:
    """A projection whose leading ``cols`` output columns (the query and key
    heads) are rotated by split RoPE before the single BF16 write:

        y = B(rope(X W^T + b))

    The rotation mixes the pair's exact values, so the only rounding is the
    write.  With ``rope_after_bf16`` the projection is written first and the
    rotation applied to the BF16 values: y = B(rope(B(X W^T + b))), the
    extra materialisation of the baseline variant."""
    X = np.asarray(X, np.float64)
    W = np.asarray(W, np.float64)
    b = np.asarray(b, np.float64)
    c = np.abs(np.asarray(cos, np.float64))
    s = np.abs(np.asarray(sin, np.float64))
    h = dh // 2
    if rope_after_bf16:
        base = linear(X, W, b, exact_ties=exact_ties)
        u, Au = base.y, np.abs(base.y)
    else:
        u = X @ W.T + b[None, :]
        Au = np.abs(X) @ np.abs(W).T + np.abs(b)[None, :]
    y64 = rope_split(u, cos, sin, dh, cols)
    A = Au.copy()
    for h0 in range(0, cols, dh):
        Aa, Ab = Au[:, h0:h0 + h], Au[:, h0 + h:h0 + dh]
        A[:, h0:h0 + h] = c * Aa + s * Ab
        A[:, h0 + h:h0 + dh] = s * Aa + c * Ab
    y = round_bf16(y64)
    fixed = 0
    slack = None
    if exact_ties:
        cf = np.asarray(cos, np.float64)
        sf = np.asarray(sin, np.float64)

        def t_exact(i, j):
            if rope_after_bf16:
                return Fraction(float(u[i, j]))
            return sum(Fraction(float(X[i, k])) * Fraction(float(W[j, k]))
                       for k in range(X.shape[1])) + Fraction(float(b[j]))

        def exact(ij):
            i, j = ij
            if j >= cols:
                return t_exact(i, j)
            h0, r = j - j % dh, j % dh
            jj = r % h
            ta, tb = t_exact(i, h0 + jj), t_exact(i, h0 + h + jj)
            cc, ss = Fraction(float(cf[i, jj])), Fraction(float(sf[i, jj]))
            return cc * ta - ss * tb if r < h else ss * ta + cc * tb
        fixed = _fix_ties(y, y64, A, (2 if rope_after_bf16 else X.shape[1] + 2) + 2, exact)
    if rope_after_bf16:
        # an FP32 pre-rotation value near a BF16 boundary may round the other way
        t64 = X @ W.T + b[None, :]
        At = np.abs(X) @ np.abs(W).T + np.abs(b)[None, :]
        d = T_REL * At
        jump = np.maximum(np.abs(round_bf16(t64 - d) - u), np.abs(round_bf16(t64 + d) - u))
        J = jump.copy()
        for h0 in range(0, cols, dh):
            Ja, Jb = jump[:, h0:h0 + h], jump[:, h0 + h:h0 + dh]
            J[:, h0:h0 + h] = c * Ja + s * Jb
            J[:, h0 + h:h0 + dh] = s * Ja + c * Jb
        slack = np.maximum(np.abs(round_bf16(y64 + J) - y), np.abs(round_bf16(y64 - J) - y))
    return Result(y=y, y64=y64, A=A, exact_fixed=fixed, slack=slack)
