"""Pins of the oracle's BF16 decoding and rounding (CPU only).

Rounding B is round-to-nearest, ties-to-even (PSI, section II-C Eq.(5)).
Pins: the worked values of Eq.(5) and Eq.(6), torch's float32 -> bfloat16
conversion (a library routine), the textbook integer rounding of a binary32
bit pattern, and the exact dyadic rounder against the float64 one.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import bf16

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _frac(s):
    return Fraction(s)


def test_eq5_extra_write_boundary_changes_result():
    g = json.load(open(os.path.join(GOLD, "eq5_double_rounding.json")))
    z, b = _frac(g["z"]), _frac(g["b"])
    twice = bf16.round_bf16(float(bf16.round_bf16(float(z))) + float(b))
    once = bf16.round_bf16(float(z + b))
    assert Fraction(float(twice)) == _frac(g["B(B(z)+b)"])
    assert Fraction(float(once)) == _frac(g["B(z+b)"])
    # the same through the exact rational rounder
    assert Fraction(bf16.round_fraction(Fraction(bf16.round_fraction(z)) + b)) == 1
    assert Fraction(bf16.round_fraction(z + b)) == Fraction(129, 128)


def test_eq6_single_rounding_of_exact_sum():
    g = json.load(open(os.path.join(GOLD, "eq6_exact_sum.json")))
    y_star = _frac(g["y_star"])
    native = _frac(g["y_native"])
    official = _frac(g["y_official"])
    assert Fraction(bf16.round_fraction(y_star)) == native
    assert Fraction(bf16.round_fraction(y_star)) != official
    assert Fraction(float(bf16.round_bf16(float(y_star)))) == native


def test_decode_all_patterns_against_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = bf16.decode(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    same = (mine == ref) | (np.isnan(mine) & np.isnan(ref))
    assert same.all()
    # signed zeros decode to signed zeros
    assert np.signbit(mine[0x8000]) and not np.signbit(mine[0])


def test_encode_roundtrip_all_finite():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bf16.decode(bits)
    fin = np.isfinite(vals)
    assert np.array_equal(bf16.encode(vals[fin]), bits[fin])


def _fp32_samples():
    rng = np.random.default_rng(1234)
    r = rng.integers(0, 2**32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    # every BF16 value with the low half set to the tie, just below and above
    hi = np.arange(65536, dtype=np.uint32) << 16
    ties = np.concatenate([hi | 0x8000, hi | 0x7FFF, hi | 0x8001, hi | 0x0001, hi | 0xFFFF])
    return np.concatenate([r, ties, hi])


def test_round_against_torch_fp32_conversion():
    u = _fp32_samples()
    f = u.view(np.float32)
    keep = np.isfinite(f)
    f = f[keep]
    mine = bf16.round_bf16(f.astype(np.float64))
    ref = torch.from_numpy(f).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(mine, ref)


def test_round_against_integer_bit_rounding():
    """Textbook RNE on the binary32 pattern: add 0x7FFF plus the kept lsb."""
    u = _fp32_samples()
    f = u.view(np.float32)
    keep = np.isfinite(f)
    u, f = u[keep].astype(np.uint64), f[keep]
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    ref = bf16.decode(r)
    mine = bf16.round_bf16(f.astype(np.float64))
    assert np.array_equal(mine, ref)


def test_round_direct_from_float64_no_double_rounding():
    # 1 + 2^-8 + 2^-40 lies just above a BF16 tie, so B rounds it up.  Through
    # float32 first, 2^-40 is lost, the value becomes the tie and rounds to 1.
    x = 1.0 + 2.0**-8 + 2.0**-40
    assert bf16.round_bf16(x) == 1.0 + 2.0**-7
    assert float(torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)) == 1.0


def test_overflow_subnormal_and_signs():
    big = (2.0 - 2.0**-8) * 2.0**127  # halfway between max finite and 2^128
    assert bf16.round_bf16(big) == np.inf
    assert bf16.round_bf16(-big) == -np.inf
    maxf = (2.0 - 2.0**-7) * 2.0**127
    assert bf16.round_bf16(np.nextafter(big, 0)) == maxf
    assert bf16.round_bf16(2.0**-133) == 2.0**-133
    assert bf16.round_bf16(2.0**-134) == 0.0          # tie to even (0)
    assert bf16.round_bf16(3 * 2.0**-135) == 2.0**-133
    assert np.signbit(bf16.round_bf16(-2.0**-140))
    assert np.isnan(bf16.round_bf16(np.nan))


def test_dyadic_rounder_matches_float_rounder():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(20000) * np.exp2(rng.integers(-140, 130, 20000))
    for v in x[:20000:7]:
        fr = Fraction(float(v))
        got = bf16.round_fraction(fr)
        want = float(bf16.round_bf16(float(v)))
        assert got == want or (np.isinf(got) and np.isinf(want))


def test_ulp_spacing():
    assert bf16.ulp(1.0) == 2.0**-7
    assert bf16.ulp(1.99) == 2.0**-7
    assert bf16.ulp(0.5) == 2.0**-8
    assert bf16.ulp(0.0) == 2.0**-133
    assert bf16.ulp(2.0**-130) == 2.0**-133


@pytest.mark.parametrize("n,e", [(0, 0), (255, 0), (257, -8), (-513, 3), (3, -135)])
def test_dyadic_small_cases(n, e):
    assert bf16.round_dyadic(n, e) == float(bf16.round_bf16(n * 2.0**e))
