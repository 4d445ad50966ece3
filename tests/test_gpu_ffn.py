"""Paged FFN on the GPU against the oracle (PSI section II-B Eq.(2), section
III-B reuse schedule: each hidden slice computed once, BF16-written, reused by
its down projection; ordered FP32 accumulation; output bias once)."""
import math

import numpy as np
import pytest
import torch

import psi_synth
from weight_streamed_bf16_gb300 import psi

from gpu_cases import check, ensure_lib, f64, grade, ops, run_ffn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _case(N, d, h, r, seed):
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(N, d, generator=g).to(torch.bfloat16)
    U = (torch.randn(h, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    V = (torch.randn(r, h, generator=g) / math.sqrt(h)).to(torch.bfloat16)
    a = (torch.randn(h, generator=g) * 0.02).to(torch.bfloat16)
    b = (torch.randn(r, generator=g) * 0.02).to(torch.bfloat16)
    return X, U, V, a, b


def test_ffn_config_paged():
    """X [1024 x 2048], W1 [8192 x 2048], W2 [2048 x 8192], 1024-wide slices,
    4-slice arena (the full configuration; the oracle runs in seconds)."""
    cfg = psi_synth.FFN
    X, U, V, a, b = psi_synth.ffn_inputs(cfg)
    y, hid_last, stats = run_ffn(X, U, V, a, b, cfg.slice, cfg.slots, return_hidden=True)
    res = ops.ffn(f64(X), f64(U), f64(V), f64(a), f64(b))
    rep = check(y, res, what="ffn config")
    assert rep["max_rel_err"] <= 1e-2
    # the last hidden slice in the workspace: BF16 values of B(phi(t)), graded
    # with the pre-activation's term magnitudes as the scale and the oracle's
    # ambiguity bound for the rounding at this boundary as slack
    S = cfg.h // cfg.slice
    J0 = (S - 1) * cfg.slice
    Xf, Uf = f64(X), f64(U)[J0:]
    t = Xf @ Uf.T + f64(a)[J0:]
    At = np.abs(Xf) @ np.abs(Uf).T + np.abs(f64(a)[J0:])
    Hl = res.H[:, J0:]
    jump = ops.hidden_rounding_jump(t, At, Hl)
    g = grade.graded_ulps(f64(hid_last), Hl, Hl, At, slack=jump)
    assert g.max() <= 2, g.max()
    assert np.count_nonzero(grade.raw_ulps(f64(hid_last), Hl)) < 1e-2 * Hl.size
    assert stats["pages_streamed"] == S and stats["h2d_bytes"] == S * cfg.page_bytes


@pytest.mark.parametrize("N,d,h,r,slice_,slots", [
    (100, 136, 192, 72, 64, 2),     # ragged tokens, widths not multiples of the tiles
    (5, 64, 64, 64, 64, 1),          # a single slice (bias and residual in one pass)
    (257, 256, 512, 320, 128, 3),    # several M tiles, N tail on the down projection
])
def test_ffn_ragged(N, d, h, r, slice_, slots):
    X, U, V, a, b = _case(N, d, h, r, N + d)
    R = torch.randn(N, r).to(torch.bfloat16)
    y = run_ffn(X, U, V, a, b, slice_, slots, residual=R)
    res = ops.ffn(f64(X), f64(U), f64(V), f64(a), f64(b), residual=f64(R))
    check(y, res, what=f"ffn {N}x{d}x{h}x{r}")


def test_ffn_pregelu_boundary():
    X, U, V, a, b = _case(128, 128, 256, 128, 3)
    y = run_ffn(X, U, V, a, b, 128, 2, flags=psi.PSI_BOUNDARY_PREGELU_BF16)
    res = ops.ffn(f64(X), f64(U), f64(V), f64(a), f64(b), pregelu_bf16=True)
    check(y, res, what="pregelu")


def test_ffn_resident_streamed_bitwise():
    X, U, V, a, b = _case(192, 256, 1024, 256, 11)
    s = run_ffn(X, U, V, a, b, 256, 2)
    r = run_ffn(X, U, V, a, b, 256, 2, flags=psi.PSI_RESIDENT)
    c = run_ffn(X, U, V, a, b, 256, 4, flags=psi.PSI_SYNC_COPY)
    five = run_ffn(X, U, V, a, b, 256, 5)
    for o in (r, c, five):
        assert torch.equal(s.view(torch.int16), o.view(torch.int16))
    # a slice group needs two slots: a one-slot arena is refused up front
    with pytest.raises(psi.PsiError) as e:
        run_ffn(X, U, V, a, b, 256, 1)
    assert e.value.status == psi.PSI_ERR_CAPACITY


def test_ffn_odd_slice_count():
    """Five slices: two groups of two and a last group of one."""
    X, U, V, a, b = _case(130, 128, 320, 96, 17)
    y = run_ffn(X, U, V, a, b, 64, 3)
    check(y, ops.ffn(f64(X), f64(U), f64(V), f64(a), f64(b)), what="odd slices")


def test_ffn_baseline_variant():
    """Baseline PSI numerics: pre-GELU BF16 write and products rounded to
    BF16 before their biases (section III-A)."""
    X, U, V, a, b = _case(130, 256, 1024, 256, 41)
    flags = psi.PSI_BOUNDARY_PREGELU_BF16 | psi.PSI_BIAS_AFTER_BF16
    y = run_ffn(X, U, V, a, b, 256, 3, flags=flags)
    res = ops.ffn(f64(X), f64(U), f64(V), f64(a), f64(b), pregelu_bf16=True,
                  bias_after_bf16=True)
    check(y, res, what="ffn baseline")
