"""Paged linear on the GPU against the oracle (PSI section IV-B projection
pages; section III-A bias before the single BF16 write)."""
import math

import pytest
import torch

import psi_synth
from weight_streamed_bf16_gb300 import psi

from gpu_cases import check, ensure_lib, f64, ops, run_linear

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def test_linear_config_single_paged():
    """X [64 x 512], W [512 x 512] in 64-row pages, 2-page arena, seed 0."""
    cfg = psi_synth.LINEAR
    X, W, b = psi_synth.linear_inputs(cfg)
    y = run_linear(X, W, b, cfg.page_rows, cfg.slots)
    res = ops.linear(f64(X), f64(W), f64(b))
    rep = check(y, res, what="linear config")
    assert rep["max_raw_ulps"] <= 2


@pytest.mark.parametrize("N,K,M,page_rows,slots", [
    (1, 64, 32, 16, 1),          # one token, one slot (copy waits for every consumer)
    (77, 200, 130, 48, 2),       # ragged tokens, K tail (200 = 3*64 + 8), ragged last page
    (300, 520, 272, 256, 3),     # multiple M tiles, N tile tail of a 256-row page
    (129, 1024, 700, 352, 2),    # page rows not a multiple of the 256 tile
])
def test_linear_ragged_shapes(N, K, M, page_rows, slots):
    g = torch.Generator().manual_seed(N * 1000 + K)
    X = torch.randn(N, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(M, K, generator=g) / math.sqrt(K)).to(torch.bfloat16)
    b = (torch.randn(M, generator=g) * 0.02).to(torch.bfloat16)
    R = torch.randn(N, M, generator=g).to(torch.bfloat16)
    y = run_linear(X, W, b, page_rows, slots, residual=R)
    res = ops.linear(f64(X), f64(W), f64(b), residual=f64(R))
    check(y, res, what=f"linear {N}x{K}x{M}")


def test_linear_strided_output():
    """Y written into a wider buffer (ldy > rows), as the fused QKV layout does."""
    g = torch.Generator().manual_seed(5)
    X = torch.randn(130, 256, generator=g).to(torch.bfloat16)
    W = (torch.randn(96, 256, generator=g) / 16).to(torch.bfloat16)
    b = (torch.randn(96, generator=g) * 0.02).to(torch.bfloat16)
    y = run_linear(X, W, b, 32, 2, ldy=136)
    check(y, ops.linear(f64(X), f64(W), f64(b)), what="strided")


def test_linear_resident_streamed_sync_bitwise():
    """Transport-only control: resident, streamed (async ring) and streamed on
    the compute stream give the same bytes (byte-preserving transport)."""
    g = torch.Generator().manual_seed(7)
    X = torch.randn(256, 512, generator=g).to(torch.bfloat16)
    W = (torch.randn(1024, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16)
    b = (torch.randn(1024, generator=g) * 0.02).to(torch.bfloat16)
    a = run_linear(X, W, b, 128, 2)
    r = run_linear(X, W, b, 128, 2, flags=psi.PSI_RESIDENT)
    s = run_linear(X, W, b, 128, 2, flags=psi.PSI_SYNC_COPY)
    one = run_linear(X, W, b, 128, 1)
    many = run_linear(X, W, b, 128, 8)
    for o in (r, s, one, many):
        assert torch.equal(a.view(torch.int16), o.view(torch.int16))


@pytest.mark.parametrize("N,M,page_rows,flags", [
    (512, 1536, 512, 0),                          # three whole pages
    (300, 1280, 512, 0),                          # ragged last page of 256 rows
    (600, 1024, 256, psi.PSI_BIAS_AFTER_BF16),    # four pages, baseline rounding order
])
def test_linear_resident_one_launch_bitwise(N, M, page_rows, flags):
    """Resident pages on CTA pairs with 256-aligned page boundaries run as one
    launch over all pages: the same tiles and per-element arithmetic as the
    per-page launches of the streamed path, so the bytes are equal."""
    g = torch.Generator().manual_seed(N + M)
    K = 512
    X = torch.randn(N, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(M, K, generator=g) / math.sqrt(K)).to(torch.bfloat16)
    b = (torch.randn(M, generator=g) * 0.02).to(torch.bfloat16)
    R = torch.randn(N, M, generator=g).to(torch.bfloat16)
    n0 = psi.psi_kernel_launches()
    s = run_linear(X, W, b, page_rows, 2, flags=flags, residual=R)
    n1 = psi.psi_kernel_launches()
    r = run_linear(X, W, b, page_rows, 2, flags=flags | psi.PSI_RESIDENT, residual=R)
    n2 = psi.psi_kernel_launches()
    assert n1 - n0 == -(-M // page_rows) and n2 - n1 == 1
    assert torch.equal(s.view(torch.int16), r.view(torch.int16))
    check(r, ops.linear(f64(X), f64(W), f64(b), residual=f64(R),
                        bias_after_bf16=bool(flags & psi.PSI_BIAS_AFTER_BF16)),
          what=f"resident one launch {N}x{K}x{M}")


@pytest.mark.parametrize("N,M,page_rows,flags,launches", [
    (512, 2560, 512, 0, 3),                          # five pages: first alone, two pairs
    (300, 1280, 512, 0, 2),                          # first alone, a pair with a ragged page
    (600, 1792, 512, psi.PSI_BIAS_AFTER_BF16, 3),    # first, a pair, the ragged last alone
    (256, 1152, 512, 0, 3),                          # last page of 128 rows: no pair
    (257, 1536, 256, 0, 4),                          # six 256-row pages, ragged tokens
])
def test_linear_streamed_page_pairs_bitwise(N, M, page_rows, flags, launches):
    """With four or more ring slots, streamed pages on CTA pairs after the
    first go two to a launch (one tensor map per page), with copies on the
    copy stream or on the compute stream; the bytes equal the
    one-page-per-launch result of a two-slot ring and the resident single
    launch."""
    g = torch.Generator().manual_seed(3 * N + M)
    K = 512
    X = torch.randn(N, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(M, K, generator=g) / math.sqrt(K)).to(torch.bfloat16)
    b = (torch.randn(M, generator=g) * 0.02).to(torch.bfloat16)
    R = torch.randn(N, M, generator=g).to(torch.bfloat16)
    pages = -(-M // page_rows)
    n0 = psi.psi_kernel_launches()
    merged = run_linear(X, W, b, page_rows, 5, flags=flags, residual=R)
    n1 = psi.psi_kernel_launches()
    single = run_linear(X, W, b, page_rows, 2, flags=flags, residual=R)
    n2 = psi.psi_kernel_launches()
    res = run_linear(X, W, b, page_rows, 2, flags=flags | psi.PSI_RESIDENT, residual=R)
    n3 = psi.psi_kernel_launches()
    sync = run_linear(X, W, b, page_rows, 5, flags=flags | psi.PSI_SYNC_COPY, residual=R)
    n4 = psi.psi_kernel_launches()
    assert n1 - n0 == launches and n2 - n1 == pages and n4 - n3 == launches
    assert torch.equal(merged.view(torch.int16), single.view(torch.int16))
    assert torch.equal(merged.view(torch.int16), res.view(torch.int16))
    assert torch.equal(merged.view(torch.int16), sync.view(torch.int16))
    check(merged, ops.linear(f64(X), f64(W), f64(b), residual=f64(R),
                             bias_after_bf16=bool(flags & psi.PSI_BIAS_AFTER_BF16)),
          what=f"streamed page pairs {N}x{K}x{M}")


def test_linear_special_values():
    """W = I gives B(x + b); an all-zero input gives B(b)."""
    X = torch.randn(64, 128).to(torch.bfloat16)
    W = torch.eye(128).to(torch.bfloat16)
    b = (torch.randn(128) * 0.5).to(torch.bfloat16)
    y = run_linear(X, W, b, 64, 2)
    rep = check(y, ops.linear(f64(X), f64(W), f64(b)))
    assert rep["max_raw_ulps"] <= 1
    z = run_linear(torch.zeros(3, 128, dtype=torch.bfloat16), W, b, 64, 2)
    assert torch.equal(z.view(torch.int16), b.expand(3, 128).contiguous().view(torch.int16))


def test_linear_baseline_bias_after_bf16():
    """The paper's baseline rounding order (section III-A): product rounded to
    BF16 before the bias is added."""
    g = torch.Generator().manual_seed(31)
    X = torch.randn(300, 512, generator=g).to(torch.bfloat16)
    W = (torch.randn(512, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16)
    b = (torch.randn(512, generator=g) * 0.5).to(torch.bfloat16)
    R = torch.randn(300, 512, generator=g).to(torch.bfloat16)
    y = run_linear(X, W, b, 256, 2, flags=psi.PSI_BIAS_AFTER_BF16, residual=R)
    res = ops.linear(f64(X), f64(W), f64(b), residual=f64(R), bias_after_bf16=True)
    check(y, res, what="bias after bf16")
    y2 = run_linear(X, W, b, 256, 2, residual=R)
    assert not torch.equal(y.view(torch.int16), y2.view(torch.int16))
