"""Full-row RMSNorm and split RoPE (PSI section II-B) on the GPU against the
oracle: the RMSNorm kernel, and the projection whose epilogue rotates the
query and key heads before its single BF16 write."""
import math

import numpy as np
import pytest
import torch

import psi_synth
from weight_streamed_bf16_gb300 import psi

from gpu_cases import (bf16, check, ensure_lib, f64, ops, run_linear, run_linear_rope,
                       run_rmsnorm)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _bf16(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


def _f32(x):
    return np.float64(np.float32(x))


# ---------------------------------------------------------------- RMSNorm --
@pytest.mark.parametrize("N,d", [
    (1, 8),         # one vector per row, most lanes idle
    (37, 200),      # ragged width (25 vectors), ragged row count
    (300, 2048),    # 8 vectors per lane
    (129, 4096),    # the block width: 16 vectors per lane kept in registers
    (40, 6144),     # wider than registers hold: the row is read twice
    (16, 8192),     # the widest row handled
])
def test_rmsnorm_shapes(N, d):
    X = _bf16((N, d), 2.0, N + d)
    g = (1 + 0.1 * torch.randn(d, generator=torch.Generator().manual_seed(d))).to(torch.bfloat16)
    eps = 1e-6
    Y = run_rmsnorm(X, g, eps)
    res = ops.rmsnorm(f64(X), f64(g), _f32(eps))
    check(Y, res, what=f"rmsnorm {N}x{d}")


def test_rmsnorm_strided_rows_and_large_eps():
    X = _bf16((50, 512), 0.01, 3)
    g = _bf16((512,), 1.0, 4)
    eps = 0.25   # comparable to the mean square: eps must sit inside the root
    Y = run_rmsnorm(X, g, eps, ldx=520, ldy=640)
    check(Y, ops.rmsnorm(f64(X), f64(g), _f32(eps)), what="strided")


def test_rmsnorm_zero_rows_and_block_shape():
    """The block's normalisation: 6144 x 4096, every row checked; a zero row
    gives zeros (eps keeps the denominator positive)."""
    cfg = psi_synth.BLOCK
    X = psi_synth.block_input(cfg).clone()
    X[5] = 0
    g1, _ = psi_synth.norm_gains(cfg)
    Y = run_rmsnorm(X, g1, cfg.eps)
    assert torch.count_nonzero(Y[5].float()) == 0
    rep = check(Y, ops.rmsnorm(f64(X), f64(g1), _f32(cfg.eps)), what="block rmsnorm")
    assert rep["max_rel_err"] <= 1e-2


# ------------------------------------------------------------ split RoPE --
@pytest.mark.parametrize("N,H,dh,page_rows", [
    (100, 2, 128, 256),    # one CTA per tile (N < 256), 256-column tiles
    (77, 4, 64, 128),      # 64-wide heads, two per epilogue warp
    (512, 4, 128, 512),    # CTA pairs (256 x 256 tiles)
    (300, 4, 128, 384),    # pairs with ragged tokens; 384-row pages split tiles
    (600, 2, 64, 192),     # ragged pages (3 x 64-wide heads per page)
])
def test_linear_rope_shapes(N, H, dh, page_rows):
    K = 256
    M = 3 * H * dh                    # Q, K, V heads; RoPE on Q and K
    X = _bf16((N, K), 1.0, N + H)
    W = _bf16((M, K), 1 / math.sqrt(K), M)
    b = _bf16((M,), 0.5, 7)
    cos, sin = psi_synth.rope_table(N, dh, pos0=3)
    Y = run_linear_rope(X, W, b, cos, sin, dh, 2 * H * dh, page_rows, 2)
    res = ops.linear_rope(f64(X), f64(W), f64(b), cos.double().numpy(), sin.double().numpy(),
                          dh, 2 * H * dh)
    check(Y, res, what=f"rope {N}x{M} dh{dh}")
    # the pass-through (value) heads equal the plain projection bitwise
    plain = run_linear(X, W, b, page_rows, 2)
    assert torch.equal(Y[:, 2 * H * dh:].view(torch.int16), plain[:, 2 * H * dh:].view(torch.int16))


@pytest.mark.parametrize("N,H,dh,page_rows", [
    (512, 4, 128, 256),    # six pages: pairs across the Q/K and the rotated/plain boundaries
    (300, 6, 64, 256),     # ragged tokens, 64-wide heads, a short last page alone
])
def test_linear_rope_page_pairs_bitwise(N, H, dh, page_rows):
    """With four or more ring slots, streamed pages after the first go two to
    a launch with the RoPE epilogue too; the bytes equal one page per launch
    (two slots) and the resident single launch."""
    K = 256
    M = 3 * H * dh
    X = _bf16((N, K), 1.0, N + 3 * H)
    W = _bf16((M, K), 1 / math.sqrt(K), M + 1)
    b = _bf16((M,), 0.5, 11)
    cos, sin = psi_synth.rope_table(N, dh, pos0=5)
    pages = -(-M // page_rows)
    n0 = psi.psi_kernel_launches()
    merged = run_linear_rope(X, W, b, cos, sin, dh, 2 * H * dh, page_rows, 5)
    n1 = psi.psi_kernel_launches()
    single = run_linear_rope(X, W, b, cos, sin, dh, 2 * H * dh, page_rows, 2)
    n2 = psi.psi_kernel_launches()
    res = run_linear_rope(X, W, b, cos, sin, dh, 2 * H * dh, page_rows, 2,
                          flags=psi.PSI_RESIDENT)
    assert n2 - n1 == pages and n1 - n0 < pages
    assert torch.equal(merged.view(torch.int16), single.view(torch.int16))
    assert torch.equal(merged.view(torch.int16), res.view(torch.int16))
    ref = ops.linear_rope(f64(X), f64(W), f64(b), cos.double().numpy(), sin.double().numpy(),
                          dh, 2 * H * dh)
    check(merged, ref, what=f"rope page pairs {N}x{M} dh{dh}")


def test_linear_rope_identity_table_is_plain_projection():
    """c = 1, s = 0: the rotated columns equal the plain projection bitwise."""
    N, K, dh, H = 300, 512, 128, 2
    M = 3 * H * dh
    X = _bf16((N, K), 1.0, 11)
    W = _bf16((M, K), 1 / math.sqrt(K), 12)
    b = _bf16((M,), 0.1, 13)
    cos = torch.ones(N, dh // 2)
    sin = torch.zeros(N, dh // 2)
    Y = run_linear_rope(X, W, b, cos, sin, dh, 2 * H * dh, 256, 2)
    plain = run_linear(X, W, b, 256, 2)
    assert torch.equal(Y.view(torch.int16), plain.view(torch.int16))


def test_linear_rope_resident_equals_streamed():
    N, K, dh, H = 512, 256, 128, 4
    M = 3 * H * dh
    X = _bf16((N, K), 1.0, 21)
    W = _bf16((M, K), 1 / math.sqrt(K), 22)
    b = _bf16((M,), 0.1, 23)
    cos, sin = psi_synth.rope_table(N, dh)
    a = run_linear_rope(X, W, b, cos, sin, dh, 2 * H * dh, 512, 2)
    r = run_linear_rope(X, W, b, cos, sin, dh, 2 * H * dh, 512, 2, flags=psi.PSI_RESIDENT)
    assert torch.equal(a.view(torch.int16), r.view(torch.int16))


@pytest.mark.parametrize("flags", [psi.PSI_ROPE_AFTER_BF16,
                                   psi.PSI_ROPE_AFTER_BF16 | psi.PSI_BIAS_AFTER_BF16])
def test_linear_rope_baseline_materialisation(flags):
    """The baseline order rounds the projection before rotating it."""
    N, K, dh, H = 256, 256, 128, 2
    M = 3 * H * dh
    X = _bf16((N, K), 1.0, 31)
    W = _bf16((M, K), 1 / math.sqrt(K), 32)
    b = _bf16((M,), 0.5, 33)
    cos, sin = psi_synth.rope_table(N, dh, pos0=100)
    Y = run_linear_rope(X, W, b, cos, sin, dh, 2 * H * dh, 256, 2, flags=flags)
    if flags & psi.PSI_BIAS_AFTER_BF16:
        base = ops.linear(f64(X), f64(W), f64(b), bias_after_bf16=True)
        rot = ops.rope_split(base.y, cos.double().numpy(), sin.double().numpy(), dh, 2 * H * dh)
        # the rotated columns: B(rope(B(B(XW^T) + b))) within 1 ulp of the
        # oracle's rotation of its own baseline projection (ambiguous inner
        # roundings are rare at these sizes)
        Yf = f64(Y)[:, :2 * H * dh]
        want = bf16.round_bf16(rot)[:, :2 * H * dh]
        du = np.abs(Yf - want) / bf16.ulp(want)
        assert (du <= 1).mean() > 0.999
    else:
        res = ops.linear_rope(f64(X), f64(W), f64(b), cos.double().numpy(),
                              sin.double().numpy(), dh, 2 * H * dh, rope_after_bf16=True)
        check(Y, res, what="rope after bf16")
        exact = ops.linear_rope(f64(X), f64(W), f64(b), cos.double().numpy(),
                                sin.double().numpy(), dh, 2 * H * dh)
        n_base = int(np.count_nonzero(f64(Y) != exact.y))
        mod = run_linear_rope(X, W, b, cos, sin, dh, 2 * H * dh, 256, 2)
        n_mod = int(np.count_nonzero(f64(mod) != exact.y))
        assert n_base > 5 * n_mod, (n_base, n_mod)


def test_linear_rope_rejects_bad_heads():
    X = _bf16((8, 64), 1.0, 1)
    W = _bf16((3 * 128, 64), 0.1, 2)
    b = _bf16((3 * 128,), 0.1, 3)
    cos, sin = psi_synth.rope_table(8, 128)
    with pytest.raises(psi.PsiError) as e:
        run_linear_rope(X, W, b, cos, sin, 128, 200, 384, 2)   # not whole heads
    assert e.value.status == psi.PSI_ERR_INVALID_ARG
    with pytest.raises(psi.PsiError) as e:
        run_linear_rope(X, W, b, cos, sin, 128, 256, 192, 2)   # page splits a head
    assert e.value.status == psi.PSI_ERR_INVALID_ARG
