"""Helpers for the GPU parity tests: run an operator through the C ABI and
hand the same input bytes to the oracle."""
from __future__ import annotations

import numpy as np
import torch

from oracle import bf16, grade, ops
from weight_streamed_bf16_gb300 import build, psi
from weight_streamed_bf16_gb300.torch_io import (Arena, FfnWeight, LinearWeight,
                                                 ffn_workspace, heads_view)

_built = False


def ensure_lib():
    global _built
    if not _built:
        build.build()
        psi.load()
        _built = True


def f64(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor -> float64 values through the oracle's own decoder."""
    bits = t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return bf16.decode(bits)


def run_linear(X, W, b, page_rows, slots, flags=0, residual=None, arena=None, ldy=None):
    """X, W, b: CPU bf16.  Returns the GPU output (CPU bf16 tensor)."""
    N, K = X.shape
    M = W.shape[0]
    ldy = ldy or (M + 7) // 8 * 8   # row stride: a multiple of 8 elements
    dev = torch.device("cuda")
    Xd = X.to(dev)
    bd = b.to(dev)
    Y = torch.full((N, ldy), float("nan"), dtype=torch.bfloat16, device=dev)
    Rd = None
    if residual is not None:
        Rd = torch.zeros((N, ldy), dtype=torch.bfloat16, device=dev)
        Rd[:, :M] = residual.to(dev)
    page_bytes = page_rows * K * 2
    page_bytes = (page_bytes + 1023) // 1024 * 1024
    own = arena is None
    if own:
        arena = Arena(page_bytes, slots)
    w = LinearWeight(W, page_bytes, page_rows=page_rows, resident=bool(flags & psi.PSI_RESIDENT))
    psi.psi_linear_paged(arena.handle, Xd.data_ptr(), N, K, w.desc(), bd.data_ptr(),
                         Rd.data_ptr() if Rd is not None else None, Y.data_ptr(), ldy, flags)
    arena.sync()
    out = Y[:, :M].cpu()
    if own:
        arena.close()
    return out


def run_ffn(X, U, V, a, b, slice_, slots, flags=0, residual=None, return_hidden=False):
    N, d = X.shape
    r = V.shape[0]
    dev = torch.device("cuda")
    Xd, ad, bd = X.to(dev), a.to(dev), b.to(dev)
    Rd = residual.to(dev) if residual is not None else None
    Y = torch.full((N, r), float("nan"), dtype=torch.bfloat16, device=dev)
    w = FfnWeight(U, V, slice_, resident=bool(flags & psi.PSI_RESIDENT))
    arena = Arena((w.page_bytes + 1023) // 1024 * 1024, slots)
    hid, acc = ffn_workspace(N, r, slice_)
    psi.psi_ffn_paged(arena.handle, Xd.data_ptr(), N, w.desc(), ad.data_ptr(), bd.data_ptr(),
                      hid.data_ptr(), acc.data_ptr(),
                      Rd.data_ptr() if Rd is not None else None, Y.data_ptr(), flags)
    arena.sync()
    stats = arena.stats()
    arena.close()
    S = U.shape[0] // slice_
    G = 2 if (S >= 2 and slice_ % 64 == 0) else 1   # slices per down pass (psi.h)
    g, u = (S - 1) // G, (S - 1) % G
    last = hid.view(2, N, 2 * slice_)[g & 1][:, u * slice_:(u + 1) * slice_].cpu()
    if return_hidden:
        return Y.cpu(), last, stats
    return Y.cpu()


def run_attention(Q, K, V, scale, key_block=128, O=None, split=False, flags=0):
    """Q [H x Nq x dh], K, V [H x Nk x dh] (device bf16 views); returns O.
    ``split``: pass a workspace, so a partial last wave is split by keys."""
    H, Nq, dh = Q.shape
    Nk = K.shape[1]
    if O is None:
        O = torch.full((H, Nq, dh), float("nan"), dtype=torch.bfloat16, device=Q.device)
    s = torch.cuda.current_stream()
    if split:
        n = psi.psi_attn_workspace_size(key_block)
        ws = torch.full((n // 4,), float("nan"), dtype=torch.float32, device=Q.device)
        psi.psi_attn_partitioned_ws(heads_view(Q), heads_view(K), heads_view(V), heads_view(O),
                                    H, Nq, Nk, dh, scale, key_block, ws.data_ptr(), n,
                                    s.cuda_stream, flags)
    else:
        psi.psi_attn_partitioned(heads_view(Q), heads_view(K), heads_view(V), heads_view(O), H,
                                 Nq, Nk, dh, scale, key_block, s.cuda_stream, flags)
    psi.psi_stream_wait(s.cuda_stream, 120000)
    return O


def run_linear_rope(X, W, b, cos, sin, dh, cols, page_rows, slots, flags=0):
    """Paged QKV-style projection with split RoPE on the first ``cols``
    output columns; cos/sin are [N x dh/2] float32 CPU tables."""
    N, K = X.shape
    M = W.shape[0]
    ldy = (M + 7) // 8 * 8
    dev = torch.device("cuda")
    Xd, bd = X.to(dev), b.to(dev)
    cd = cos.to(dev).contiguous()
    sd = sin.to(dev).contiguous()
    Y = torch.full((N, ldy), float("nan"), dtype=torch.bfloat16, device=dev)
    page_bytes = (page_rows * K * 2 + 1023) // 1024 * 1024
    arena = Arena(page_bytes, slots)
    w = LinearWeight(W, page_bytes, page_rows=page_rows, resident=bool(flags & psi.PSI_RESIDENT))
    rope = psi.psi_rope(cd.data_ptr(), sd.data_ptr(), cd.shape[1], cols, dh, 0)
    try:
        psi.psi_linear_rope_paged(arena.handle, Xd.data_ptr(), N, K, w.desc(), bd.data_ptr(),
                                  rope, Y.data_ptr(), ldy, flags)
        arena.sync()
    finally:
        arena.close()
    return Y[:, :M].cpu()


def run_rmsnorm(X, gamma, eps, ldx=None, ldy=None):
    """X [N x d] CPU bf16 -> GPU RMSNorm output (CPU bf16 [N x d])."""
    N, d = X.shape
    ldx = ldx or d
    ldy = ldy or d
    dev = torch.device("cuda")
    Xb = torch.zeros((N, ldx), dtype=torch.bfloat16)
    Xb[:, :d] = X
    Xd = Xb.to(dev)
    gd = gamma.to(dev)
    Y = torch.full((N, ldy), float("nan"), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.current_stream()
    psi.psi_rmsnorm(Xd.data_ptr(), ldx, N, d, gd.data_ptr(), eps, Y.data_ptr(), ldy,
                    s.cuda_stream)
    torch.cuda.synchronize()
    return Y[:, :d].cpu()


# Every parity call: each element within 2 graded BF16 ulp of the oracle,
# the normwise error max|dy| / max|y_oracle| at most 1e-2, and at most one
# element in a thousand that passes only because of the oracle's slack for
# ambiguous inner roundings (a correct FP32 evaluation flips such a rounding
# rarely; a kernel leaning on the slack everywhere would be wrong).
MAX_REL_ERR = 1e-2
MAX_SLACK_FRAC = 1e-3


def check(y_gpu: torch.Tensor, res, tol=2.0, what=""):
    rep = grade.report(f64(y_gpu), res, tol)
    print(f"{what}: n {rep['n']} max graded {rep['max_graded_ulps']:.3f} ulp, max raw "
          f"{rep['max_raw_ulps']}, differing {rep['n_differing']}, max rel "
          f"{rep['max_rel_err']:.3e}, rel L2 {rep['rel_l2']:.3e}, pass by slack "
          f"{rep['n_pass_by_slack']}")
    assert rep["pass"], f"{what}: {rep}"
    assert rep["max_rel_err"] <= MAX_REL_ERR, f"{what}: {rep}"
    assert rep["n_pass_by_slack"] <= MAX_SLACK_FRAC * rep["n"], f"{what}: {rep}"
    return rep


__all__ = ["ensure_lib", "f64", "run_linear", "run_linear_rope", "run_rmsnorm", "run_ffn",
           "run_attention", "check", "ops",
           "grade", "bf16"]
