"""Synthetic transformer block and stack over the C ABI.

Composition of one block (operator shapes of the paged-operator study):

    h  = B(X Wqkv^T + bqkv)                      psi_linear_paged   [N x 3*H*dh]
    a  = attention(Q, K, V), heads read in place  psi_attn_partitioned [N x H*dh]
    x1 = B(X + a Wo^T + bo)                      psi_linear_paged (residual X)
    y  = B(x1 + F(x1))                           psi_ffn_paged (residual x1)

With ``BlockShape.prenorm`` the block is a pre-norm block with the two
partitioned operators of section II-B:

    n0 = RMSNorm(X; gamma1)                      psi_rmsnorm
    h  = B(rope(n0 Wqkv^T + bqkv))               psi_linear_rope_paged (Q, K heads)
    a, x1 as above
    n1 = RMSNorm(x1; gamma2)                     psi_rmsnorm
    y  = B(x1 + F(n1))                           psi_ffn_paged (residual x1)

Weights live in pinned host memory and stream through one arena; the page
ring continues across operators and blocks, so it never drains between
them.  This module only sequences library calls and holds buffers.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

from . import psi
from .torch_io import Arena, FfnWeight, LinearWeight, ffn_workspace


@dataclass
class BlockShape:
    d: int = 4096
    N: int = 6144
    heads: int = 32
    dh: int = 128
    hidden: int = 16384
    slice: int = 1024
    page_bytes: int = 16 << 20
    key_block: int = 128
    prenorm: bool = False
    eps: float = 1e-6

    @property
    def qkv(self) -> int:
        return 3 * self.heads * self.dh


class BlockWeights:
    """Pinned host copies (and optional resident device copies) of one block."""

    def __init__(self, w: dict, shape: BlockShape, resident: bool = False, device="cuda"):
        s = shape
        self.shape = s
        self.qkv = LinearWeight(w["Wqkv"], s.page_bytes, resident=resident, device=device)
        self.out = LinearWeight(w["Wo"], s.page_bytes, resident=resident, device=device)
        self.ffn = FfnWeight(w["W1"], w["W2"], s.slice, resident=resident, device=device)
        if self.ffn.page_bytes > s.page_bytes:
            raise ValueError("FFN page does not fit the page size")
        self.bqkv = w["bqkv"].to(device)
        self.bo = w["bo"].to(device)
        self.a1 = w["a1"].to(device)
        self.b1 = w["b1"].to(device)
        self.gamma1 = w["gamma1"].to(device) if "gamma1" in w else None
        self.gamma2 = w["gamma2"].to(device) if "gamma2" in w else None
        if s.prenorm and (self.gamma1 is None or self.gamma2 is None):
            raise ValueError("a pre-norm block needs gamma1 and gamma2")

    @property
    def host_bytes(self) -> int:
        return (self.qkv.host.numel() * 2 + self.out.host.numel() * 2 +
                self.ffn.host.numel())


class BlockRunner:
    """Activation buffers and the arena for running blocks on one device."""

    def __init__(self, shape: BlockShape, arena: Arena, device="cuda", rope=None):
        """``rope``: (cos, sin) FP32 tables [N x dh/2] (any device), required
        for a pre-norm block."""
        s = shape
        self.s = s
        self.arena = arena
        self.xn = None
        if s.prenorm:
            if rope is None:
                raise ValueError("a pre-norm block needs the RoPE tables")
            self.cos = rope[0].to(device=device, dtype=torch.float32).contiguous()
            self.sin = rope[1].to(device=device, dtype=torch.float32).contiguous()
            if self.cos.shape != (s.N, s.dh // 2) or self.sin.shape != self.cos.shape:
                raise ValueError("RoPE tables must be [N x dh/2]")
            self.rope = psi.psi_rope(self.cos.data_ptr(), self.sin.data_ptr(), s.dh // 2,
                                     2 * s.heads * s.dh, s.dh, 0)
            self.xn = torch.empty(s.N, s.d, dtype=torch.bfloat16, device=device)
        self.h = torch.empty(s.N, s.qkv, dtype=torch.bfloat16, device=device)
        self.att = torch.empty(s.N, s.heads * s.dh, dtype=torch.bfloat16, device=device)
        self.x1 = torch.empty(s.N, s.d, dtype=torch.bfloat16, device=device)
        self.hid, self.acc = ffn_workspace(s.N, s.d, s.slice, device)
        self.attn_launches = 0

    def _heads(self, t: torch.Tensor, col0: int, ld: int) -> psi.psi_heads:
        return psi.psi_heads(t.data_ptr() + 2 * col0, ld, self.s.dh)

    def forward(self, X: torch.Tensor, W: BlockWeights, Y: torch.Tensor, flags: int = 0,
                marks=None):
        """Y = block(X); X and Y are [N x d] device BF16 (Y may not alias X).
        ``marks``: optional list of 5 CUDA events recorded on the compute
        stream at the operator boundaries (timing only)."""
        s, A = self.s, self.arena.handle
        H, dh, N = s.heads, s.dh, s.N
        cs = self.arena.compute

        def mark(i):
            if marks is not None:
                marks[i].record(cs)

        mark(0)
        if s.prenorm:
            psi.psi_rmsnorm(X.data_ptr(), s.d, N, s.d, W.gamma1.data_ptr(), s.eps,
                            self.xn.data_ptr(), s.d, cs.cuda_stream)
            psi.psi_linear_rope_paged(A, self.xn.data_ptr(), N, s.d, W.qkv.desc(),
                                      W.bqkv.data_ptr(), self.rope, self.h.data_ptr(), s.qkv,
                                      flags)
        else:
            psi.psi_linear_paged(A, X.data_ptr(), N, s.d, W.qkv.desc(), W.bqkv.data_ptr(), None,
                                 self.h.data_ptr(), s.qkv, flags)
        mark(1)
        q = self._heads(self.h, 0, s.qkv)
        k = self._heads(self.h, H * dh, s.qkv)
        v = self._heads(self.h, 2 * H * dh, s.qkv)
        o = self._heads(self.att, 0, H * dh)
        psi.psi_attn_partitioned(q, k, v, o, H, N, N, dh, 1.0 / math.sqrt(dh), s.key_block,
                                 cs.cuda_stream, 0)
        self.attn_launches += 1
        mark(2)
        psi.psi_linear_paged(A, self.att.data_ptr(), N, H * dh, W.out.desc(), W.bo.data_ptr(),
                             X.data_ptr(), self.x1.data_ptr(), s.d, flags)
        mark(3)
        ffn_in = self.x1
        if s.prenorm:
            psi.psi_rmsnorm(self.x1.data_ptr(), s.d, N, s.d, W.gamma2.data_ptr(), s.eps,
                            self.xn.data_ptr(), s.d, cs.cuda_stream)
            ffn_in = self.xn
        psi.psi_ffn_paged(A, ffn_in.data_ptr(), N, W.ffn.desc(), W.a1.data_ptr(),
                          W.b1.data_ptr(), self.hid.data_ptr(), self.acc.data_ptr(),
                          self.x1.data_ptr(), Y.data_ptr(), flags)
        mark(4)

    def stack(self, X: torch.Tensor, blocks: list, Y: torch.Tensor, tmp: torch.Tensor,
              flags: int = 0):
        """Run blocks in order; X is preserved, the result lands in Y."""
        src = X
        bufs = [Y, tmp] if len(blocks) % 2 == 1 else [tmp, Y]
        for i, W in enumerate(blocks):
            dst = bufs[i % 2]
            self.forward(src, W, dst, flags)
            src = dst
        return Y
