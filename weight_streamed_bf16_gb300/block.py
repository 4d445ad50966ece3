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

    def __init__(self, shape: BlockShape, arena: Arena, device="cuda", rope=None,
                 attn_tail_split: bool = True):
        """``rope``: (cos, sin) FP32 tables [N x dh/2] (any device), required
        for a pre-norm block.  ``attn_tail_split``: give attention its
        workspace, so the units of a partial last wave are cut into key
        ranges (psi_attn_partitioned_ws); off, every (head, query tile) unit
        is computed whole, the same way at any grid size."""
        s = shape
        self.s = s
        self.arena = arena
        self.attn_tail_split = attn_tail_split
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
        # attention tail-split workspace (FP32 partial states)
        nws = psi.psi_attn_workspace_size(s.key_block)
        self.attn_ws = torch.empty(nws // 4, dtype=torch.float32, device=device)

    def _heads(self, t: torch.Tensor, col0: int, ld: int) -> psi.psi_heads:
        return psi.psi_heads(t.data_ptr() + 2 * col0, ld, self.s.dh)

    def forward(self, X: torch.Tensor, W: BlockWeights, Y: torch.Tensor, flags: int = 0,
                marks=None):
        """Y = block(X); X and Y are [N x d] device BF16 (Y may not alias X).
        ``marks``: optional list of CUDA events recorded on the compute
        stream at the operator boundaries (timing only): 5 of them (start,
        after QKV, attention, out-projection, FFN), 7 for a pre-norm block
        (start, after norm 1, QKV, attention, out-projection, norm 2, FFN)."""
        s, A = self.s, self.arena.handle
        H, dh, N = s.heads, s.dh, s.N
        cs = self.arena.compute

        pn = 1 if s.prenorm else 0

        def mark(i):
            if marks is not None:
                marks[i].record(cs)

        mark(0)
        if s.prenorm:
            psi.psi_rmsnorm(X.data_ptr(), s.d, N, s.d, W.gamma1.data_ptr(), s.eps,
                            self.xn.data_ptr(), s.d, cs.cuda_stream)
            mark(1)
            psi.psi_linear_rope_paged(A, self.xn.data_ptr(), N, s.d, W.qkv.desc(),
                                      W.bqkv.data_ptr(), self.rope, self.h.data_ptr(), s.qkv,
                                      flags)
        else:
            psi.psi_linear_paged(A, X.data_ptr(), N, s.d, W.qkv.desc(), W.bqkv.data_ptr(), None,
                                 self.h.data_ptr(), s.qkv, flags)
        mark(1 + pn)
        q = self._heads(self.h, 0, s.qkv)
        k = self._heads(self.h, H * dh, s.qkv)
        v = self._heads(self.h, 2 * H * dh, s.qkv)
        o = self._heads(self.att, 0, H * dh)
        if self.attn_tail_split:
            psi.psi_attn_partitioned_ws(q, k, v, o, H, N, N, dh, 1.0 / math.sqrt(dh),
                                        s.key_block, self.attn_ws.data_ptr(),
                                        self.attn_ws.numel() * 4, cs.cuda_stream, 0)
        else:
            psi.psi_attn_partitioned(q, k, v, o, H, N, N, dh, 1.0 / math.sqrt(dh), s.key_block,
                                     cs.cuda_stream, 0)
        mark(2 + pn)
        psi.psi_linear_paged(A, self.att.data_ptr(), N, H * dh, W.out.desc(), W.bo.data_ptr(),
                             X.data_ptr(), self.x1.data_ptr(), s.d, flags)
        mark(3 + pn)
        ffn_in = self.x1
        if s.prenorm:
            psi.psi_rmsnorm(self.x1.data_ptr(), s.d, N, s.d, W.gamma2.data_ptr(), s.eps,
                            self.xn.data_ptr(), s.d, cs.cuda_stream)
            mark(5)
            ffn_in = self.xn
        psi.psi_ffn_paged(A, ffn_in.data_ptr(), N, W.ffn.desc(), W.a1.data_ptr(),
                          W.b1.data_ptr(), self.hid.data_ptr(), self.acc.data_ptr(),
                          self.x1.data_ptr(), Y.data_ptr(), flags)
        mark(4 + 2 * pn)

    # ------------------------------------------------- journaled branches --
    ROLE_STATE = 0

    def branch_schedule(self, nblocks: int, nbranch: int, keep_updated: bool = True):
        """(block, branch) steps.  With ``keep_updated`` the branch order
        alternates per block (0..B-1, then B-1..0), so the branch that ends a
        block starts the next one and its updated state stays resident."""
        steps = []
        for b in range(nblocks):
            order = list(range(nbranch))
            if keep_updated and b % 2 == 1:
                order.reverse()
            steps += [(b, r) for r in order]
        return steps

    def run_branches(self, blocks: list, journal, nbranch: int, flags: int = 0,
                     keep_updated: bool = True, inputs=None, outputs=None):
        """Run every block over ``nbranch`` branch states kept in the host
        journal (section II-D).  Branch r's input is entry (0, r, ROLE_STATE),
        or the device tensor inputs[r]; its output becomes entry
        (len(blocks), r, ROLE_STATE), or is written to outputs[r].

        Only three [N x d] state buffers live on the device: the active
        input, the active output, and the next step's input, reloaded while
        the current step computes.  A state that the next step consumes
        directly stays resident (no journal round trip); every other
        updated state is committed, and the superseded entry dropped.  The
        journal orders all copies against the compute stream; the only
        compute-side waits are the fences before a buffer that a commit may
        still be reading is overwritten."""
        s = self.s
        if not hasattr(self, "states"):
            self.states = [torch.empty(s.N, s.d, dtype=torch.bfloat16, device=self.x1.device)
                           for _ in range(3)]
        st = self.states
        L = len(blocks)
        steps = self.branch_schedule(L, nbranch, keep_updated)
        key = lambda b, r: (b, r, self.ROLE_STATE)  # noqa: E731
        committed = set() if inputs is not None else {key(0, r) for r in range(nbranch)}
        last_commit = [-1, -1, -1]          # step index of each buffer's latest commit

        def take(k):                        # reload entry k into buffer idx, then use it
            journal.acquire(k)
            journal.drop(k)
            committed.discard(k)

        b0, r0 = steps[0]
        if inputs is not None:
            cur_t, cur_i = inputs[r0], None
        else:
            cur_t, cur_i = st[0], 0
            journal.reload(key(b0, r0), cur_t)
            take(key(b0, r0))
        for i, (b, r) in enumerate(steps):
            nxt = steps[i + 1] if i + 1 < len(steps) else None
            resident_next = nxt is not None and nxt == (b + 1, r)
            external_next = nxt is not None and inputs is not None and nxt[0] == 0
            to_output = outputs is not None and b == L - 1
            free = sorted((k for k in range(3) if k != cur_i), key=lambda k: last_commit[k])
            pre = None
            if (nxt is not None and not resident_next and not external_next and
                    key(*nxt) in committed):
                pre = free.pop(0)
                journal.reload(key(*nxt), st[pre])
            if to_output:
                out_t, out_i = outputs[r], None
            else:
                out_i = free.pop(0)
                out_t = st[out_i]
            journal.fence(out_t)
            self.forward(cur_t, blocks[b], out_t, flags)
            if not resident_next and not to_output:
                journal.commit(key(b + 1, r), out_t)
                committed.add(key(b + 1, r))
                last_commit[out_i] = i
            if nxt is None:
                break
            if resident_next:
                cur_t, cur_i = out_t, out_i
                continue
            if external_next:
                cur_t, cur_i = inputs[nxt[1]], None
                continue
            if pre is None:                 # its entry was committed just now
                pre = free.pop(0)
                journal.reload(key(*nxt), st[pre])
            take(key(*nxt))
            cur_t, cur_i = st[pre], pre

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
