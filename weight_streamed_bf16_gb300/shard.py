"""Output-column sharding of the synthetic block over several devices.

Every operator of the block is split by output columns: part r of R computes
a contiguous range of each operator's output columns from its own weight
pages, so every output element still receives its complete dot product on
one device and the gathered columns are the single-device result bit for bit
(the column-partition invariant of section II-B; the paper's projection
probes of section IV-B group output columns the same way):

    QKV projection   the Q, K and V rows of the part's heads: three row
                     ranges of Wqkv, each streamed page by page
    attention        the part's heads, read in place (no exchange)
    gather           the attention output of every part (all heads)
    out-projection   the part's rows of Wo -> its columns of x1 (+ X)
    gather           x1
    FFN              every hidden slice J, with U_J (all of it: each output
                     column needs every hidden channel) and the part's rows
                     of V: its own packed page image, pages U_J || V_(c0:c1),J
    gather           y

Sharding the FFN by hidden slices instead would need an FP32 reduction
across devices in another order than the single device's, so it is not used.
Each part streams its own pages through its own arena; the per-part host
bytes per block are 3 of 6 QKV pages, 1 of 2 out-projection pages and 16
FFN pages of 8 + 8/R MiB (R = 2: 256 of 384 MiB).

Attention is bitwise equal to the single-device block when both compute
every (head, query tile) unit whole; the tail split of a partial last wave
(``attn_tail_split``) cuts units by key ranges, which changes the rounding of
those units, and where it falls depends on the number of heads per part.

This module only plans the partition, sequences library calls and, between
phases, gathers column blocks with torch.distributed (NCCL on GPUs; any
backend, e.g. gloo, for the host-side logic).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

from . import psi
from .block import BlockShape
from .torch_io import Arena, FfnWeight, LinearWeight, ffn_workspace

COL_ALIGN = 256   # column boundaries on whole 256-wide page-GEMM tiles


@dataclass(frozen=True)
class ShardPlan:
    """The columns part ``part`` of ``parts`` owns in every operator."""
    shape: BlockShape
    parts: int
    part: int

    @property
    def heads(self) -> tuple[int, int]:
        return psi.psi_plan_columns(self.shape.heads, 1, self.parts, self.part)

    @property
    def qkv_rows(self) -> list[tuple[int, int]]:
        """Rows of Wqkv (= columns of h) for the part's Q, K and V heads."""
        s = self.shape
        h0, h1 = self.heads
        w = s.heads * s.dh
        return [(p * w + h0 * s.dh, p * w + h1 * s.dh) for p in range(3)]

    @property
    def att_cols(self) -> tuple[int, int]:
        h0, h1 = self.heads
        return h0 * self.shape.dh, h1 * self.shape.dh

    @property
    def out_cols(self) -> tuple[int, int]:
        """Columns of x1 and y (rows of Wo and of V)."""
        return psi.psi_plan_columns(self.shape.d, COL_ALIGN, self.parts, self.part)

    def all(self, attr: str) -> list[tuple[int, int]]:
        """``attr``'s ranges of every part, in part order."""
        return [getattr(ShardPlan(self.shape, self.parts, q), attr) for q in range(self.parts)]


class ShardWeights:
    """One part's weights: views of the block's pinned host weights for the
    projections (row ranges, streamed in place) and its own packed FFN page
    image (U_J with the part's rows of V)."""

    def __init__(self, w: dict, plan: ShardPlan, resident: bool = False, device="cuda"):
        s = plan.shape
        self.plan = plan
        pb = s.page_bytes
        Wqkv, Wo = w["Wqkv"], w["Wo"]
        self.qkv = [LinearWeight(Wqkv[r0:r1], pb, resident=resident, device=device)
                    for r0, r1 in plan.qkv_rows]
        c0, c1 = plan.out_cols
        self.out = LinearWeight(Wo[c0:c1], pb, resident=resident, device=device)
        self.ffn = FfnWeight(w["W1"], w["W2"][c0:c1], s.slice, resident=resident, device=device)
        if self.ffn.page_bytes > pb:
            raise ValueError("FFN page does not fit the page size")
        dev = torch.device(device)
        self.bqkv = [w["bqkv"][r0:r1].to(dev) for r0, r1 in plan.qkv_rows]
        self.bo = w["bo"][c0:c1].to(dev)
        self.a1 = w["a1"].to(dev)
        self.b1 = w["b1"][c0:c1].to(dev)
        self.gamma1 = w["gamma1"].to(dev) if "gamma1" in w else None
        self.gamma2 = w["gamma2"].to(dev) if "gamma2" in w else None

    @property
    def host_bytes(self) -> int:
        return (sum(q.host.numel() for q in self.qkv) * 2 + self.out.host.numel() * 2 +
                self.ffn.host.numel())


class ShardBuffers:
    """Full-width activations of the block on one device.  A part writes
    only its own columns of each; the gathers fill in the others'."""

    def __init__(self, shape: BlockShape, device="cuda"):
        s = shape
        dev = torch.device(device)
        self.h = torch.empty(s.N, s.qkv, dtype=torch.bfloat16, device=dev)
        self.att = torch.empty(s.N, s.heads * s.dh, dtype=torch.bfloat16, device=dev)
        self.x1 = torch.empty(s.N, s.d, dtype=torch.bfloat16, device=dev)
        self.xn = (torch.empty(s.N, s.d, dtype=torch.bfloat16, device=dev)
                   if s.prenorm else None)


class ShardRunner:
    """The phases of one part's share of a block forward, on one arena."""

    PHASES = ("qkv", "attention", "out_proj", "ffn")
    GATHERED = {"attention": "att", "out_proj": "x1", "ffn": "y"}

    def __init__(self, plan: ShardPlan, arena: Arena, bufs: ShardBuffers, device="cuda",
                 rope=None, attn_tail_split: bool = False):
        s = plan.shape
        self.plan, self.s, self.arena, self.b = plan, s, arena, bufs
        c0, c1 = plan.out_cols
        self.hid, self.acc = ffn_workspace(s.N, max(c1 - c0, 8), s.slice, device)
        self.attn_tail_split = attn_tail_split
        nws = psi.psi_attn_workspace_size(s.key_block)
        self.attn_ws = (torch.empty(nws // 4, dtype=torch.float32, device=device)
                        if attn_tail_split else None)
        if s.prenorm:
            if rope is None:
                raise ValueError("a pre-norm block needs the RoPE tables")
            self.cos = rope[0].to(device=device, dtype=torch.float32).contiguous()
            self.sin = rope[1].to(device=device, dtype=torch.float32).contiguous()

    def _heads(self, t: torch.Tensor, col0: int, ld: int) -> psi.psi_heads:
        return psi.psi_heads(t.data_ptr() + 2 * col0, ld, self.s.dh)

    def gathered(self, Y: torch.Tensor) -> dict:
        """The tensors gathered after the phases: attention output, x1, y."""
        return {"att": self.b.att, "x1": self.b.x1, "y": Y}

    def run_phase(self, name: str, X, W, Y, flags: int = 0):
        """Enqueue a phase on the arena's compute stream."""
        with torch.cuda.stream(self.arena.compute):
            self.phase(name, X, W, Y, flags)

    def before_collective(self):
        """The collective's stream (torch's current one) waits for the phase."""
        torch.cuda.current_stream().wait_stream(self.arena.compute)

    def after_collective(self):
        """The compute stream waits for the gathered columns."""
        self.arena.compute.wait_stream(torch.cuda.current_stream())

    def phase(self, name: str, X: torch.Tensor, W: ShardWeights, Y: torch.Tensor,
              flags: int = 0):
        """Enqueue phase ``name`` of this part on the arena's compute stream:
        X, Y [N x d] device BF16 (the block input and output)."""
        s, A, b, p = self.s, self.arena.handle, self.b, self.plan
        cs = self.arena.compute
        N = s.N
        if name == "qkv":
            src = X
            if s.prenorm:
                psi.psi_rmsnorm(X.data_ptr(), s.d, N, s.d, W.gamma1.data_ptr(), s.eps,
                                b.xn.data_ptr(), s.d, cs.cuda_stream)
                src = b.xn
            for part, ((r0, r1), w, bias) in enumerate(zip(p.qkv_rows, W.qkv, W.bqkv)):
                out = b.h.data_ptr() + 2 * r0
                if s.prenorm and part < 2:      # the query and key heads are rotated
                    rope = psi.psi_rope(self.cos.data_ptr(), self.sin.data_ptr(), s.dh // 2,
                                        r1 - r0, s.dh, 0)
                    psi.psi_linear_rope_paged(A, src.data_ptr(), N, s.d, w.desc(),
                                              bias.data_ptr(), rope, out, s.qkv, flags)
                else:
                    psi.psi_linear_paged(A, src.data_ptr(), N, s.d, w.desc(), bias.data_ptr(),
                                         None, out, s.qkv, flags)
        elif name == "attention":
            h0, h1 = p.heads
            if h1 == h0:
                return
            (q0, _), (k0, _), (v0, _) = p.qkv_rows
            q = self._heads(b.h, q0, s.qkv)
            k = self._heads(b.h, k0, s.qkv)
            v = self._heads(b.h, v0, s.qkv)
            o = self._heads(b.att, p.att_cols[0], s.heads * s.dh)
            sc = 1.0 / math.sqrt(s.dh)
            if self.attn_tail_split:
                psi.psi_attn_partitioned_ws(q, k, v, o, h1 - h0, N, N, s.dh, sc, s.key_block,
                                            self.attn_ws.data_ptr(), self.attn_ws.numel() * 4,
                                            cs.cuda_stream, 0)
            else:
                psi.psi_attn_partitioned(q, k, v, o, h1 - h0, N, N, s.dh, sc, s.key_block,
                                         cs.cuda_stream, 0)
        elif name == "out_proj":
            c0, c1 = p.out_cols
            if c1 == c0:
                return
            psi.psi_linear_paged(A, b.att.data_ptr(), N, s.heads * s.dh, W.out.desc(),
                                 W.bo.data_ptr(), X.data_ptr() + 2 * c0,
                                 b.x1.data_ptr() + 2 * c0, s.d, flags)
        elif name == "ffn":
            c0, c1 = p.out_cols
            if c1 == c0:
                return
            src = b.x1
            if s.prenorm:
                psi.psi_rmsnorm(b.x1.data_ptr(), s.d, N, s.d, W.gamma2.data_ptr(), s.eps,
                                b.xn.data_ptr(), s.d, cs.cuda_stream)
                src = b.xn
            psi.psi_ffn_paged_strided(A, src.data_ptr(), N, W.ffn.desc(), W.a1.data_ptr(),
                                      W.b1.data_ptr(), self.hid.data_ptr(), self.acc.data_ptr(),
                                      b.x1.data_ptr() + 2 * c0, Y.data_ptr() + 2 * c0, s.d,
                                      flags)
        else:
            raise ValueError(f"unknown phase {name}")


def gather_columns(T: torch.Tensor, ranges: list[tuple[int, int]], rank: int, group=None):
    """All-gather column blocks of a row-major [rows x cols] tensor: rank q
    owns columns ranges[q] of T (every range the same width); afterwards
    every rank holds every block.  One all_gather of contiguous copies, then
    each block is placed at its columns."""
    import torch.distributed as dist
    widths = {b - a for a, b in ranges}
    if len(widths) != 1:
        raise ValueError("gather_columns needs column blocks of equal width")
    c0, c1 = ranges[rank]
    own = T[:, c0:c1].contiguous()
    parts = [torch.empty_like(own) for _ in ranges]
    dist.all_gather(parts, own, group=group)
    for q, (a, b) in enumerate(ranges):
        if q != rank:
            T[:, a:b].copy_(parts[q])


def forward_sharded(runner, X: torch.Tensor, W, Y: torch.Tensor, flags: int = 0, group=None):
    """One block forward of this rank's part, with the column gathers
    between phases (torch.distributed, one process per device): after the
    attention phase the attention output, after the out-projection x1, after
    the FFN y.  ``runner`` is a ShardRunner (or any object with its
    ``plan``, ``run_phase``, ``gathered``, ``before_collective`` and
    ``after_collective``); the collective runs on torch's current stream,
    ordered after the phase and before the next one by the runner's hooks."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    plan = runner.plan
    ranges = {"att": plan.all("att_cols"), "x1": plan.all("out_cols"),
              "y": plan.all("out_cols")}
    bufs = runner.gathered(Y)
    for name in ShardRunner.PHASES:
        runner.run_phase(name, X, W, Y, flags)
        g = ShardRunner.GATHERED.get(name)
        if g is not None:
            runner.before_collective()
            gather_columns(bufs[g], ranges[g], rank, group)
            runner.after_collective()


def forward_parts_in_turn(runners: list[ShardRunner], X: torch.Tensor, weights: list,
                          Y: torch.Tensor, flags: int = 0):
    """Every part of a block forward on this one device, phase by phase,
    all parts writing their columns into the same full-width buffers (the
    gathers are then no-ops): the exactness check of the partition on one
    GPU.  ``runners`` share one ShardBuffers and one arena."""
    for name in ShardRunner.PHASES:
        for rn, W in zip(runners, weights):
            rn.phase(name, X, W, Y, flags)
