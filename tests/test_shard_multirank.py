"""Output-column sharding, host side (CPU, gloo): the partition plan and the
column gathers between the block's phases.

Two gloo ranks each compute their part's columns of the out-projection,
the FFN and the attention heads with the oracle standing in for the GPU
kernels, gather them with the same ``gather_columns`` the GPU path uses,
and compare the gathered tensors with the unsharded oracle bit for bit:
the column-partition invariant of section II-B (each output entry gets its
complete dot product on one device).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from weight_streamed_bf16_gb300 import build, psi


@pytest.fixture(scope="module")
def lib():
    build.build()
    return psi.load()


def test_plan_columns_partitions(lib):
    for cols, align, parts in [(4096, 256, 2), (4096, 256, 3), (4096, 256, 8), (100, 64, 4),
                               (12288, 128, 5), (0, 8, 3), (7, 1, 7)]:
        rs = [psi.psi_plan_columns(cols, align, parts, r) for r in range(parts)]
        assert rs[0][0] == 0 and rs[-1][1] == cols
        for (a0, a1), (b0, b1) in zip(rs, rs[1:]):
            assert a1 == b0                          # contiguous, disjoint, ordered
        for a, b in rs:
            assert a <= b and (a % align == 0 or a == cols) and (b % align == 0 or b == cols)
        widths = [b - a for a, b in rs]
        assert max(widths) - min(widths) <= align
        assert widths == sorted(widths, reverse=True)   # larger parts first
    for bad in [(-1, 8, 2, 0), (8, 0, 2, 0), (8, 8, 0, 0), (8, 8, 2, 2), (8, 8, 2, -1)]:
        with pytest.raises(psi.PsiError) as e:
            psi.psi_plan_columns(*bad)
        assert e.value.status == psi.PSI_ERR_INVALID_ARG


def test_block_plan_heads_and_rows(lib):
    from weight_streamed_bf16_gb300.block import BlockShape
    from weight_streamed_bf16_gb300.shard import ShardPlan
    s = BlockShape()                                   # d 4096, 32 heads x 128
    for R in (1, 2, 4, 8):
        plans = [ShardPlan(s, R, r) for r in range(R)]
        rows = sorted(x for p in plans for x in p.qkv_rows)
        assert rows[0][0] == 0 and rows[-1][1] == s.qkv
        assert all(a[1] == b[0] for a, b in zip(rows, rows[1:]))
        for p in plans:
            h0, h1 = p.heads
            q, k, v = p.qkv_rows
            w = s.heads * s.dh
            assert q == (h0 * s.dh, h1 * s.dh)
            assert k == (w + h0 * s.dh, w + h1 * s.dh) and v == (2 * w + h0 * s.dh, 2 * w + h1 * s.dh)
            assert p.att_cols == (h0 * s.dh, h1 * s.dh)
            c0, c1 = p.out_cols
            assert c1 - c0 == s.d // R and c0 % 256 == 0
        # one page of 2048 rows per Q, K and V range when R = 2: the rank's
        # pages are {p : p mod 2 = r} of the six 16 MiB QKV pages
        if R == 2:
            assert [p.qkv_rows for p in plans][1] == [(2048, 4096), (6144, 8192), (10240, 12288)]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import bf16, ops
        from weight_streamed_bf16_gb300 import build as b, psi as p
        from weight_streamed_bf16_gb300.block import BlockShape
        from weight_streamed_bf16_gb300.shard import ShardPlan, gather_columns
        b.build()
        p.load()
        rng = np.random.default_rng(5)             # the same draws on every rank

        def rb(shape, sd=1.0):
            return bf16.round_bf16(rng.standard_normal(shape) * sd)

        s = BlockShape(d=512, N=12, heads=4, dh=128, hidden=512, slice=256)
        plan = ShardPlan(s, world, rank)
        N, d, Hd = s.N, s.d, s.heads * s.dh
        X = rb((N, d))
        att_in = rb((N, Hd))
        Wo, bo = rb((d, Hd), Hd ** -0.5), rb((d,), 0.02)
        U, a = rb((s.hidden, d), d ** -0.5), rb((s.hidden,), 0.02)
        V, bb = rb((d, s.hidden), s.hidden ** -0.5), rb((d,), 0.02)
        Q, K, Vv = rb((s.heads, N, s.dh)), rb((s.heads, N, s.dh)), rb((s.heads, N, s.dh))
        res = {}
        # out-projection: this rank's rows of Wo -> its columns of x1
        c0, c1 = plan.out_cols
        T = torch.full((N, d), float("nan"), dtype=torch.float64)
        T[:, c0:c1] = torch.from_numpy(
            ops.linear(att_in, Wo[c0:c1], bo[c0:c1], residual=X[:, c0:c1]).y)
        gather_columns(T, plan.all("out_cols"), rank)
        res["x1"] = np.array_equal(T.numpy(), ops.linear(att_in, Wo, bo, residual=X).y)
        x1 = T.numpy()
        # FFN: all of U, this rank's rows of V -> its columns of y
        T = torch.full((N, d), float("nan"), dtype=torch.float64)
        T[:, c0:c1] = torch.from_numpy(
            ops.ffn(x1, U, V[c0:c1], a, bb[c0:c1], residual=x1[:, c0:c1]).y)
        gather_columns(T, plan.all("out_cols"), rank)
        res["y"] = np.array_equal(T.numpy(), ops.ffn(x1, U, V, a, bb, residual=x1).y)
        # attention: this rank's heads -> their columns of att
        h0, h1 = plan.heads
        T = torch.full((N, Hd), float("nan"), dtype=torch.float64)
        for h in range(h0, h1):
            T[:, h * s.dh:(h + 1) * s.dh] = torch.from_numpy(
                ops.attention(Q[h], K[h], Vv[h], s.dh ** -0.5).y)
        gather_columns(T, plan.all("att_cols"), rank)
        full = np.concatenate([ops.attention(Q[h], K[h], Vv[h], s.dh ** -0.5).y
                               for h in range(s.heads)], axis=1)
        res["att"] = np.array_equal(T.numpy(), full)
        res["cols"] = (c0, c1, h0, h1)
        out[rank] = res
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_gathered_columns_equal_unsharded(lib):
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0]["cols"] == (0, 256, 0, 2) and out[1]["cols"] == (256, 512, 2, 4)
    for r in range(2):
        assert out[r]["x1"] and out[r]["y"] and out[r]["att"], out[r]


class _OracleRunner:
    """A part of the block computed by the oracle on the host, with the
    interface forward_sharded drives (the GPU runner's phases, with float64
    tensors in place of device buffers and no streams)."""

    def __init__(self, plan, w, ops):
        s = plan.shape
        self.plan, self.s, self.w, self.ops = plan, s, w, ops
        self.h = torch.full((s.N, s.qkv), float("nan"), dtype=torch.float64)
        self.att = torch.full((s.N, s.heads * s.dh), float("nan"), dtype=torch.float64)
        self.x1 = torch.full((s.N, s.d), float("nan"), dtype=torch.float64)

    def gathered(self, Y):
        return {"att": self.att, "x1": self.x1, "y": Y}

    def before_collective(self):
        pass

    def after_collective(self):
        pass

    def run_phase(self, name, X, W, Y, flags=0):
        s, w, ops, p = self.s, self.w, self.ops, self.plan
        Xn = X.numpy()
        if name == "qkv":
            for r0, r1 in p.qkv_rows:
                self.h[:, r0:r1] = torch.from_numpy(
                    ops.linear(Xn, w["Wqkv"][r0:r1], w["bqkv"][r0:r1]).y)
        elif name == "attention":
            h0, h1 = p.heads
            Hd = s.heads * s.dh
            hn = self.h.numpy()
            for hd in range(h0, h1):
                c = slice(hd * s.dh, (hd + 1) * s.dh)
                q = hn[:, hd * s.dh:(hd + 1) * s.dh]
                k = hn[:, Hd + hd * s.dh:Hd + (hd + 1) * s.dh]
                v = hn[:, 2 * Hd + hd * s.dh:2 * Hd + (hd + 1) * s.dh]
                self.att[:, c] = torch.from_numpy(ops.attention(q, k, v, s.dh ** -0.5).y)
        elif name == "out_proj":
            c0, c1 = p.out_cols
            self.x1[:, c0:c1] = torch.from_numpy(
                ops.linear(self.att.numpy(), w["Wo"][c0:c1], w["bo"][c0:c1],
                           residual=Xn[:, c0:c1]).y)
        elif name == "ffn":
            c0, c1 = p.out_cols
            x1 = self.x1.numpy()
            Y[:, c0:c1] = torch.from_numpy(
                ops.ffn(x1, w["W1"], w["W2"][c0:c1], w["a1"], w["b1"][c0:c1],
                        residual=x1[:, c0:c1]).y)


def _block_worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import bf16, ops
        from weight_streamed_bf16_gb300 import build as b, psi as p
        from weight_streamed_bf16_gb300.block import BlockShape
        from weight_streamed_bf16_gb300.shard import ShardPlan, forward_sharded
        b.build()
        p.load()
        rng = np.random.default_rng(9)             # the same draws on every rank

        def rb(shape, sd=1.0):
            return bf16.round_bf16(rng.standard_normal(shape) * sd)

        s = BlockShape(d=512, N=10, heads=4, dh=128, hidden=512, slice=256)
        Hd = s.heads * s.dh
        w = {"Wqkv": rb((s.qkv, s.d), s.d ** -0.5), "bqkv": rb((s.qkv,), 0.02),
             "Wo": rb((s.d, Hd), Hd ** -0.5), "bo": rb((s.d,), 0.02),
             "W1": rb((s.hidden, s.d), s.d ** -0.5), "a1": rb((s.hidden,), 0.02),
             "W2": rb((s.d, s.hidden), s.hidden ** -0.5), "b1": rb((s.d,), 0.02)}
        X = torch.from_numpy(rb((s.N, s.d)))
        runner = _OracleRunner(ShardPlan(s, world, rank), w, ops)
        Y = torch.full((s.N, s.d), float("nan"), dtype=torch.float64)
        forward_sharded(runner, X, None, Y)
        # the unsharded block, one operator after the other
        Xn = X.numpy()
        h = ops.linear(Xn, w["Wqkv"], w["bqkv"]).y
        att = np.concatenate([ops.attention(h[:, i * s.dh:(i + 1) * s.dh],
                                            h[:, Hd + i * s.dh:Hd + (i + 1) * s.dh],
                                            h[:, 2 * Hd + i * s.dh:2 * Hd + (i + 1) * s.dh],
                                            s.dh ** -0.5).y for i in range(s.heads)], axis=1)
        x1 = ops.linear(att, w["Wo"], w["bo"], residual=Xn).y
        y = ops.ffn(x1, w["W1"], w["W2"], w["a1"], w["b1"], residual=x1).y
        out[rank] = (np.array_equal(runner.att.numpy(), att),
                     np.array_equal(runner.x1.numpy(), x1), np.array_equal(Y.numpy(), y))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_sharded_block_forward_equals_unsharded(lib):
    """forward_sharded (the phases and the column gathers between them) over
    two gloo ranks, each part computed by the oracle: the gathered attention
    output, x1 and block output equal the unsharded block bit for bit."""
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_block_worker, args=(2, port, out), nprocs=2, join=True)
    for r in range(2):
        assert out[r] == (True, True, True), (r, out[r])


def test_gather_rejects_unequal_blocks():
    from weight_streamed_bf16_gb300.shard import gather_columns
    with pytest.raises(ValueError):
        gather_columns(torch.zeros(2, 10), [(0, 6), (6, 10)], 0)
