"""Output-column sharding on one GPU: every part of a partition run in turn
through the C ABI, each writing its columns into the same full-width
output, gives the unpartitioned result bit for bit (the column-partition
invariant of section II-B: each output entry gets its complete dot product
from one part).  The multi-device gathers are covered on CPU
(tests/test_shard_multirank.py)."""
import math

import pytest
import torch

import psi_synth
from weight_streamed_bf16_gb300 import psi
from weight_streamed_bf16_gb300.block import BlockRunner, BlockShape, BlockWeights
from weight_streamed_bf16_gb300.shard import (ShardBuffers, ShardPlan, ShardRunner,
                                              ShardWeights, forward_parts_in_turn)
from weight_streamed_bf16_gb300.torch_io import Arena, FfnWeight, LinearWeight, ffn_workspace

from gpu_cases import check, ensure_lib, f64, ops

pytestmark = pytest.mark.gpu
MiB = 1 << 20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _bits(t):
    return t.contiguous().view(torch.int16)


@pytest.mark.parametrize("parts", [2, 3])
@pytest.mark.parametrize("flags", [0, psi.PSI_RESIDENT])
def test_linear_column_parts_bitwise(parts, flags):
    g = torch.Generator().manual_seed(parts)
    N, K, M = 300, 512, 768
    X = torch.randn(N, K, generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn(M, K, generator=g) / math.sqrt(K)).to(torch.bfloat16)
    b = (torch.randn(M, generator=g) * 0.02).to(torch.bfloat16).cuda()
    R = torch.randn(N, M, generator=g).to(torch.bfloat16).cuda()
    pb = 128 * K * 2
    arena = Arena(pb, 2)
    res = bool(flags & psi.PSI_RESIDENT)
    full = LinearWeight(W, pb, page_rows=128, resident=res)
    ref = torch.empty(N, M, dtype=torch.bfloat16, device="cuda")
    psi.psi_linear_paged(arena.handle, X.data_ptr(), N, K, full.desc(), b.data_ptr(),
                         R.data_ptr(), ref.data_ptr(), M, flags)
    Y = torch.full((N, M), float("nan"), dtype=torch.bfloat16, device="cuda")
    for r in range(parts):
        c0, c1 = psi.psi_plan_columns(M, 256, parts, r)
        w = LinearWeight(W[c0:c1], pb, page_rows=128, resident=res)
        psi.psi_linear_paged(arena.handle, X.data_ptr(), N, K, w.desc(), b.data_ptr() + 2 * c0,
                             R.data_ptr() + 2 * c0, Y.data_ptr() + 2 * c0, M, flags)
    arena.sync()
    arena.close()
    assert torch.equal(_bits(Y), _bits(ref))


@pytest.mark.parametrize("parts", [2, 3])
@pytest.mark.parametrize("flags", [0, psi.PSI_RESIDENT,
                                   psi.PSI_RESIDENT | psi.PSI_BOUNDARY_PREGELU_BF16])
def test_ffn_output_column_parts_bitwise(parts, flags):
    """All of U and the part's rows of V per part (its own page image): the
    gathered output columns equal the unpartitioned FFN."""
    g = torch.Generator().manual_seed(10 + parts)
    N, d, h, r, sl = 300, 512, 2048, 768, 256
    X = torch.randn(N, d, generator=g).to(torch.bfloat16)
    U = (torch.randn(h, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    V = (torch.randn(r, h, generator=g) / math.sqrt(h)).to(torch.bfloat16)
    a = (torch.randn(h, generator=g) * 0.02).to(torch.bfloat16).cuda()
    b = (torch.randn(r, generator=g) * 0.02).to(torch.bfloat16).cuda()
    Res = torch.randn(N, r, generator=g).to(torch.bfloat16).cuda()
    Xd = X.cuda()
    res = bool(flags & psi.PSI_RESIDENT)
    wf = FfnWeight(U, V, sl, resident=res)
    arena = Arena(wf.page_bytes, 2)
    hid, acc = ffn_workspace(N, r, sl)
    ref = torch.empty(N, r, dtype=torch.bfloat16, device="cuda")
    psi.psi_ffn_paged(arena.handle, Xd.data_ptr(), N, wf.desc(), a.data_ptr(), b.data_ptr(),
                      hid.data_ptr(), acc.data_ptr(), Res.data_ptr(), ref.data_ptr(), flags)
    Y = torch.full((N, r), float("nan"), dtype=torch.bfloat16, device="cuda")
    for q in range(parts):
        c0, c1 = psi.psi_plan_columns(r, 256, parts, q)
        w = FfnWeight(U, V[c0:c1], sl, resident=res)
        psi.psi_ffn_paged_strided(arena.handle, Xd.data_ptr(), N, w.desc(), a.data_ptr(),
                                  b.data_ptr() + 2 * c0, hid.data_ptr(), acc.data_ptr(),
                                  Res.data_ptr() + 2 * c0, Y.data_ptr() + 2 * c0, r, flags)
    arena.sync()
    arena.close()
    assert torch.equal(_bits(Y), _bits(ref))
    # and the partitioned result is the FFN of the oracle on sampled rows
    rows = slice(0, 64)
    check(Y[rows].cpu(), ops.ffn(f64(X[rows]), f64(U), f64(V), f64(a.cpu()), f64(b.cpu()),
                                 residual=f64(Res[rows].cpu()),
                                 pregelu_bf16=bool(flags & psi.PSI_BOUNDARY_PREGELU_BF16)),
          what=f"ffn in {parts} column parts")


def test_ffn_strided_rejects_short_ldy():
    w = psi.psi_ffn_weight(None, 256, 64, 64, 64, 64)
    with pytest.raises(psi.PsiError) as e:
        psi.psi_ffn_paged_strided(256, 256, 8, w, 256, 256, 256, 256, None, 256, 32,
                                  psi.PSI_RESIDENT)
    assert e.value.status == psi.PSI_ERR_INVALID_ARG


CFG = psi_synth.BLOCK


def _block_case(prenorm):
    shape = BlockShape(d=CFG.d, N=CFG.N, heads=CFG.heads, dh=CFG.dh, hidden=CFG.hidden,
                       slice=CFG.slice, page_bytes=CFG.page_bytes, prenorm=prenorm, eps=CFG.eps)
    w = psi_synth.block_weights(CFG, block=0, device="cuda")
    if prenorm:
        w["gamma1"], w["gamma2"] = psi_synth.norm_gains(CFG, block=0, device="cuda")
    w = {k: v.cpu() for k, v in w.items()}
    rope = psi_synth.rope_table(CFG.N, CFG.dh) if prenorm else None
    X = psi_synth.block_input(CFG, device="cuda")
    return shape, w, rope, X


@pytest.mark.parametrize("parts,prenorm", [(2, False), (4, False), (2, True)])
def test_block_column_parts_bitwise(parts, prenorm):
    """The full synthetic block (d 4096, 6144 tokens) in 2 or 4 output-column
    parts, weights streamed through one 80 MiB arena part after part, against
    the unpartitioned block with resident weights; attention computes every
    unit whole in both."""
    shape, w, rope, X = _block_case(prenorm)
    arena = Arena(CFG.page_bytes, 5)
    ref_runner = BlockRunner(shape, arena, rope=rope, attn_tail_split=False)
    bw = BlockWeights(w, shape, resident=True)
    ref = torch.empty_like(X)
    ref_runner.forward(X, bw, ref, psi.PSI_RESIDENT)
    arena.sync()
    del bw
    bufs = ShardBuffers(shape)
    plans = [ShardPlan(shape, parts, r) for r in range(parts)]
    runners = [ShardRunner(p, arena, bufs, rope=rope) for p in plans]
    weights = [ShardWeights(w, p) for p in plans]
    Y = torch.full_like(X, float("nan"))
    forward_parts_in_turn(runners, X, weights, Y, 0)
    arena.sync()
    st = arena.stats()
    arena.close()
    assert torch.equal(_bits(Y), _bits(ref))
    assert torch.equal(_bits(bufs.att), _bits(ref_runner.att))
    # per part, a third fewer host bytes than the whole block when R = 2
    per_part = weights[0].host_bytes
    assert per_part == sum(x.host_bytes for x in weights) // parts
    if parts == 2:
        assert per_part == 256 * MiB
    # each part streamed its own pages: its Q, K, V and out-projection row
    # ranges page by page, and every hidden slice once
    want = sum(sum(-(-lw.rows // lw.page_rows) for lw in x.qkv + [x.out]) +
               shape.hidden // shape.slice for x in weights)
    assert st["pages_streamed"] == want


def test_block_one_part_is_the_block():
    """A one-part plan runs the same calls' arithmetic as the unsharded
    block (tail split off in both)."""
    shape, w, rope, X = _block_case(False)
    arena = Arena(CFG.page_bytes, 5)
    ref_runner = BlockRunner(shape, arena, attn_tail_split=False)
    ref = torch.empty_like(X)
    # the pinned host weights must outlive the asynchronous page copies
    bw = BlockWeights(w, shape)
    ref_runner.forward(X, bw, ref, 0)
    bufs = ShardBuffers(shape)
    p = ShardPlan(shape, 1, 0)
    sw = ShardWeights(w, p)
    Y = torch.full_like(X, float("nan"))
    forward_parts_in_turn([ShardRunner(p, arena, bufs)], X, [sw], Y, 0)
    arena.sync()
    arena.close()
    del bw, sw
    assert torch.equal(_bits(Y), _bits(ref))


def test_forward_sharded_one_rank_nccl():
    """forward_sharded on a one-rank NCCL group (its phases on the arena's
    stream, the column gathers as NCCL all-gathers on torch's stream)
    equals the unsharded block with the attention tail split off."""
    import os
    import socket

    import torch.distributed as dist
    from weight_streamed_bf16_gb300.shard import forward_sharded
    shape, w, rope, X = _block_case(False)
    arena = Arena(CFG.page_bytes, 5)
    ref_runner = BlockRunner(shape, arena, attn_tail_split=False)
    bw = BlockWeights(w, shape)
    ref = torch.empty_like(X)
    ref_runner.forward(X, bw, ref, 0)
    arena.sync()
    sk = socket.socket()
    sk.bind(("127.0.0.1", 0))
    port = sk.getsockname()[1]
    sk.close()
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        p = ShardPlan(shape, 1, 0)
        sw = ShardWeights(w, p)
        runner = ShardRunner(p, arena, ShardBuffers(shape))
        Y = torch.full_like(X, float("nan"))
        forward_sharded(runner, X, sw, Y, 0)
        torch.cuda.synchronize()
        arena.sync()
    finally:
        dist.destroy_process_group()
        arena.close()
    del bw, sw
    assert torch.equal(_bits(Y), _bits(ref))
