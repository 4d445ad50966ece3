"""The indexed host journal (PSI section II-D, asynchronous transport of
section III-B) on the GPU: byte-preserving round trips, producer and
consumer ordering, slot reuse, argument and capacity errors, injected
copy failures, and the journaled multi-branch stack, which must give the
bytes of the same blocks run with every state resident."""
import pytest
import torch

import psi_synth
from weight_streamed_bf16_gb300 import psi
from weight_streamed_bf16_gb300.block import BlockRunner, BlockShape, BlockWeights
from weight_streamed_bf16_gb300.torch_io import Arena, Journal

from gpu_cases import ensure_lib

pytestmark = pytest.mark.gpu
MiB = 1 << 20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


@pytest.fixture
def aj():
    arena = Arena(1 << 20, 2)
    j = Journal(arena, 8 * MiB, 3)
    yield arena, j
    j.close()
    arena.sync()
    arena.close()


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def test_round_trip_is_bitwise(aj):
    arena, j = aj
    g = torch.Generator(device="cuda").manual_seed(1)
    x = torch.randn(1000, 4096, generator=g, device="cuda").to(torch.bfloat16)  # 7.8 MiB
    y = torch.empty_like(x)
    j.commit((0, 0, 0), x)
    j.reload((0, 0, 0), y)
    j.acquire((0, 0, 0))
    arena.sync()
    assert torch.equal(_bits(x), _bits(y))
    assert torch.equal(_bits(j.host_tensor((0, 0, 0), x).cuda()), _bits(x))
    st = j.stats()
    assert st["commits"] == 1 and st["reloads"] == 1 and st["host_waits"] == 1
    assert st["d2h_bytes"] == st["h2d_bytes"] == x.numel() * 2


def test_commit_waits_for_the_producer(aj):
    """The source is written by a long kernel on the compute stream; the
    commit is enqueued right after it, with no host synchronisation."""
    arena, j = aj
    a = torch.randn(4096, 4096, device="cuda")
    pattern = torch.arange(2048 * 1024, dtype=torch.float32, device="cuda").view(2048, 1024)
    src = torch.zeros(2048, 1024, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(arena.compute):
        for _ in range(8):
            a = a @ a.T * (1.0 / 4096)            # keeps the stream busy
        src.copy_(pattern)
        j.commit((1, 0, 0), src)
    arena.sync()
    got = j.host_tensor((1, 0, 0), src)
    assert torch.equal(got, pattern.cpu())


def test_reload_keeps_consumer_dependencies(aj):
    """A kernel on the compute stream still reads dst when the reload is
    enqueued: it sees the old bytes; after acquire the stream sees the new."""
    arena, j = aj
    new = torch.full((2048, 1024), 2.0, device="cuda")
    j.commit((2, 0, 0), new)
    arena.sync()
    dst = torch.full((2048, 1024), 1.0, device="cuda")
    a = torch.randn(4096, 4096, device="cuda")
    with torch.cuda.stream(arena.compute):
        for _ in range(8):
            a = a @ a.T * (1.0 / 4096)
        before = dst.sum()                      # reads the old contents
        j.reload((2, 0, 0), dst)
        j.acquire((2, 0, 0))
        after = dst.sum()
    arena.sync()
    assert before.item() == 2048 * 1024
    assert after.item() == 2 * 2048 * 1024


def test_slot_reuse_waits_for_the_last_reload(aj):
    arena, j = aj
    d1 = torch.full((1024, 1024), 1.0, device="cuda")
    d2 = torch.full((1024, 1024), 2.0, device="cuda")
    b1, b2 = torch.empty_like(d1), torch.empty_like(d1)
    j.commit((3, 0, 0), d1)
    j.reload((3, 0, 0), b1)
    j.commit((3, 0, 0), d2)       # same slot: waits until b1's reload has read it
    j.reload((3, 0, 0), b2)
    j.acquire((3, 0, 0))
    arena.sync()
    assert torch.equal(b1, d1) and torch.equal(b2, d2)


def test_fence_orders_overwrite_after_commit(aj):
    arena, j = aj
    x = torch.full((2048, 1024), 5.0, device="cuda")
    with torch.cuda.stream(arena.compute):
        j.commit((4, 0, 0), x)
        j.fence(x)
        x.fill_(7.0)
    arena.sync()
    assert torch.equal(j.host_tensor((4, 0, 0), x), torch.full((2048, 1024), 5.0))


def test_errors_and_capacity(aj):
    arena, j = aj
    x = torch.zeros(256, dtype=torch.float32, device="cuda")
    with pytest.raises(psi.PsiError) as e:
        j.reload((9, 9, 9), x)
    assert e.value.status == psi.PSI_ERR_INVALID_ARG and "no entry" in str(e.value)
    j.commit((5, 0, 0), x)
    with pytest.raises(psi.PsiError) as e:
        j.acquire((5, 0, 0))            # nothing reloaded
    assert e.value.status == psi.PSI_ERR_INVALID_ARG
    with pytest.raises(psi.PsiError) as e:
        j.reload((5, 0, 0), torch.zeros(128, device="cuda"))   # other size
    assert e.value.status == psi.PSI_ERR_INVALID_ARG
    big = torch.zeros(8 * MiB // 4 + 1, dtype=torch.float32, device="cuda")
    with pytest.raises(psi.PsiError) as e:
        j.commit((6, 0, 0), big)
    assert e.value.status == psi.PSI_ERR_CAPACITY
    j.commit((6, 0, 0), x)
    j.commit((7, 0, 0), x)
    with pytest.raises(psi.PsiError) as e:
        j.commit((8, 0, 0), x)          # three slots, three entries
    assert e.value.status == psi.PSI_ERR_CAPACITY
    j.drop((6, 0, 0))
    j.commit((8, 0, 0), x)
    assert j.stats()["slots_in_use"] == 3


def test_pageable_host_region_is_refused():
    arena = Arena(1 << 20, 2)
    host = torch.empty(1 << 20, dtype=torch.uint8)      # not pinned
    with pytest.raises(psi.PsiError) as e:
        psi.psi_journal_create(arena.handle, host.data_ptr(), 1 << 20, 1 << 16)
    assert e.value.status == psi.PSI_ERR_INVALID_ARG
    arena.close()


def test_injected_copy_failure_enqueues_nothing(aj):
    arena, j = aj
    x = torch.full((256,), 3.0, device="cuda")
    psi.psi_journal_fail_next_copy(j.handle)
    with pytest.raises(psi.PsiError) as e:
        j.commit((10, 0, 0), x)
    assert e.value.status == psi.PSI_ERR_CUDA
    assert j.stats()["commits"] == 0 and j.stats()["slots_in_use"] == 0
    j.commit((10, 0, 0), x)
    psi.psi_journal_fail_next_copy(j.handle)
    with pytest.raises(psi.PsiError):
        j.reload((10, 0, 0), torch.empty_like(x))
    y = torch.empty_like(x)
    j.reload((10, 0, 0), y)
    j.acquire((10, 0, 0))
    arena.sync()
    assert torch.equal(x, y)


# -------------------------------------------- journaled multi-branch stack --
CFG = psi_synth.BLOCK


def _shape():
    return BlockShape(d=CFG.d, N=CFG.N, heads=CFG.heads, dh=CFG.dh, hidden=CFG.hidden,
                      slice=CFG.slice, page_bytes=CFG.page_bytes)


@pytest.mark.parametrize("keep,io", [(True, "journal"), (False, "journal"), (True, "device")])
def test_journaled_branches_equal_resident_states(keep, io):
    """Two blocks over two branch states: the journaled schedule (three
    device state buffers, reloads ahead of compute) gives the bytes of each
    branch's stack run with its states on the device (the transport theorem
    of section III-B: byte-preserving, event-ordered copies)."""
    nb, nbranch = 2, 2
    blocks = []
    for b in range(nb):
        w = {k: v.cpu() for k, v in psi_synth.block_weights(CFG, block=b, device="cuda").items()}
        blocks.append(BlockWeights(w, _shape(), resident=True))
    Xs = [psi_synth.block_input(CFG, device="cuda") * (1.0 - 0.5 * r) for r in range(nbranch)]
    Xs = [x.to(torch.bfloat16) for x in Xs]
    arena = Arena(CFG.page_bytes, 5)
    runner = BlockRunner(_shape(), arena)
    want = []
    for x in Xs:
        Y, tmp = torch.empty_like(x), torch.empty_like(x)
        runner.stack(x, blocks, Y, tmp, 0)
        want.append(Y.clone())
    arena.sync()
    state_bytes = CFG.N * CFG.d * 2
    j = Journal(arena, state_bytes, 2 * nbranch)
    steps = nb * nbranch
    skipped = (nb - 1) if keep else 0
    if io == "journal":
        for r, x in enumerate(Xs):
            j.commit((0, r, 0), x)
        runner.run_branches(blocks, j, nbranch, 0, keep_updated=keep)
        arena.sync()
        for r in range(nbranch):
            got = j.host_tensor((nb, r, 0), Xs[0])
            assert torch.equal(got.view(torch.int16), want[r].cpu().view(torch.int16))
        st = j.stats()
        assert st["reloads"] == steps - skipped
        assert st["commits"] == nbranch + steps - skipped
        assert st["host_waits"] == nbranch           # only the final host views
    else:
        Ys = [torch.empty_like(x) for x in Xs]
        runner.run_branches(blocks, j, nbranch, 0, keep_updated=keep, inputs=Xs, outputs=Ys)
        arena.sync()
        for r in range(nbranch):
            assert torch.equal(Ys[r].view(torch.int16), want[r].view(torch.int16))
        st = j.stats()
        assert st["reloads"] == st["commits"] == steps - skipped - nbranch
        assert st["host_waits"] == 0 and st["slots_in_use"] == 0
    j.close()
    arena.close()
