"""Arena rules and failure detection on the GPU, with no fault and no hang.

PSI section II-A: each page has at most one unreleased request; reuse
follows the copy and consumer dependencies.  Section II-D: page lifecycle.
Table V of the capacity study: a weight tile larger than the page fails.
Failures are made on the host (an injected copy error, a second request on
an unreleased page) or by a bounded in-kernel wait that is left to expire.
"""
import math

import pytest
import torch

from weight_streamed_bf16_gb300 import psi
from weight_streamed_bf16_gb300.torch_io import Arena, LinearWeight

from gpu_cases import check, ensure_lib, f64, ops, run_linear

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _small():
    g = torch.Generator().manual_seed(3)
    X = torch.randn(64, 128, generator=g).to(torch.bfloat16)
    W = (torch.randn(64, 128, generator=g) / 12).to(torch.bfloat16)
    b = (torch.randn(64, generator=g) * 0.02).to(torch.bfloat16)
    return X, W, b


def test_page_busy_until_released():
    a = Arena(1 << 16, 2)
    src = torch.zeros(1 << 15, dtype=torch.uint8, pin_memory=True)
    p0 = psi.psi_page_stream(a.handle, src.data_ptr(), src.numel())
    p1 = psi.psi_page_stream(a.handle, src.data_ptr(), src.numel())
    assert (p0.slot, p1.slot) == (0, 1)
    with pytest.raises(psi.PsiError) as e:    # slot 0 again, still requested
        psi.psi_page_stream(a.handle, src.data_ptr(), src.numel())
    assert e.value.status == psi.PSI_ERR_PAGE_BUSY
    psi.psi_page_release(a.handle, p0)
    with pytest.raises(psi.PsiError) as e:    # double release
        psi.psi_page_release(a.handle, p0)
    assert e.value.status == psi.PSI_ERR_INVALID_ARG
    p2 = psi.psi_page_stream(a.handle, src.data_ptr(), src.numel())
    assert p2.slot == 0 and p2.seq > p1.seq
    psi.psi_page_release(a.handle, p1)
    psi.psi_page_release(a.handle, p2)
    a.sync()
    st = a.stats()
    assert st["pages_streamed"] == 3 and st["h2d_bytes"] == 3 * src.numel()
    a.close()


def test_page_bytes_round_trip():
    """Byte-preserving transport: what lands in the slot is the host slice."""
    a = Arena(1 << 16, 3)
    src = torch.randint(0, 255, (5, 1 << 16), dtype=torch.uint8).pin_memory()
    for i in range(5):
        p = psi.psi_page_stream(a.handle, src[i].data_ptr(), 1 << 16)
        a.sync()
        slot = a.buf[p.dev - a.buf.data_ptr():p.dev - a.buf.data_ptr() + (1 << 16)]
        assert torch.equal(slot.cpu(), src[i])
        psi.psi_page_release(a.handle, p)
    a.close()


def test_capacity_and_argument_errors():
    X, W, b = _small()
    a = Arena(1 << 14, 2)   # 16 KiB pages: 64 rows x 128 x 2 B = 16 KiB fits; 80 does not
    w = LinearWeight(torch.cat([W, W[:16]]), 1 << 14, page_rows=80)
    Xd, bd = X.cuda(), torch.cat([b, b[:16]]).cuda()
    Y = torch.empty(64, 80, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(psi.PsiError) as e:
        psi.psi_linear_paged(a.handle, Xd.data_ptr(), 64, 128, w.desc(), bd.data_ptr(), None,
                             Y.data_ptr(), 80, 0)
    assert e.value.status == psi.PSI_ERR_CAPACITY
    with pytest.raises(psi.PsiError) as e:     # misaligned output pointer
        psi.psi_linear_paged(a.handle, Xd.data_ptr(), 64, 128, w.desc(), bd.data_ptr(), None,
                             Y.data_ptr() + 2, 80, 0)
    assert e.value.status == psi.PSI_ERR_INVALID_ARG
    with pytest.raises(psi.PsiError) as e:     # K mismatch
        psi.psi_linear_paged(a.handle, Xd.data_ptr(), 64, 136, w.desc(), bd.data_ptr(), None,
                             Y.data_ptr(), 80, 0)
    assert e.value.status == psi.PSI_ERR_INVALID_ARG
    a.sync()
    a.close()


def test_injected_copy_failure_leaves_arena_usable():
    X, W, b = _small()
    a = Arena(64 * 128 * 2, 2)
    psi.psi_arena_fail_next_copy(a.handle)
    with pytest.raises(psi.PsiError) as e:
        run_linear(X, W, b, 64, 2, arena=a)
    assert e.value.status == psi.PSI_ERR_CUDA and "injected" in str(e.value)
    y = run_linear(X, W, b, 64, 2, arena=a)
    check(y, ops.linear(f64(X), f64(W), f64(b)))
    a.close()


def test_bounded_kernel_wait_expires_and_reports():
    """A page GEMM whose producer issues no copies: its consumers' waits
    expire after 2 ms, the kernel records the error and returns; psi_sync
    reports PSI_ERR_DEVICE and the next call runs normally."""
    X, W, b = _small()
    a = Arena(64 * 128 * 2, 2)
    psi.psi_debug_stall_next_gemm(2_000_000)
    Xd, bd = X.cuda(), b.cuda()
    Y = torch.empty(64, 64, dtype=torch.bfloat16, device="cuda")
    w = LinearWeight(W, 64 * 128 * 2, page_rows=64)
    psi.psi_linear_paged(a.handle, Xd.data_ptr(), 64, 128, w.desc(), bd.data_ptr(), None,
                         Y.data_ptr(), 64, 0)
    with pytest.raises(psi.PsiError) as e:
        a.sync(60000)
    assert e.value.status == psi.PSI_ERR_DEVICE and "bounded wait" in str(e.value)
    a.sync()   # the error record was cleared by the report
    y = run_linear(X, W, b, 64, 2, arena=a)
    check(y, ops.linear(f64(X), f64(W), f64(b)))
    a.close()


def test_sync_timeout_is_reported():
    """psi_sync with a zero deadline while a copy is in flight: PSI_ERR_TIMEOUT
    or (if the copy already finished) OK; never a hang."""
    a = Arena(64 << 20, 2)
    src = torch.empty(64 << 20, dtype=torch.uint8, pin_memory=True)
    p = psi.psi_page_stream(a.handle, src.data_ptr(), src.numel())
    try:
        psi.psi_sync(a.handle, 0)
    except psi.PsiError as e:
        assert e.status == psi.PSI_ERR_TIMEOUT
    psi.psi_page_release(a.handle, p)
    a.sync()
    a.close()


def test_no_device_allocation_by_the_library():
    """Rule (i) of section II-A: the library's calls allocate no device memory
    (torch's allocator is the only one; its reserved bytes do not move and the
    device's free memory is unchanged across the calls)."""
    X, W, b = _small()
    a = Arena(64 * 128 * 2, 2)
    Xd, bd = X.cuda(), b.cuda()
    Y = torch.empty(64, 64, dtype=torch.bfloat16, device="cuda")
    w = LinearWeight(W, 64 * 128 * 2, page_rows=64)
    psi.psi_linear_paged(a.handle, Xd.data_ptr(), 64, 128, w.desc(), bd.data_ptr(), None,
                         Y.data_ptr(), 64, 0)
    a.sync()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        psi.psi_linear_paged(a.handle, Xd.data_ptr(), 64, 128, w.desc(), bd.data_ptr(), None,
                             Y.data_ptr(), 64, 0)
    a.sync()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    a.close()


def test_page_timeline_follows_the_lifecycle():
    """Section II-D on the device clock: every page GEMM starts after the copy
    into its slot ended, and a slot's next copy starts after the GEMM that
    read the previous page ended (event timestamps of the page trace)."""
    g = torch.Generator().manual_seed(11)
    N, K, M, pr = 512, 512, 7 * 256, 256
    X = torch.randn(N, K, generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn(M, K, generator=g) / 24).to(torch.bfloat16)
    b = (torch.randn(M, generator=g) * 0.02).to(torch.bfloat16).cuda()
    a = Arena(pr * K * 2, 2)
    w = LinearWeight(W, pr * K * 2, page_rows=pr)
    Y = torch.empty(N, M, dtype=torch.bfloat16, device="cuda")
    psi.psi_arena_trace_begin(a.handle, 64)
    for _ in range(2):
        psi.psi_linear_paged(a.handle, X.data_ptr(), N, K, w.desc(), b.data_ptr(), None,
                             Y.data_ptr(), M, 0)
    a.sync()
    rec = psi.psi_arena_trace_get(a.handle)
    copies = [r for r in rec if r["kind"] == "copy"]
    gemms = [r for r in rec if r["kind"] == "gemm"]
    assert len(copies) == 14 and len(gemms) == 14
    assert all(r["end_ms"] >= r["start_ms"] >= 0 for r in rec)
    assert all(r["stream"] == 2 and r["work"] == pr * K * 2 for r in copies)
    assert all(r["slot"] in (0, 1) and r["work"] == 2.0 * N * pr * K for r in gemms)
    eps = 2e-3  # event timer resolution, ms
    by_seq = sorted(copies, key=lambda r: r["seq"])
    by_launch = sorted(gemms, key=lambda r: r["seq"])
    for i, (c, gm) in enumerate(zip(by_seq, by_launch)):
        assert gm["slot"] == c["slot"] == i % 2
        assert gm["start_ms"] >= c["end_ms"] - eps          # ready before consumed
        if i >= 2:
            assert c["start_ms"] >= by_launch[i - 2]["end_ms"] - eps  # slot released first
    st = a.stats()
    assert st["timed_copies"] == 14 and st["timed_gemms"] == 14
    a.close()
