"""The C-ABI library builds, loads and exports every declared entry point;
host-only entry points (plans, packing, argument checks) work without a GPU.
"""
import ctypes as C
import os
import re

import pytest
import torch

from weight_streamed_bf16_gb300 import build, psi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return psi.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "psi.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(psi_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(names) == sorted(psi.EXPORTS)


def test_version_and_status_strings(lib):
    assert "sm_103a" in psi.psi_version()
    assert psi.psi_status_string(psi.PSI_ERR_PAGE_BUSY) == "PSI_ERR_PAGE_BUSY"
    assert psi.psi_status_string(99) == "PSI_ERR_UNKNOWN"


def test_plan_linear(lib):
    # 64-row pages of a [512 x 512] weight in 64 KiB pages
    assert psi.psi_plan_linear(512, 512, 64 * 1024) == 64
    # 16 MiB pages of [12288 x 4096]: 2048 rows (a multiple of 256)
    assert psi.psi_plan_linear(12288, 4096, 16 << 20) == 2048
    # a weight that fits one page is one page
    assert psi.psi_plan_linear(100, 64, 1 << 20) == 100
    # the plan depends on the page only
    assert psi.psi_plan_linear(4096, 4096, 16 << 20) == 2048
    with pytest.raises(psi.PsiError) as e:
        psi.psi_plan_linear(4096, 4096, 8 * 4096 * 2)  # 8 rows < 16
    assert e.value.status == psi.PSI_ERR_CAPACITY


def test_ffn_page_bytes_and_workspace(lib):
    assert psi.psi_ffn_page_bytes(2048, 2048, 1024) == 8 << 20
    assert psi.psi_ffn_page_bytes(4096, 4096, 1024) == 16 << 20
    hb, ab = psi.psi_ffn_workspace(1024, 2048, 1024)
    assert hb == 2 * 2 * 1024 * 1024 * 2 and ab == 1024 * 2048 * 4


def test_ffn_pack_layout(lib):
    d, h, r, sl = 24, 64, 40, 16
    U = torch.arange(h * d, dtype=torch.int32).to(torch.int16).view(h, d)
    V = (torch.arange(r * h, dtype=torch.int32) * 7).to(torch.int16).view(r, h)
    pb = psi.psi_ffn_page_bytes(d, r, sl)
    dst = torch.zeros((h // sl) * pb // 2, dtype=torch.int16)
    psi.psi_ffn_pack(U.data_ptr(), V.data_ptr(), d, h, r, sl, dst.data_ptr())
    for J in range(h // sl):
        page = dst[J * pb // 2:(J + 1) * pb // 2]
        assert torch.equal(page[:sl * d].view(sl, d), U[J * sl:(J + 1) * sl])
        assert torch.equal(page[sl * d:].view(r, sl), V[:, J * sl:(J + 1) * sl])


def test_ffn_pack_rejects_ragged_hidden(lib):
    with pytest.raises(psi.PsiError) as e:
        psi.psi_ffn_pack(1, 1, 8, 100, 8, 64, 1)
    assert e.value.status == psi.PSI_ERR_INVALID_ARG


def test_arena_create_argument_checks(lib):
    with pytest.raises(psi.PsiError) as e:
        psi.psi_arena_create(0, 1 << 20, 1 << 16, 0, 0)
    assert e.value.status == psi.PSI_ERR_INVALID_ARG
    with pytest.raises(psi.PsiError) as e:
        psi.psi_arena_create(1024, 1 << 20, 1000, 0, 0)  # page not a multiple of 1024
    assert e.value.status == psi.PSI_ERR_INVALID_ARG
    with pytest.raises(psi.PsiError) as e:
        psi.psi_arena_create(1024, 1 << 10, 1 << 16, 0, 0)  # smaller than one page
    assert e.value.status == psi.PSI_ERR_CAPACITY
    assert "aligned" in psi.psi_last_error() or "page" in psi.psi_last_error()


def test_operator_argument_checks_need_no_gpu(lib):
    W = psi.psi_linear_weight(None, None, 64, 64, 64)
    r = lib.psi_linear_paged(None, None, 1, 64, C.byref(W), None, None, None, 64, 0)
    assert r == psi.PSI_ERR_INVALID_ARG
    q = psi.psi_heads(None, 128, 0)
    r = lib.psi_attn_partitioned(C.byref(q), C.byref(q), C.byref(q), C.byref(q), 1, 1, 0,
                                 128, 0.1, 128, None, 0)
    assert r == psi.PSI_ERR_INVALID_ARG


def test_header_documents_no_device_allocation():
    text = open(os.path.join(ROOT, "include", "psi.h")).read()
    assert "never" in text and "allocat" in text
    src = os.path.join(ROOT, "weight_streamed_bf16_gb300", "csrc")
    for f in os.listdir(src):
        body = open(os.path.join(src, f)).read()
        assert not re.search(r"\b(cudaMalloc\w*|cudaFree\w*|cuMemAlloc\w*)\s*\(", body), f


def test_rmsnorm_argument_checks_need_no_gpu(lib):
    """Shape, alignment and overlap checks of psi_rmsnorm return before any
    CUDA call (fake 16-byte aligned addresses; nothing is dereferenced)."""
    X, g, Y = 1 << 20, 1 << 21, 1 << 22
    bad = [
        (None, 64, 4, 64, g, 1e-6, Y, 64, psi.PSI_ERR_INVALID_ARG),   # null X
        (X, 64, 4, 60, g, 1e-6, Y, 64, psi.PSI_ERR_INVALID_ARG),      # d % 8
        (X, 32, 4, 64, g, 1e-6, Y, 64, psi.PSI_ERR_INVALID_ARG),      # ldx < d
        (X, 16384, 4, 16384, g, 1e-6, Y, 16384, psi.PSI_ERR_UNSUPPORTED),  # d > 8192
        (X, 64, 4, 64, g, -1.0, Y, 64, psi.PSI_ERR_INVALID_ARG),      # eps < 0
        (X, 64, 4, 64, g, float("nan"), Y, 64, psi.PSI_ERR_INVALID_ARG),
        (X + 2, 64, 4, 64, g, 1e-6, Y, 64, psi.PSI_ERR_INVALID_ARG),  # misaligned
        (X, 64, 4, 64, g, 1e-6, X + 64, 64, psi.PSI_ERR_INVALID_ARG),  # Y overlaps X
    ]
    for *args, want in bad:
        assert lib.psi_rmsnorm(*args, None) == want, args
    assert lib.psi_rmsnorm(X, 64, 0, 64, g, 1e-6, Y, 64, None) == psi.PSI_OK  # no rows


def test_linear_rope_argument_checks_need_no_gpu(lib):
    W = psi.psi_linear_weight(None, None, 64, 64, 64)
    rope = psi.psi_rope(1 << 20, 1 << 21, 64, 64, 128, 0)
    r = lib.psi_linear_rope_paged(None, None, 1, 64, C.byref(W), None, C.byref(rope), None,
                                  64, 0)
    assert r == psi.PSI_ERR_INVALID_ARG
    r = lib.psi_linear_rope_paged(1, 1, 1, 64, C.byref(W), 1, None, 1, 64, 0)
    assert r == psi.PSI_ERR_INVALID_ARG and "rope" in psi.psi_last_error()


def test_trace_argument_checks_need_no_gpu(lib):
    n = C.c_size_t(7)
    assert lib.psi_arena_trace_begin(None, 16) == psi.PSI_ERR_INVALID_ARG
    assert lib.psi_arena_trace_get(None, None, 0, C.byref(n)) == psi.PSI_ERR_INVALID_ARG
    assert n.value == 7
    assert C.sizeof(psi.psi_trace_record) == 48
    text = open(os.path.join(ROOT, "include", "psi.h")).read()
    assert "PSI_TRACE_COPY = 0, PSI_TRACE_GEMM = 1" in text


def test_unknown_and_unhonoured_flags_are_refused_without_a_gpu(lib):
    """Every operator entry point refuses a flag bit it does not honour with
    PSI_ERR_UNSUPPORTED, before it looks at any other argument or makes any
    CUDA call (null pointers everywhere: nothing is dereferenced)."""
    UNS = psi.PSI_ERR_UNSUPPORTED
    unknown = 0x1000
    W = psi.psi_linear_weight(None, None, 64, 64, 64)
    FW = psi.psi_ffn_weight(None, None, 64, 128, 64, 64)
    rope = psi.psi_rope(1 << 20, 1 << 21, 64, 64, 128, 0)
    q = psi.psi_heads(None, 128, 0)
    pg = psi.psi_page()

    def linear(f):
        return lib.psi_linear_paged(None, None, 1, 64, C.byref(W), None, None, None, 64, f)

    def linear_rope(f):
        return lib.psi_linear_rope_paged(None, None, 1, 64, C.byref(W), None, C.byref(rope),
                                         None, 64, f)

    def ffn(f):
        return lib.psi_ffn_paged(None, None, 1, C.byref(FW), None, None, None, None, None,
                                 None, f)

    def attn(f):
        return lib.psi_attn_partitioned(C.byref(q), C.byref(q), C.byref(q), C.byref(q), 1, 1,
                                        1, 128, 0.1, 128, None, f)

    def attn_ws(f):
        return lib.psi_attn_partitioned_ws(C.byref(q), C.byref(q), C.byref(q), C.byref(q), 1,
                                           1, 1, 128, 0.1, 128, None, 0, None, f)

    def noalloc(f):
        return lib.psi_ffn_resident_noalloc(None, 1, C.byref(FW), None, None, None, None, None,
                                            f)

    def page_stream(f):
        return lib.psi_page_stream(None, None, 0, f, C.byref(pg))

    honoured = {
        linear: psi.PSI_RESIDENT | psi.PSI_SYNC_COPY | psi.PSI_BIAS_AFTER_BF16,
        linear_rope: (psi.PSI_RESIDENT | psi.PSI_SYNC_COPY | psi.PSI_BIAS_AFTER_BF16
                      | psi.PSI_ROPE_AFTER_BF16),
        ffn: (psi.PSI_RESIDENT | psi.PSI_SYNC_COPY | psi.PSI_BOUNDARY_PREGELU_BF16
              | psi.PSI_BIAS_AFTER_BF16),
        attn: psi.PSI_ATTN_BF16_WEIGHTS,
        attn_ws: psi.PSI_ATTN_BF16_WEIGHTS,
        noalloc: psi.PSI_RESIDENT | psi.PSI_BOUNDARY_PREGELU_BF16 | psi.PSI_BIAS_AFTER_BF16,
        page_stream: psi.PSI_SYNC_COPY,
    }
    every = (psi.PSI_RESIDENT | psi.PSI_SYNC_COPY | psi.PSI_BOUNDARY_PREGELU_BF16
             | psi.PSI_BIAS_AFTER_BF16 | psi.PSI_ATTN_BF16_WEIGHTS | psi.PSI_ROPE_AFTER_BF16)
    for call, ok in honoured.items():
        name = call.__name__
        assert call(unknown) == UNS, name
        assert "0x1000" in psi.psi_last_error(), name
        for bit in range(6):
            f = 1 << bit
            r = call(f)
            if f & ok:
                assert r != UNS, (name, hex(f))   # refused later, for the null pointers
            else:
                assert r == UNS, (name, hex(f))
        assert call(ok) != UNS, name
        assert every & ~ok and call(every) == UNS, name
