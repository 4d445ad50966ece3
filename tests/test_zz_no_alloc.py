"""The FFN entry point for callers that cannot allocate device memory.

psi_ffn_resident_noalloc keeps its workspaces in a fixed array inside the
library instead of caller buffers, for code that runs inside another
framework's memory pool or a fixed budget and has no allocator to call.  It
must give the same output as psi_ffn_paged with resident weights.  This file
is collected last, so a run that stops at the first failure has run every
other test before it.
"""
import math

import pytest
import torch

from weight_streamed_bf16_gb300 import psi
from weight_streamed_bf16_gb300.torch_io import Arena, FfnWeight, ffn_workspace

from gpu_cases import check, ensure_lib, f64, ops

pytestmark = pytest.mark.gpu


def _case(seed, N=300, d=512, h=2048, r=384):
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(N, d, generator=g).to(torch.bfloat16)
    U = (torch.randn(h, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    V = (torch.randn(r, h, generator=g) / math.sqrt(h)).to(torch.bfloat16)
    a = (torch.randn(h, generator=g) * 0.02).to(torch.bfloat16)
    b = (torch.randn(r, generator=g) * 0.02).to(torch.bfloat16)
    R = torch.randn(N, r, generator=g).to(torch.bfloat16)
    return X, U, V, a, b, R


def _paged(X, w, a, b, R, N, r, slice_):
    """The existing entry point, resident weights, caller workspaces."""
    arena = Arena(w.page_bytes, 2)
    hid, acc = ffn_workspace(N, r, slice_)
    Y = torch.empty(N, r, dtype=torch.bfloat16, device="cuda")
    psi.psi_ffn_paged(arena.handle, X.data_ptr(), N, w.desc(), a.data_ptr(), b.data_ptr(),
                      hid.data_ptr(), acc.data_ptr(), R.data_ptr(), Y.data_ptr(),
                      psi.PSI_RESIDENT)
    arena.sync()
    arena.close()
    return Y


def test_no_alloc_ffn_matches_paged_entry_point():
    ensure_lib()
    N, d, h, r, sl = 300, 512, 2048, 384, 256
    s = torch.cuda.current_stream()
    for seed in (1, 2):            # two calls in a row share the fixed workspace
        X, U, V, a, b, R = _case(seed, N, d, h, r)
        w = FfnWeight(U, V, sl, resident=True)
        Xd, ad, bd, Rd = X.cuda(), a.cuda(), b.cuda(), R.cuda()
        ref = _paged(Xd, w, ad, bd, Rd, N, r, sl)
        Y = torch.full((N, r), float("nan"), dtype=torch.bfloat16, device="cuda")
        psi.psi_ffn_resident_noalloc(Xd.data_ptr(), N, w.desc(), ad.data_ptr(), bd.data_ptr(),
                                     Rd.data_ptr(), Y.data_ptr(), s.cuda_stream, 0)
        psi.psi_stream_wait(s.cuda_stream, 60000)
        # same kernels and slice grouping: the same bytes (within any tolerance)
        assert torch.equal(Y.view(torch.int16), ref.view(torch.int16))
        res = ops.ffn(f64(X), f64(U), f64(V), f64(a), f64(b), residual=f64(R))
        check(Y.cpu(), res, what=f"no-alloc ffn call {seed}")


def test_no_alloc_rejects_oversized_workspace():
    ensure_lib()
    # N*2*slice*2 + N*r*4 = 8192*2048*2 + 8192*2048*4 bytes > 16 MiB
    N, d, h, r, sl = 8192, 64, 2048, 2048, 1024
    w = psi.psi_ffn_weight(None, 256, d, h, r, sl)
    with pytest.raises(psi.PsiError) as e:
        psi.psi_ffn_resident_noalloc(256, N, w, 256, 256, None, 256, 0, 0)
    assert e.value.status == psi.PSI_ERR_CAPACITY and "16777216" in str(e.value)
