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

SCRATCH = 16 << 20   # the fixed array's size, in bytes


def _case(seed, N, d, h, r):
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(N, d, generator=g).to(torch.bfloat16)
    U = (torch.randn(h, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    V = (torch.randn(r, h, generator=g) / math.sqrt(h)).to(torch.bfloat16)
    a = (torch.randn(h, generator=g) * 0.02).to(torch.bfloat16)
    b = (torch.randn(r, generator=g) * 0.02).to(torch.bfloat16)
    R = torch.randn(N, r, generator=g).to(torch.bfloat16)
    return X, U, V, a, b, R


def _paged(X, w, a, b, R, N, r, slice_, flags):
    """The existing entry point, resident weights, caller workspaces."""
    arena = Arena(w.page_bytes, 2)
    hid, acc = ffn_workspace(N, r, slice_)
    Y = torch.empty(N, r, dtype=torch.bfloat16, device="cuda")
    psi.psi_ffn_paged(arena.handle, X.data_ptr(), N, w.desc(), a.data_ptr(), b.data_ptr(),
                      hid.data_ptr(), acc.data_ptr(), None if R is None else R.data_ptr(),
                      Y.data_ptr(), psi.PSI_RESIDENT | flags)
    arena.sync()
    arena.close()
    return Y


def _workspace_bytes(N, h, r, sl):
    S = h // sl
    G = 2 if (S >= 2 and sl % 64 == 0) else 1
    return (N * G * sl * 2 + 255) // 256 * 256 + N * r * 4


# (N, d, h, r, slice, residual, flags): every epilogue path of the call
CASES = [
    # two slices per down pass, all groups full
    (300, 512, 2048, 384, 256, True, 0),
    # odd slice count: the last group has one slice (no K split)
    (200, 256, 768, 256, 256, False, 0),
    # one slice: a single down projection that writes Y directly
    (130, 256, 256, 128, 256, True, 0),
    # slice not a multiple of 64: one slice per down pass
    (96, 128, 240, 64, 48, False, 0),
    # the paper's extra pre-GELU write, and the baseline rounding order
    (257, 256, 1024, 192, 256, True, psi.PSI_BOUNDARY_PREGELU_BF16),
    (257, 256, 1024, 192, 256, False, psi.PSI_BIAS_AFTER_BF16),
    # a workspace that fills the fixed array exactly
    (2048, 256, 512, 1792, 256, True, 0),
]


@pytest.mark.parametrize("N,d,h,r,sl,with_res,flags", CASES)
def test_no_alloc_ffn_matches_paged_entry_point(N, d, h, r, sl, with_res, flags):
    ensure_lib()
    assert _workspace_bytes(N, h, r, sl) <= SCRATCH
    s = torch.cuda.current_stream()
    for seed in (1, 2):            # two calls in a row share the fixed workspace
        X, U, V, a, b, R = _case(seed + N, N, d, h, r)
        if not with_res:
            R = None
        w = FfnWeight(U, V, sl, resident=True)
        Xd, ad, bd = X.cuda(), a.cuda(), b.cuda()
        Rd = None if R is None else R.cuda()
        ref = _paged(Xd, w, ad, bd, Rd, N, r, sl, flags)
        Y = torch.full((N, r), float("nan"), dtype=torch.bfloat16, device="cuda")
        psi.psi_ffn_resident_noalloc(Xd.data_ptr(), N, w.desc(), ad.data_ptr(), bd.data_ptr(),
                                     None if Rd is None else Rd.data_ptr(), Y.data_ptr(),
                                     s.cuda_stream, flags)
        psi.psi_stream_wait(s.cuda_stream, 60000)
        # same grouping, accumulation order and epilogue arithmetic: the same
        # bytes (within any tolerance)
        assert torch.equal(Y.view(torch.int16), ref.view(torch.int16))
        rows = slice(0, min(N, 96))   # the oracle on a leading block of rows
        res = ops.ffn(f64(X[rows]), f64(U), f64(V), f64(a), f64(b),
                      residual=None if R is None else f64(R[rows]),
                      pregelu_bf16=bool(flags & psi.PSI_BOUNDARY_PREGELU_BF16),
                      bias_after_bf16=bool(flags & psi.PSI_BIAS_AFTER_BF16))
        check(Y[rows].cpu(), res, what=f"no-alloc ffn {N}x{d}->{h}->{r} call {seed}")


def test_no_alloc_rejects_oversized_workspace():
    ensure_lib()
    # N*2*slice*2 + N*r*4 = 8192*2048*2 + 8192*2048*4 bytes > 16 MiB
    N, d, h, r, sl = 8192, 64, 2048, 2048, 1024
    w = psi.psi_ffn_weight(None, 256, d, h, r, sl)
    with pytest.raises(psi.PsiError) as e:
        psi.psi_ffn_resident_noalloc(256, N, w, 256, 256, None, 256, 0, 0)
    assert e.value.status == psi.PSI_ERR_CAPACITY and str(SCRATCH) in str(e.value)
    # one row more than the exact fit of the largest case above
    N, d, h, r, sl = 2049, 256, 512, 1792, 256
    assert _workspace_bytes(N, h, r, sl) > SCRATCH
    w = psi.psi_ffn_weight(None, 256, d, h, r, sl)
    with pytest.raises(psi.PsiError) as e:
        psi.psi_ffn_resident_noalloc(256, N, w, 256, 256, None, 256, 0, 0)
    assert e.value.status == psi.PSI_ERR_CAPACITY
