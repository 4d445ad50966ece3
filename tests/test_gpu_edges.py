"""Edge cases of the paged operators on the GPU: empty inputs, single tokens,
the narrowest K, zero operands (the result is the rounded bias), inputs
wider than one k-block and the largest single page the config allows."""
import math

import numpy as np
import pytest
import torch

from weight_streamed_bf16_gb300 import psi
from weight_streamed_bf16_gb300.torch_io import Arena, LinearWeight, heads_view

from gpu_cases import bf16, check, ensure_lib, f64, ops, run_attention, run_ffn, run_linear

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _bf16(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


def test_linear_zero_tokens_enqueues_nothing():
    W = _bf16((256, 128), 0.1, 1)
    b = _bf16((256,), 0.1, 2)
    arena = Arena(256 * 128 * 2, 2)
    w = LinearWeight(W, 256 * 128 * 2)
    X = torch.empty(1, 128, dtype=torch.bfloat16, device="cuda")
    Y = torch.full((1, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    bd = b.cuda()
    psi.psi_linear_paged(arena.handle, X.data_ptr(), 0, 128, w.desc(), bd.data_ptr(), None,
                         Y.data_ptr(), 256, 0)
    arena.sync()
    assert torch.all(Y == 7.0)
    arena.close()


def test_attention_zero_queries_enqueues_nothing():
    Q = torch.empty(2, 1, 128, dtype=torch.bfloat16, device="cuda")
    K = _bf16((2, 8, 128), 1.0, 3).cuda()
    O = torch.full((2, 1, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream()
    psi.psi_attn_partitioned(heads_view(Q), heads_view(K), heads_view(K), heads_view(O), 2, 0, 8,
                             128, 0.1, 128, s.cuda_stream, 0)
    torch.cuda.synchronize()
    assert torch.all(O == 5.0)


@pytest.mark.parametrize("N,K,M", [(1, 64, 64), (1, 8, 200), (3, 8, 16), (2, 16384, 320)])
def test_linear_single_tokens_and_narrow_or_wide_k(N, K, M):
    X = _bf16((N, K), 1.0, N + K)
    W = _bf16((M, K), 1 / math.sqrt(K), M)
    b = _bf16((M,), 0.1, 5)
    page_rows = min(M, 128)
    Y = run_linear(X, W, b, page_rows, 2)
    check(Y, ops.linear(f64(X), f64(W), f64(b)), what=f"linear {N}x{K}x{M}")


def test_linear_zero_operands_give_the_rounded_bias():
    N, K, M = 300, 512, 384
    X = torch.zeros(N, K, dtype=torch.bfloat16)
    W = _bf16((M, K), 0.1, 6)
    b = _bf16((M,), 3.0, 7)
    Y = run_linear(X, W, b, 128, 2)
    assert torch.equal(Y.view(torch.int16), b.expand(N, M).contiguous().view(torch.int16))
    W0 = torch.zeros(M, K, dtype=torch.bfloat16)
    Y0 = run_linear(_bf16((N, K), 1.0, 8), W0, b, 128, 2)
    assert torch.equal(Y0.view(torch.int16), b.expand(N, M).contiguous().view(torch.int16))


def test_ffn_single_token_and_zero_input():
    d, h, r, sl = 256, 512, 256, 128
    U = _bf16((h, d), 1 / math.sqrt(d), 9)
    V = _bf16((r, h), 1 / math.sqrt(h), 10)
    a = _bf16((h,), 0.5, 11)
    bb = _bf16((r,), 0.5, 12)
    for X in (_bf16((1, d), 1.0, 13), torch.zeros(5, d, dtype=torch.bfloat16)):
        Y = run_ffn(X, U, V, a, bb, sl, 2)
        check(Y, ops.ffn(f64(X), f64(U), f64(V), f64(a), f64(bb)), what=f"ffn {X.shape[0]} rows")


def test_attention_single_query_and_long_keys():
    g = torch.Generator().manual_seed(14)
    Q = torch.randn(3, 1, 128, generator=g).to(torch.bfloat16)
    K = torch.randn(3, 5000, 128, generator=g).to(torch.bfloat16)
    V = torch.randn(3, 5000, 128, generator=g).to(torch.bfloat16)
    for kb in (128, 256):
        O = run_attention(Q.cuda(), K.cuda(), V.cuda(), 1 / math.sqrt(128), key_block=kb).cpu()
        check(O, ops.attention_heads(f64(Q), f64(K), f64(V), 1 / math.sqrt(128)),
              what=f"one query, kb {kb}")


def test_attention_equal_keys_give_the_mean_of_values():
    """All keys equal: every weight is the same, O = B(mean of v) per column
    (the sum of 512 BF16 values over 512 is exact in FP32 here)."""
    g = torch.Generator().manual_seed(15)
    Q = torch.randn(1, 256, 128, generator=g).to(torch.bfloat16)
    K = torch.randn(1, 1, 128, generator=g).to(torch.bfloat16).expand(1, 512, 128).contiguous()
    V = (torch.randint(-8, 8, (1, 512, 128), generator=g).float() / 8).to(torch.bfloat16)
    O = run_attention(Q.cuda(), K.cuda(), V.cuda(), 0.1, key_block=128).cpu()
    want = bf16.round_bf16(f64(V)[0].mean(axis=0))
    assert np.array_equal(f64(O)[0], np.broadcast_to(want, (256, 128)))
