"""Partitioned attention on the GPU against the oracle (PSI section II-B
Eqs.(3)-(4), FP32 online accumulation of section III-A)."""
import math

import numpy as np
import pytest
import torch

import psi_synth
from weight_streamed_bf16_gb300 import psi

from gpu_cases import check, ensure_lib, f64, ops, run_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _qkv(H, Nq, Nk, seed, dh=128):
    g = torch.Generator().manual_seed(seed)
    Q = torch.randn(H, Nq, dh, generator=g).to(torch.bfloat16)
    K = torch.randn(H, Nk, dh, generator=g).to(torch.bfloat16)
    V = torch.randn(H, Nk, dh, generator=g).to(torch.bfloat16)
    return Q, K, V


@pytest.mark.parametrize("key_block", [128, 256])
@pytest.mark.parametrize("H,Nq,Nk", [
    (1, 128, 128),     # one tile each
    (2, 200, 300),     # ragged queries and keys (last key tile 44 keys)
    (3, 64, 1),        # a single key: O = B(v)
    (1, 130, 129),     # one key past a tile boundary
    (2, 256, 1024),    # several key blocks (online rescaling)
    (1, 384, 384),     # 256-key blocks: the last block has one 128-key sub-tile
])
def test_attention_shapes(H, Nq, Nk, key_block):
    Q, K, V = _qkv(H, Nq, Nk, H * 7 + Nq + Nk)
    sc = 1 / math.sqrt(128)
    O = run_attention(Q.cuda(), K.cuda(), V.cuda(), sc, key_block=key_block).cpu()
    res = ops.attention_heads(f64(Q), f64(K), f64(V), sc)
    rep = check(O, res, what=f"attn {H}x{Nq}x{Nk}")
    assert rep["all_finite"]


@pytest.mark.parametrize("key_block", [128, 256])
def test_attention_single_key_exact(key_block):
    Q, K, V = _qkv(2, 100, 1, 3)
    O = run_attention(Q.cuda(), K.cuda(), V.cuda(), 0.1, key_block=key_block).cpu()
    assert torch.equal(O.view(torch.int16), V.expand(2, 100, 128).contiguous().view(torch.int16))


def test_attention_key_block_partitions_agree():
    """Eq.(4) gives the dense result for any complete key partition: 128- and
    256-key blocks differ only by rounding (both within tolerance of the
    oracle, and close to each other)."""
    Q, K, V = _qkv(2, 256, 1000, 5)
    sc = 1 / math.sqrt(128)
    a = run_attention(Q.cuda(), K.cuda(), V.cuda(), sc, key_block=128).cpu()
    b = run_attention(Q.cuda(), K.cuda(), V.cuda(), sc, key_block=256).cpu()
    res = ops.attention_heads(f64(Q), f64(K), f64(V), sc)
    check(a, res, what="kb128")
    check(b, res, what="kb256")
    d = (a.float() - b.float()).abs().max().item()
    assert d <= 2 ** -6


@pytest.fixture(scope="module")
def attn_config_run():
    """Q, K, V [32 x 4096 x 128], scale 1/sqrt(128), key blocks of 256: the
    full configuration on the GPU, once for the tests below."""
    cfg = psi_synth.ATTN
    Q, K, V = psi_synth.attn_inputs(cfg)
    O = run_attention(Q.cuda(), K.cuda(), V.cuda(), cfg.scale, key_block=cfg.key_block).cpu()
    return cfg, f64(Q), f64(K), f64(V), O


def test_attention_config_sampled_rows(attn_config_run):
    """Every head of the attention configuration on sampled query rows."""
    cfg, Qf, Kf, Vf, O = attn_config_run
    rows = np.array([0, 1, 127, 128, 2047, 2048, 4000, 4095])
    worst = 0.0
    for h in range(cfg.heads):
        res = ops.attention(Qf[h], Kf[h], Vf[h], cfg.scale, rows=rows)
        rep = check(O[h][rows], res, what=f"head {h}")
        worst = max(worst, rep["max_rel_err"])
    assert worst <= 1e-2
    assert np.isfinite(f64(O)).all()


@pytest.mark.parametrize("head", [0, 15, 31])
def test_attention_config_full_rows(attn_config_run, head):
    """All 4096 query rows of a head of the attention configuration (the
    first, a middle and the last head), element by element against the dense
    float64 softmax of Eq.(3)."""
    cfg, Qf, Kf, Vf, O = attn_config_run
    res = ops.attention(Qf[head], Kf[head], Vf[head], cfg.scale)
    rep = check(O[head], res, what=f"head {head}, all rows")
    assert rep["n"] == cfg.N * cfg.dh


@pytest.mark.parametrize("key_block", [128, 256])
def test_attention_interleaved_layout(key_block):
    """Heads interleaved within a token row (the fused QKV projection output):
    Q, K, V read in place from [tokens x 3*H*dh], O written to [tokens x H*dh]."""
    H, N, dh = 4, 300, 128
    g = torch.Generator().manual_seed(21)
    qkv = torch.randn(N, 3 * H * dh, generator=g).to(torch.bfloat16).cuda()
    view = qkv.view(N, 3, H, dh)
    Q = view[:, 0].permute(1, 0, 2)   # [H x N x dh], strides (dh, 3*H*dh, 1)
    K = view[:, 1].permute(1, 0, 2)
    V = view[:, 2].permute(1, 0, 2)
    Obuf = torch.full((N, H * dh), float("nan"), dtype=torch.bfloat16, device="cuda")
    O = Obuf.view(N, H, dh).permute(1, 0, 2)
    run_attention(Q, K, V, 1 / math.sqrt(dh), key_block=key_block, O=O)
    ref = run_attention(Q.contiguous(), K.contiguous(), V.contiguous(), 1 / math.sqrt(dh),
                        key_block=key_block)
    assert torch.equal(O.contiguous().view(torch.int16), ref.view(torch.int16))
    res = ops.attention_heads(f64(Q), f64(K), f64(V), 1 / math.sqrt(dh))
    check(O.contiguous().cpu(), res, what="interleaved")


def test_attention_rejects_unsupported():
    Q, K, V = _qkv(1, 8, 8, 1)
    with pytest.raises(psi.PsiError) as e:
        run_attention(Q.cuda(), K.cuda(), V.cuda(), 0.1, key_block=64)
    assert e.value.status == psi.PSI_ERR_UNSUPPORTED


@pytest.mark.parametrize("key_block", [128, 256])
def test_attention_bf16_numerator_weights(key_block):
    """The baseline variant (section III-A): numerator weights rounded to
    BF16, graded against the oracle's online recurrence over the same key
    blocks; its error against exact attention is far above the FP32-weight
    kernel's."""
    Q, K, V = _qkv(2, 256, 1000, 9)
    sc = 1 / math.sqrt(128)
    s = torch.cuda.current_stream()
    O = torch.empty(2, 256, 128, dtype=torch.bfloat16, device="cuda")
    from weight_streamed_bf16_gb300.torch_io import heads_view
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    psi.psi_attn_partitioned(heads_view(Qd), heads_view(Kd), heads_view(Vd), heads_view(O), 2,
                             256, 1000, 128, sc, key_block, s.cuda_stream,
                             psi.PSI_ATTN_BF16_WEIGHTS)
    psi.psi_stream_wait(s.cuda_stream)
    Of = O.cpu()
    for h in range(2):
        res = ops.attention_bf16_weights(f64(Q)[h], f64(K)[h], f64(V)[h], sc, key_block)
        check(Of[h], res, what=f"bf16 weights head {h}")
    # against exact attention rounded once, the BF16 weights leave many more
    # differing BF16 elements than the FP32 weights (the paper's probe metric)
    exact = ops.attention_heads(f64(Q), f64(K), f64(V), sc)
    fp32 = run_attention(Qd, Kd, Vd, sc, key_block=key_block).cpu()
    n_b = int(np.count_nonzero(f64(Of) != exact.y))
    n_f = int(np.count_nonzero(f64(fp32) != exact.y))
    assert n_b > 3 * n_f, (n_b, n_f)


@pytest.mark.parametrize("key_block,H,Nq,Nk", [
    (128, 20, 2048, 2048),   # 160 units of 256 queries: 8 tail units, 16 key ranges each
    (256, 10, 2048, 2000),   # 160 units of 128 queries, ragged last key block
    (128, 20, 2000, 1500),   # ragged queries in the tail units, 12 key blocks
])
def test_attention_tail_split(key_block, H, Nq, Nk):
    """With a workspace, the partial last wave of (head, query tile) units
    is split into key ranges and merged by Eq.(4)'s update; the split units
    (the last ones: the last heads) still match the oracle, and the other
    units are bitwise those of the unsplit kernel."""
    Q, K, V = _qkv(H, Nq, Nk, H + Nq + Nk)
    sc = 1 / math.sqrt(128)
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    a = run_attention(Qd, Kd, Vd, sc, key_block=key_block, split=True).cpu()
    b = run_attention(Qd, Kd, Vd, sc, key_block=key_block).cpu()
    assert torch.isfinite(a.float()).all()
    rows = np.array([0, 1, 127, 128, 255, 1000, Nq - 2, Nq - 1])
    for hd in (0, H - 2, H - 1):
        res = ops.attention(f64(Q)[hd], f64(K)[hd], f64(V)[hd], sc, rows=rows)
        check(a[hd][rows], res, what=f"split head {hd}")
    # the first heads are whole units in both launches
    assert torch.equal(a[:H // 2].view(torch.int16), b[:H // 2].view(torch.int16))
    assert (a.float() - b.float()).abs().max().item() <= 2 ** -6


@pytest.mark.parametrize("key_block,H,Nk", [
    (128, 20, 2048),
    (256, 10, 2000),   # key ranges start inside the K ring's three stages; ragged last block
])
def test_attention_tail_split_full_rows(key_block, H, Nk):
    """Every row of the split units against the oracle (one tail head)."""
    Nq = 2048
    Q, K, V = _qkv(H, Nq, Nk, 77)
    sc = 1 / math.sqrt(128)
    a = run_attention(Q.cuda(), K.cuda(), V.cuda(), sc, key_block=key_block, split=True).cpu()
    res = ops.attention(f64(Q)[H - 1], f64(K)[H - 1], f64(V)[H - 1], sc)
    check(a[H - 1], res, what=f"tail head, all rows, key blocks of {key_block}")


def test_attention_workspace_too_small():
    Q, K, V = _qkv(1, 8, 8, 1)
    O = torch.empty(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(16, dtype=torch.float32, device="cuda")
    from weight_streamed_bf16_gb300.torch_io import heads_view
    with pytest.raises(psi.PsiError) as e:
        psi.psi_attn_partitioned_ws(heads_view(Q.cuda()), heads_view(K.cuda()),
                                    heads_view(V.cuda()), heads_view(O), 1, 8, 8, 128, 0.1, 128,
                                    ws.data_ptr(), 64, torch.cuda.current_stream().cuda_stream)
    assert e.value.status == psi.PSI_ERR_INVALID_ARG


@pytest.mark.parametrize("key_block", [128, 256])
@pytest.mark.parametrize("sign", [1, -1])
@pytest.mark.parametrize("flags", [0, psi.PSI_ATTN_BF16_WEIGHTS])
def test_attention_reference_moves_in_later_blocks(key_block, sign, flags):
    """Scores that grow by about 13 (log2 units) every 256 keys move the
    reference point of the exponents after the first block (reading of
    Eq.(4) with a lagging reference): O is rescaled in tensor memory, and
    with 256-key blocks sub-tile 0's weights, formed ahead against the old
    reference, are formed again.  A negative scale turns the extremum into a
    minimum."""
    g = torch.Generator().manual_seed(21 + key_block + sign)
    H, Nq, Nk, dh = 2, 256, 1024, 128
    Q = (1.0 + 0.01 * torch.randn(H, Nq, dh, generator=g)).to(torch.bfloat16)
    level = (torch.arange(Nk) // 256).to(torch.float32) * (100.0 / dh) * sign
    K = (level[None, :, None] + 0.05 * torch.randn(H, Nk, dh, generator=g)).to(torch.bfloat16)
    V = torch.randn(H, Nk, dh, generator=g).to(torch.bfloat16)
    scale = sign / math.sqrt(dh)
    O = run_attention(Q.cuda(), K.cuda(), V.cuda(), scale, key_block=key_block, flags=flags).cpu()
    what = f"moving reference, kb {key_block}, sign {sign}, flags {flags}"
    if flags & psi.PSI_ATTN_BF16_WEIGHTS:
        for h in range(H):
            check(O[h], ops.attention_bf16_weights(f64(Q)[h], f64(K)[h], f64(V)[h], scale,
                                                   key_block), what=f"{what}, head {h}")
    else:
        check(O, ops.attention_heads(f64(Q), f64(K), f64(V), scale), what=what)
