"""The synthetic block (d 4096, 6144 tokens, 32 heads x 128, FFN 16384) and a
short stack of it, at full size on the GPU.

Parity: same-input operator probes (PSI section IV-B): every operator's GPU
output is compared with the oracle on sampled rows, fed the GPU's own BF16
inputs to that operator.  Transport controls (section IV-C/IV-D, Table V):
resident weights, streamed weights through 32/80/256 MiB arenas and
compute-stream copies give bitwise-identical outputs.
"""
import math

import numpy as np
import pytest
import torch

import psi_synth
from weight_streamed_bf16_gb300 import psi
from weight_streamed_bf16_gb300.block import BlockRunner, BlockShape, BlockWeights
from weight_streamed_bf16_gb300.torch_io import Arena

from gpu_cases import check, ensure_lib, f64, ops

pytestmark = pytest.mark.gpu
MiB = 1 << 20
CFG = psi_synth.BLOCK


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _shape():
    return BlockShape(d=CFG.d, N=CFG.N, heads=CFG.heads, dh=CFG.dh, hidden=CFG.hidden,
                      slice=CFG.slice, page_bytes=CFG.page_bytes)


def _weights(block, resident):
    w = psi_synth.block_weights(CFG, block=block, device="cuda")
    w = {k: v.cpu() for k, v in w.items()}
    return w, BlockWeights(w, _shape(), resident=resident)


@pytest.fixture(scope="module")
def block_run():
    w, bw = _weights(0, resident=True)
    arena = Arena(CFG.page_bytes, 5)
    runner = BlockRunner(_shape(), arena)
    X = psi_synth.block_input(CFG, device="cuda")
    Y = torch.empty_like(X)
    runner.forward(X, bw, Y, 0)       # streamed through the 80 MiB arena
    arena.sync()
    Yr = torch.empty_like(X)
    runner.forward(X, bw, Yr, psi.PSI_RESIDENT)
    arena.sync()
    out = {"X": X.cpu(), "h": runner.h.cpu(), "att": runner.att.cpu(),
           "x1": runner.x1.cpu(), "Y": Y.cpu(), "Yr": Yr.cpu(), "w": w}
    arena.close()
    return out


ROWS = np.array([0, 1, 127, 128, 2049, 4095, 5000, 6143])


def test_block_qkv_probe(block_run):
    r, w = block_run, block_run["w"]
    res = ops.linear(f64(r["X"][ROWS]), f64(w["Wqkv"]), f64(w["bqkv"]))
    rep = check(r["h"][ROWS], res, what="qkv")
    assert rep["max_rel_err"] <= 1e-2


def test_block_attention_probe(block_run):
    r = block_run
    H, dh = CFG.heads, CFG.dh
    h = f64(r["h"])
    att = r["att"]
    for hd in (0, 7, 31):
        q = h[ROWS, hd * dh:(hd + 1) * dh]
        k = h[:, H * dh + hd * dh:H * dh + (hd + 1) * dh]
        v = h[:, 2 * H * dh + hd * dh:2 * H * dh + (hd + 1) * dh]
        res = ops.attention(q, k, v, 1 / math.sqrt(dh))
        check(att[ROWS, hd * dh:(hd + 1) * dh], res, what=f"attention head {hd}")


@pytest.mark.parametrize("hd", [0, 31])
def test_block_attention_full_rows(block_run, hd):
    """All 6144 query rows of a head of the block's attention (key blocks of
    128, heads read in place from the fused QKV output), against the dense
    float64 softmax: head 0 runs in whole units, head 31 holds the partial
    last wave, whose units the kernel cuts into key ranges and merges by the
    Eq.(4) update (768 units on 152 SMs leave 8 for the tail split: head 31's
    query rows 4096..6143)."""
    r = block_run
    H, dh = CFG.heads, CFG.dh
    h = f64(r["h"])
    q = h[:, hd * dh:(hd + 1) * dh]
    k = h[:, H * dh + hd * dh:H * dh + (hd + 1) * dh]
    v = h[:, 2 * H * dh + hd * dh:2 * H * dh + (hd + 1) * dh]
    res = ops.attention(q, k, v, 1 / math.sqrt(dh))
    rep = check(r["att"][:, hd * dh:(hd + 1) * dh], res, what=f"block attention head {hd}")
    assert rep["n"] == CFG.N * dh


# 256 token rows spread over all 6144 (every 24th, first and last included)
WIDE = np.unique(np.concatenate([np.arange(0, CFG.N, 24), [CFG.N - 1]]))


def test_block_projection_probes_wide(block_run):
    """The block's QKV projection, out-projection and FFN on 257 token rows
    spread over the whole sequence, each fed the GPU's own BF16 inputs to the
    operator (the same-input probes of section IV-B), element by element."""
    r, w = block_run, block_run["w"]
    res = ops.linear(f64(r["X"][WIDE]), f64(w["Wqkv"]), f64(w["bqkv"]))
    check(r["h"][WIDE], res, what="qkv, 257 rows")
    res = ops.linear(f64(r["att"][WIDE]), f64(w["Wo"]), f64(w["bo"]),
                     residual=f64(r["X"][WIDE]))
    check(r["x1"][WIDE], res, what="out-proj, 257 rows")
    x1 = f64(r["x1"][WIDE])
    res = ops.ffn(x1, f64(w["W1"]), f64(w["W2"]), f64(w["a1"]), f64(w["b1"]), residual=x1)
    check(r["Y"][WIDE], res, what="ffn, 257 rows")


def test_stack_last_block_probes():
    """A 4-block stack streamed through the 80 MiB arena: the last block's
    operators against the oracle on its own GPU inputs (QKV, attention of
    two heads, out-projection and FFN on sampled rows), so accuracy holds
    after the residual stream has passed three blocks."""
    ws = [_weights(b, resident=False) for b in range(4)]
    X = psi_synth.block_input(CFG, device="cuda")
    arena = Arena(CFG.page_bytes, 5)
    runner = BlockRunner(_shape(), arena)
    Y, tmp = torch.empty_like(X), torch.empty_like(X)
    runner.stack(X, [bw for _, bw in ws], Y, tmp, 0)   # block 3 reads tmp, writes Y
    arena.sync()
    w = ws[3][0]
    x_in, h, att, x1, y = (t.cpu() for t in (tmp, runner.h, runner.att, runner.x1, Y))
    arena.close()
    rows = WIDE[::4]
    check(h[rows], ops.linear(f64(x_in[rows]), f64(w["Wqkv"]), f64(w["bqkv"])),
          what="stack block 3 qkv")
    H, dh = CFG.heads, CFG.dh
    hf = f64(h)
    for hd in (5, 30):
        q = hf[rows, hd * dh:(hd + 1) * dh]
        k = hf[:, H * dh + hd * dh:H * dh + (hd + 1) * dh]
        v = hf[:, 2 * H * dh + hd * dh:2 * H * dh + (hd + 1) * dh]
        check(att[rows, hd * dh:(hd + 1) * dh], ops.attention(q, k, v, 1 / math.sqrt(dh)),
              what=f"stack block 3 attention head {hd}")
    check(x1[rows], ops.linear(f64(att[rows]), f64(w["Wo"]), f64(w["bo"]),
                               residual=f64(x_in[rows])), what="stack block 3 out-proj")
    x1r = f64(x1[rows])
    check(y[rows], ops.ffn(x1r, f64(w["W1"]), f64(w["W2"]), f64(w["a1"]), f64(w["b1"]),
                           residual=x1r), what="stack block 3 ffn")
    assert torch.isfinite(y.float()).all()


def test_block_out_proj_probe(block_run):
    r, w = block_run, block_run["w"]
    res = ops.linear(f64(r["att"][ROWS]), f64(w["Wo"]), f64(w["bo"]),
                     residual=f64(r["X"][ROWS]))
    check(r["x1"][ROWS], res, what="out-proj")


def test_block_ffn_probe(block_run):
    r, w = block_run, block_run["w"]
    x1 = f64(r["x1"][ROWS])
    res = ops.ffn(x1, f64(w["W1"]), f64(w["W2"]), f64(w["a1"]), f64(w["b1"]), residual=x1)
    rep = check(r["Y"][ROWS], res, what="ffn")
    assert rep["max_rel_err"] <= 1e-2


def test_block_resident_equals_streamed(block_run):
    assert torch.equal(block_run["Y"].view(torch.int16), block_run["Yr"].view(torch.int16))
    assert torch.isfinite(block_run["Y"].float()).all()


def test_stack_transport_controls_bitwise():
    """Two blocks (the ring continues across operators and blocks): 32, 80
    and 256 MiB arenas, compute-stream copies and resident weights all give
    the same output bytes."""
    blocks = [_weights(b, resident=True)[1] for b in range(2)]
    X = psi_synth.block_input(CFG, device="cuda")
    outs = []
    for arena_mib, flags in [(80, 0), (32, 0), (256, 0), (80, psi.PSI_SYNC_COPY),
                             (80, psi.PSI_RESIDENT)]:
        arena = Arena(CFG.page_bytes, arena_mib * MiB // CFG.page_bytes)
        runner = BlockRunner(_shape(), arena)
        Y, tmp = torch.empty_like(X), torch.empty_like(X)
        runner.stack(X, blocks, Y, tmp, flags)
        arena.sync()
        st = arena.stats()
        if not flags & psi.PSI_RESIDENT:
            assert st["pages_streamed"] == 2 * 24
            assert st["h2d_bytes"] == 2 * CFG.weight_bytes
        outs.append(Y.cpu())
        arena.close()
    for o in outs[1:]:
        assert torch.equal(outs[0].view(torch.int16), o.view(torch.int16))


# ---------------------------------------------------- pre-norm block (f2) --
def _pn_shape():
    return BlockShape(d=CFG.d, N=CFG.N, heads=CFG.heads, dh=CFG.dh, hidden=CFG.hidden,
                      slice=CFG.slice, page_bytes=CFG.page_bytes, prenorm=True, eps=CFG.eps)


@pytest.fixture(scope="module")
def prenorm_run():
    w = {k: v.cpu() for k, v in psi_synth.block_weights(CFG, block=0, device="cuda").items()}
    w["gamma1"], w["gamma2"] = psi_synth.norm_gains(CFG)
    bw = BlockWeights(w, _pn_shape(), resident=True)
    cos, sin = psi_synth.rope_table(CFG.N, CFG.dh)
    arena = Arena(CFG.page_bytes, 5)
    runner = BlockRunner(_pn_shape(), arena, rope=(cos, sin))
    X = psi_synth.block_input(CFG, device="cuda")
    Y = torch.empty_like(X)
    runner.forward(X, bw, Y, 0)
    arena.sync()
    Yr = torch.empty_like(X)
    runner.forward(X, bw, Yr, psi.PSI_RESIDENT)
    arena.sync()
    # the first normalisation's output, recomputed by the same kernel (its
    # buffer is reused by the second one)
    n0 = torch.empty_like(X)
    psi.psi_rmsnorm(X.data_ptr(), CFG.d, CFG.N, CFG.d, bw.gamma1.data_ptr(), CFG.eps,
                    n0.data_ptr(), CFG.d, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    out = {"X": X.cpu(), "n0": n0.cpu(), "h": runner.h.cpu(), "att": runner.att.cpu(),
           "x1": runner.x1.cpu(), "n1": runner.xn.cpu(), "Y": Y.cpu(), "Yr": Yr.cpu(),
           "w": w, "cos": cos.double().numpy(), "sin": sin.double().numpy()}
    arena.close()
    return out


def test_prenorm_norm_probes(prenorm_run):
    r, w = prenorm_run, prenorm_run["w"]
    eps = np.float64(np.float32(CFG.eps))
    check(r["n0"][ROWS], ops.rmsnorm(f64(r["X"][ROWS]), f64(w["gamma1"]), eps), what="norm 1")
    check(r["n1"][ROWS], ops.rmsnorm(f64(r["x1"][ROWS]), f64(w["gamma2"]), eps), what="norm 2")


def test_prenorm_qkv_rope_probe(prenorm_run):
    r, w = prenorm_run, prenorm_run["w"]
    H, dh = CFG.heads, CFG.dh
    res = ops.linear_rope(f64(r["n0"][ROWS]), f64(w["Wqkv"]), f64(w["bqkv"]),
                          r["cos"][ROWS], r["sin"][ROWS], dh, 2 * H * dh)
    rep = check(r["h"][ROWS], res, what="qkv rope")
    assert rep["max_rel_err"] <= 1e-2


def test_prenorm_attention_and_ffn_probes(prenorm_run):
    r, w = prenorm_run, prenorm_run["w"]
    H, dh = CFG.heads, CFG.dh
    h = f64(r["h"])
    for hd in (0, 31):
        q = h[ROWS, hd * dh:(hd + 1) * dh]
        k = h[:, H * dh + hd * dh:H * dh + (hd + 1) * dh]
        v = h[:, 2 * H * dh + hd * dh:2 * H * dh + (hd + 1) * dh]
        check(r["att"][ROWS, hd * dh:(hd + 1) * dh], ops.attention(q, k, v, 1 / math.sqrt(dh)),
              what=f"attention head {hd}")
    res = ops.ffn(f64(r["n1"][ROWS]), f64(w["W1"]), f64(w["W2"]), f64(w["a1"]), f64(w["b1"]),
                  residual=f64(r["x1"][ROWS]))
    rep = check(r["Y"][ROWS], res, what="ffn")
    assert rep["max_rel_err"] <= 1e-2


def test_prenorm_resident_equals_streamed(prenorm_run):
    assert torch.equal(prenorm_run["Y"].view(torch.int16), prenorm_run["Yr"].view(torch.int16))
    assert torch.isfinite(prenorm_run["Y"].float()).all()
