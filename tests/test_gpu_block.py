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
