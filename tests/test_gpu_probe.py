"""Same-input operator probes: the modified numerics against the paper's
baseline variant on identical inputs (PSI section IV-B, with section III-A's
two changes: FP32 bias before the single BF16 write, FP32 exponential
weights in attention).

The paper probed a full-shape audio FFN up projection (1,032,192 outputs =
126 tokens x 8192 hidden) and an audio self-attention (258,048 outputs).
These probes use the same token count and widths on seeded synthetic
inputs, count differing BF16 elements against the exact result rounded
once (the oracle), and report relative L2 errors.  Run with -s to see the
numbers.
"""
import json
import math

import numpy as np
import pytest
import torch

from weight_streamed_bf16_gb300 import psi
from weight_streamed_bf16_gb300.torch_io import heads_view

from gpu_cases import ensure_lib, f64, ops, run_linear

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _stats(y, ref_exact_bf16, ref64):
    """Differing BF16 elements and rel-L2 against the exact result rounded
    once (the paper's probe metrics), and rel-L2 against the unrounded
    float64 value."""
    yf = f64(y)
    nrm = np.linalg.norm(ref64.ravel())
    return {"differing": int(np.count_nonzero(yf != ref_exact_bf16)),
            "rel_l2": float(np.linalg.norm((yf - ref_exact_bf16).ravel()) / nrm),
            "rel_l2_vs_f64": float(np.linalg.norm((yf - ref64).ravel()) / nrm)}


def test_probe_projection_bias_order():
    """126 tokens x 8192 hidden up projection (d 2048), bias ~N(0, 0.5^2) so
    that the bias is comparable to the product."""
    g = torch.Generator().manual_seed(126)
    X = torch.randn(126, 2048, generator=g).to(torch.bfloat16)
    U = (torch.randn(8192, 2048, generator=g) / math.sqrt(2048)).to(torch.bfloat16)
    a = (torch.randn(8192, generator=g) * 0.5).to(torch.bfloat16)
    mod = run_linear(X, U, a, 2048, 2)
    base = run_linear(X, U, a, 2048, 2, flags=psi.PSI_BIAS_AFTER_BF16)
    ex = ops.linear(f64(X), f64(U), f64(a))
    s_mod, s_base = _stats(mod, ex.y, ex.y64), _stats(base, ex.y, ex.y64)
    n_between = int(torch.count_nonzero(mod.view(torch.int16) != base.view(torch.int16)))
    print(json.dumps({"probe": "projection 126x2048 -> 8192", "elements": mod.numel(),
                      "modified_vs_baseline_differing": n_between,
                      "modified": s_mod, "baseline": s_base}))
    assert s_mod["differing"] * 10 < s_base["differing"]
    assert n_between > 0.01 * mod.numel()


def test_probe_attention_weights():
    """126 tokens, 32 heads x 128: FP32 against BF16 numerator weights."""
    g = torch.Generator().manual_seed(127)
    H, N, dh = 32, 126, 128
    Q = torch.randn(H, N, dh, generator=g).to(torch.bfloat16)
    K = torch.randn(H, N, dh, generator=g).to(torch.bfloat16)
    V = torch.randn(H, N, dh, generator=g).to(torch.bfloat16)
    sc = 1 / math.sqrt(dh)
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    s = torch.cuda.current_stream()
    outs = {}
    for name, flags in [("modified", 0), ("baseline", psi.PSI_ATTN_BF16_WEIGHTS)]:
        O = torch.empty_like(Qd)
        psi.psi_attn_partitioned(heads_view(Qd), heads_view(Kd), heads_view(Vd), heads_view(O), H,
                                 N, N, dh, sc, 128, s.cuda_stream, flags)
        psi.psi_stream_wait(s.cuda_stream)
        outs[name] = O.cpu()
    ex = ops.attention_heads(f64(Q), f64(K), f64(V), sc)
    s_mod = _stats(outs["modified"], ex.y, ex.y64)
    s_base = _stats(outs["baseline"], ex.y, ex.y64)
    print(json.dumps({"probe": "attention 126 tokens, 32 x 128", "elements": outs["modified"].numel(),
                      "modified": s_mod, "baseline": s_base}))
    assert s_mod["differing"] * 5 < s_base["differing"]
    assert s_mod["rel_l2"] < s_base["rel_l2"]
