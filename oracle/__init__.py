"""CPU oracle for the paged BF16 operators of PSI (test infrastructure).

This package is test infrastructure, not product code.  Only the tests, the
smoke check of ``__graft_entry__`` and the CPU-baseline leg of ``bench.py``
may import it.  It shares no code with the CUDA library: it has its own BF16
decoder and round-to-nearest-even, and evaluates every operator from its
plain dense definition in float64, rounding once to BF16 at each declared
write boundary.

Source: Precision-Preserving Subtensor Inference (PSI, arXiv 2611.08023),
section II-B Eqs.(2)-(4) (partitioned FFN, online-softmax attention,
full-row RMS normalisation, split RoPE), section II-C Eq.(5) (BF16
round-to-nearest-even and write boundaries), section III-A (bias added
before the single BF16 write, FP32-fidelity attention weights, and the
baseline variant without those changes) and section IV-B Eq.(6) (the exact
sum of an output element, rounded a single time).

Modules
-------
bf16    decoding, encoding and rounding of BF16 values (float64 and exact
        dyadic rationals)
ops     linear (and its baseline rounding order), FFN, attention (dense,
        online, and with BF16 numerator weights), RMSNorm, split RoPE and
        the projection with RoPE
grade   ulp distances and the tolerance used to compare a result with the
        oracle

Parity status: every function here is pinned by tests under ``tests/``
against the worked values of Eq.(5) and Eq.(6), closed forms, library
routines and exact rational brute force; none is "parity unpinned".
"""
from . import bf16, ops, grade  # noqa: F401
