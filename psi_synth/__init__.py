"""Seeded synthetic inputs for the paged BF16 operators.

This module is shared by the CUDA path (tests, bench) and by the oracle's
callers.  It holds random draws, shapes and seeds only: none of the arithmetic
of the operators.  Values are drawn as float32 normals from a torch generator
seeded per (seed, tensor id), scaled by the stated standard deviation, and
rounded once to bfloat16 by torch's own conversion (the input recipe; the same
bytes are handed to the GPU and to the oracle).

Workload shapes follow the five synthetic configurations of the paged-operator
study (PSI: Precision-Preserving Subtensor Inference, arXiv 2611.08023,
section II-B Eq.(2) for the operator shapes, section IV for the tile and arena
sizes):

* linear   : X [64 x 512], W [512 x 512], 64-row pages, 2-page arena
* ffn      : X [1024 x 2048], U [8192 x 2048], V [2048 x 8192], 1024-wide
             hidden slices, 4-slice arena
* attention: Q, K, V [32 x 4096 x 128], scale 1/sqrt(128), key blocks
* block    : d 4096, 6144 tokens, QKV [12288 x 4096], out-proj [4096 x 4096],
             FFN 4096 -> 16384 -> 4096, 16 MiB pages, 80 MiB arena
* stack    : 48 blocks of the block workload
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

__all__ = [
    "normal_bf16", "LinearCfg", "FfnCfg", "AttnCfg", "BlockCfg",
    "LINEAR", "FFN", "ATTN", "BLOCK", "STACK_BLOCKS", "tensor_ids",
    "linear_inputs", "ffn_inputs", "attn_inputs", "block_weights",
    "block_input",
]

MiB = 1 << 20


def _mix(seed: int, stream: int) -> int:
    """Distinct generator seed per (seed, tensor id); splitmix64 finaliser."""
    z = (seed * 0x9E3779B97F4A7C15 + stream * 0xBF58476D1CE4E5B9 + 1) & (2**64 - 1)
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & (2**64 - 1)
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & (2**64 - 1)
    z ^= z >> 31
    return z & 0x7FFF_FFFF_FFFF_FFFF


def normal_bf16(shape, std: float, seed: int, stream: int,
                device: str | torch.device = "cpu") -> torch.Tensor:
    """N(0, std^2) drawn in float32 on `device`, then rounded to bfloat16."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(_mix(seed, stream))
    t = torch.randn(tuple(shape), generator=g, device=dev, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


# --------------------------------------------------------------------------
# configurations
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class LinearCfg:
    N: int = 64          # tokens
    K: int = 512         # input width
    M: int = 512         # output width (rows of W)
    page_rows: int = 64  # output rows per weight page
    slots: int = 2       # pages in the arena
    seed: int = 0

    @property
    def page_bytes(self) -> int:
        return self.page_rows * self.K * 2

    @property
    def flops(self) -> int:
        return 2 * self.N * self.K * self.M


@dataclass(frozen=True)
class FfnCfg:
    N: int = 1024
    d: int = 2048        # model width (input of U, output of V)
    h: int = 8192        # hidden width
    slice: int = 1024    # hidden channels per page
    slots: int = 4
    seed: int = 0

    @property
    def r(self) -> int:  # output width of the down projection
        return self.d

    @property
    def page_bytes(self) -> int:
        return 2 * self.slice * self.d * 2  # U_J (slice x d) + V_:,J (r x slice)

    @property
    def flops(self) -> int:
        return 2 * 2 * self.N * self.d * self.h


@dataclass(frozen=True)
class AttnCfg:
    heads: int = 32
    N: int = 4096
    dh: int = 128
    key_block: int = 256
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dh)

    @property
    def flops(self) -> int:
        return 4 * self.heads * self.N * self.N * self.dh


@dataclass(frozen=True)
class BlockCfg:
    d: int = 4096
    N: int = 6144
    heads: int = 32
    dh: int = 128
    hidden: int = 16384
    slice: int = 1024
    page_bytes: int = 16 * MiB
    arena_bytes: int = 80 * MiB
    key_block: int = 256
    seed: int = 0
    eps: float = 1e-6      # RMSNorm epsilon of the pre-norm variant

    @property
    def qkv_rows(self) -> int:
        return 3 * self.heads * self.dh

    @property
    def weight_bytes(self) -> int:
        d, h = self.d, self.hidden
        return 2 * (self.qkv_rows * d + d * d + h * d + d * h)

    @property
    def linear_flops(self) -> int:
        d, h, N = self.d, self.hidden, self.N
        return 2 * N * d * (self.qkv_rows + d + 2 * h)

    @property
    def attn_flops(self) -> int:
        return 4 * self.heads * self.N * self.N * self.dh

    @property
    def flops(self) -> int:
        return self.linear_flops + self.attn_flops


LINEAR = LinearCfg()
FFN = FfnCfg()
ATTN = AttnCfg()
BLOCK = BlockCfg()
STACK_BLOCKS = 48

# tensor ids: one generator stream per tensor (per block for stacked weights)
tensor_ids = {
    "X": 1, "W": 2, "b": 3, "U": 4, "V": 5, "a": 6, "b2": 7,
    "Q": 8, "K": 9, "Vt": 10,
    "Wqkv": 11, "bqkv": 12, "Wo": 13, "bo": 14, "W1": 15, "a1": 16,
    "W2": 17, "b1": 18, "gamma1": 19, "gamma2": 20,
}


def _tid(name: str, block: int = 0) -> int:
    return tensor_ids[name] + 1000 * block


def linear_inputs(cfg: LinearCfg = LINEAR, device="cpu"):
    """X ~ N(0,1), W ~ N(0,1/K), b ~ N(0, 0.02^2)."""
    X = normal_bf16((cfg.N, cfg.K), 1.0, cfg.seed, _tid("X"), device)
    W = normal_bf16((cfg.M, cfg.K), 1.0 / math.sqrt(cfg.K), cfg.seed, _tid("W"), device)
    b = normal_bf16((cfg.M,), 0.02, cfg.seed, _tid("b"), device)
    return X, W, b


def ffn_inputs(cfg: FfnCfg = FFN, device="cpu"):
    """X ~ N(0,1), U [h x d] ~ N(0,1/d), V [r x h] ~ N(0,1/h), a, b ~ N(0,0.02^2)."""
    X = normal_bf16((cfg.N, cfg.d), 1.0, cfg.seed, _tid("X"), device)
    U = normal_bf16((cfg.h, cfg.d), 1.0 / math.sqrt(cfg.d), cfg.seed, _tid("U"), device)
    V = normal_bf16((cfg.r, cfg.h), 1.0 / math.sqrt(cfg.h), cfg.seed, _tid("V"), device)
    a = normal_bf16((cfg.h,), 0.02, cfg.seed, _tid("a"), device)
    b = normal_bf16((cfg.r,), 0.02, cfg.seed, _tid("b2"), device)
    return X, U, V, a, b


def attn_inputs(cfg: AttnCfg = ATTN, device="cpu"):
    """Q, K, V [heads x N x dh] ~ N(0,1)."""
    shp = (cfg.heads, cfg.N, cfg.dh)
    Q = normal_bf16(shp, 1.0, cfg.seed, _tid("Q"), device)
    K = normal_bf16(shp, 1.0, cfg.seed, _tid("K"), device)
    V = normal_bf16(shp, 1.0, cfg.seed, _tid("Vt"), device)
    return Q, K, V


def block_input(cfg: BlockCfg = BLOCK, device="cpu"):
    """Block input X [N x d] ~ N(0,1)."""
    return normal_bf16((cfg.N, cfg.d), 1.0, cfg.seed, _tid("X"), device)


def block_weights(cfg: BlockCfg = BLOCK, block: int = 0, device="cpu"):
    """Weights of one synthetic block, ~N(0, 1/fan_in), biases ~N(0, 0.02^2).

    Returns a dict with Wqkv [3*heads*dh x d], bqkv, Wo [d x d], bo,
    W1 (= U) [hidden x d], a1, W2 (= V) [d x hidden], b1.
    """
    d, h, s = cfg.d, cfg.hidden, cfg.seed
    q = cfg.qkv_rows
    return {
        "Wqkv": normal_bf16((q, d), 1.0 / math.sqrt(d), s, _tid("Wqkv", block), device),
        "bqkv": normal_bf16((q,), 0.02, s, _tid("bqkv", block), device),
        "Wo": normal_bf16((d, d), 1.0 / math.sqrt(d), s, _tid("Wo", block), device),
        "bo": normal_bf16((d,), 0.02, s, _tid("bo", block), device),
        "W1": normal_bf16((h, d), 1.0 / math.sqrt(d), s, _tid("W1", block), device),
        "a1": normal_bf16((h,), 0.02, s, _tid("a1", block), device),
        "W2": normal_bf16((d, h), 1.0 / math.sqrt(h), s, _tid("W2", block), device),
        "b1": normal_bf16((d,), 0.02, s, _tid("b1", block), device),
    }


def norm_gains(cfg: BlockCfg = BLOCK, block: int = 0, device="cpu"):
    """RMSNorm gains gamma1 (before the QKV projection) and gamma2 (before
    the FFN), each [d] ~ 1 + N(0, 0.1^2), drawn in FP32 and rounded to BF16."""
    out = []
    for name in ("gamma1", "gamma2"):
        g = torch.Generator(device="cpu").manual_seed(_mix(cfg.seed, _tid(name, block)))
        v = (1.0 + 0.1 * torch.randn(cfg.d, generator=g)).to(torch.bfloat16)
        out.append(v.to(device))
    return tuple(out)


def rope_table(n_tokens: int, dh: int, base: float = 10000.0, pos0: int = 0):
    """The cos/sin table a model hands to split RoPE: token n at position
    pos0 + n, frequency base^(-2j/dh) for j < dh/2, angles and their cos/sin
    in float64, rounded to FP32.  Returns two float32 CPU tensors
    [n_tokens x dh/2]."""
    pos = np.arange(pos0, pos0 + n_tokens, dtype=np.float64)[:, None]
    inv = base ** (-2.0 * np.arange(dh // 2, dtype=np.float64) / dh)
    ang = pos * inv[None, :]
    return (torch.from_numpy(np.cos(ang).astype(np.float32)),
            torch.from_numpy(np.sin(ang).astype(np.float32)))
