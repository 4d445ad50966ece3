"""Benchmark of the paged BF16 hot path on GB300.

Default workload: one synthetic transformer block (d_model 4096, 6144
tokens, fused QKV [12288 x 4096], out-proj [4096 x 4096], FFN 4096 -> 16384
-> 4096 tanh-GELU) whose 402,653,184 bytes of BF16 weights sit in pinned
host memory and stream as 16 MiB pages through an 80 MiB arena every step.
A step is one block forward: paged QKV projection, partitioned attention,
paged out-projection (+ residual), paged FFN (+ residual).

Printed: one JSON line (rank 0).  value = algorithmic block TFLOP/s
(3.092 TFLOP per block per GPU, summed over ranks); page ingest GB/s and
the roofline of the dominant kernel (the page GEMM) are reported beside it,
and, after the headline's timed region, `configs` holds the other
configurations of the study (single paged linear, paged FFN, partitioned
attention with key blocks of 256, and the 48-block stack's arena sweep with
its bitwise transport control).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl psi|reference]
                    [--workload block|ffn|linear|attention|stack]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged BF16 block TFLOP/s and page-ingest GB/s at 1 GB300, % of roofline"
MiB = 1 << 20
L2_FLUSH_BYTES = 256 * MiB


# ------------------------------------------------------------------ utils --
def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def source_digest(*names):
    h = hashlib.sha256()
    for n in names:
        h.update(open(os.path.join(ROOT, "weight_streamed_bf16_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:16]


def profile_traffic(kernel_file: str, digest: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", kernel_file)
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p):
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_digest") != digest:
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1])]
        mx = [num(r[2]) for r in rows if num(r[2])]
        pw = [num(r[3]) for r in rows if num(r[3])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": reasons}


def h2d_probe(torch, dev, nbytes=1 << 30, reps=3, streams=1):
    """Host-to-device bandwidth (GB/s, best of `reps`) of `nbytes` of pinned
    host memory copied by `streams` concurrent cudaMemcpyAsync calls, one
    per stream on equal parts; the interval runs from an event before the
    first copy to the join of the last."""
    src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream()
    side = [torch.cuda.Stream(dev) for _ in range(streams)]
    part = nbytes // streams
    best = 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        done = []
        for i, ss in enumerate(side):
            ss.wait_event(e0)
            with torch.cuda.stream(ss):
                dst[i * part:(i + 1) * part].copy_(src[i * part:(i + 1) * part],
                                                   non_blocking=True)
            e = torch.cuda.Event()
            e.record(ss)
            done.append(e)
        for e in done:
            s.wait_event(e)
        e1.record(s)
        e1.synchronize()
        best = max(best, part * streams / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del src, dst
    return best


def gemm_alone(torch, dev, wl, peaks, flush, launches=20):
    """The page GEMM where it is compute-bound: the block's first QKV page
    (2048 x 4096, resident) against X [6144 x 4096], one launch per event
    pair on the compute stream, L2 flushed before each launch; and the whole
    resident QKV projection (6 pages on the compute and auxiliary streams)
    timed the same way.  Algorithmic FLOPs 2*M*N*K over the event time,
    against the burst peak (a kernel timed alone)."""
    from weight_streamed_bf16_gb300 import psi
    from weight_streamed_bf16_gb300.torch_io import Arena
    bw = wl.blocks[0]
    X = wl.X if wl.X.dim() == 2 else wl.X[0]
    N, K = X.shape
    rows = bw.qkv.page_rows
    Wp = bw.qkv.host[:rows].to(dev)
    Wall = bw.qkv.host.to(dev)
    Y = torch.empty(N, bw.qkv.rows, dtype=torch.bfloat16, device=dev)
    arena = Arena(wl.shape.page_bytes, 1, device=dev)
    s = arena.compute
    page = psi.psi_linear_weight(0, Wp.data_ptr(), rows, K, rows)
    full = psi.psi_linear_weight(0, Wall.data_ptr(), bw.qkv.rows, K, rows)
    out = {}
    for name, desc, m in (("page", page, rows), ("qkv_resident", full, bw.qkv.rows)):
        def run():
            psi.psi_linear_paged(arena.handle, X.data_ptr(), N, K, desc, bw.bqkv.data_ptr(), None,
                                 Y.data_ptr(), bw.qkv.rows, psi.PSI_RESIDENT)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(launches)]
        with torch.cuda.stream(s):
            for _ in range(3):
                run()
            for e0, e1 in ev:
                flush.fill_(7)
                e0.record(s)
                run()
                e1.record(s)
        arena.sync()
        ms = sorted(a.elapsed_time(b) for a, b in ev)
        med = ms[len(ms) // 2]
        fl = 2.0 * N * m * K
        ach = fl / (med * 1e-3) / 1e12
        out[name] = {"ms": med, "flops": fl, "achieved": ach,
                     "frac": ach / peaks["bf16_tflops"]}
    arena.close()
    # The same two products through cuBLAS (torch.matmul), timed the same
    # way: a reference point for the kernel on this shape, not part of the
    # product path (which never calls a library GEMM).
    lib = {}
    for name, W, m in (("page", Wp, rows), ("qkv_resident", Wall, bw.qkv.rows)):
        Yl = torch.empty(N, m, dtype=torch.bfloat16, device=dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(launches)]
        with torch.cuda.stream(s):
            for _ in range(3):
                torch.matmul(X, W.t(), out=Yl)
            for e0, e1 in ev:
                flush.fill_(7)
                e0.record(s)
                torch.matmul(X, W.t(), out=Yl)
                e1.record(s)
        torch.cuda.synchronize()
        ms = sorted(a.elapsed_time(b) for a, b in ev)
        med = ms[len(ms) // 2]
        lib[name] = {"ms": med, "achieved": 2.0 * N * m * K / (med * 1e-3) / 1e12}
        del Yl
    out["cublas_same_shape"] = lib
    del Wp, Wall, Y
    return out


def ingest_alone(torch, dev, link_gbs, flush, steps=20):
    """Page ingest where it is transfer-bound: the streamed FFN configuration
    (8 pages of 8 MiB through a 4-slot arena, 68.7 GFLOP of page GEMMs, so
    the 67.1 MB of copies bound it), one step per event pair, L2 flushed
    before each and every copy of the step after its start event; weight
    bytes over the step time (median) against the H2D probe."""
    wl = FfnWorkload(torch, dev)
    s = wl.stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    with torch.cuda.stream(s):
        for _ in range(3):
            wl.step()
        for e0, e1 in ev:
            flush.fill_(5)
            e0.record(s)
            # the step's page copies start after its start event (none runs
            # ahead into the flush), so the interval holds all of its bytes
            wl.arena.copy.wait_event(e0)
            wl.step()
            e1.record(s)
    wl.arena.sync()
    ms = sorted(a.elapsed_time(b) for a, b in ev)
    med = ms[len(ms) // 2]
    gbs = wl.weight_h2d / (med * 1e-3) / 1e9
    out = {"workload": wl.name, "ms_per_step": med, "bytes_per_step": wl.weight_h2d,
           "achieved_gbs": gbs, "link_probe_gbs": link_gbs, "frac_of_link": gbs / link_gbs,
           "tflops": wl.flops / (med * 1e-3) / 1e12}
    wl.arena.close()
    return out


def aggregate_ranks(dist, device, total_ms: float, flops_per_step: float, steps: int,
                    world: int, work_ranks: int | None = None):
    """Whole-job figures: the slowest rank's time (max over ranks) bounds the
    job.  In a replicas run every rank processed `steps` steps of its own
    workload, so value = world * flops_per_step * steps / max_time; a run
    whose ranks share one workload per step (work_ranks = 1) counts it once.
    No data-path collective: only this one max-reduction of the timing."""
    import torch
    if dist is not None and world > 1:
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / steps
    n = world if work_ranks is None else work_ranks
    return total_ms, ms_per_step, flops_per_step * n / (ms_per_step * 1e-3) / 1e12


# -------------------------------------------------------------- workloads --
class Workload:
    name = ""
    flops = 0.0            # algorithmic FLOPs per step
    weight_h2d = 0         # weight bytes streamed per step
    timed_alone = False    # dominant kernel timed alone (burst peak) or in a long step

    def step(self):
        raise NotImplementedError

    def launches(self) -> int:
        raise NotImplementedError


def workload_name(args) -> str:
    """The workload description both arms print in config.workload."""
    import dataclasses

    import psi_synth
    w = args.workload
    if getattr(args, "shard", False) and w == "block":
        cfg = psi_synth.BLOCK
        return (f"synthetic transformer block x1 split by output columns over {args.gpus} "
                f"GPU(s): d_model {cfg.d}, {cfg.N} tokens, {cfg.heads} heads x {cfg.dh}, "
                f"QKV {cfg.qkv_rows}x{cfg.d} + out {cfg.d}x{cfg.d} + FFN "
                f"{cfg.d}->{cfg.hidden}->{cfg.d} tanh-GELU, {cfg.page_bytes // MiB} MiB pages, "
                f"{args.arena_mib} MiB arena per GPU, weights streamed from pinned host, "
                f"columns all-gathered between phases")
    if w in ("block", "stack"):
        cfg = psi_synth.BLOCK
        blocks = 1 if w == "block" else args.blocks
        slots = args.arena_mib * MiB // cfg.page_bytes
        journal = w == "stack" and args.journal
        branches = args.branches if w == "stack" else 1
        return (("pre-norm (RMSNorm, split RoPE on Q/K) " if args.prenorm else "") +
                f"synthetic transformer block x{blocks}: d_model {cfg.d}, {cfg.N} tokens, "
                f"{cfg.heads} heads x {cfg.dh}, QKV {cfg.qkv_rows}x{cfg.d} + out "
                f"{cfg.d}x{cfg.d} + FFN {cfg.d}->{cfg.hidden}->{cfg.d} tanh-GELU, "
                f"{cfg.page_bytes // MiB} MiB pages, {args.arena_mib} MiB arena "
                f"({slots} slots), weights "
                f"{'resident' if args.resident else 'streamed from pinned host'}" +
                (f", {branches} branch states" if branches > 1 or journal else "") +
                (" kept in the host journal (3 device state buffers)" if journal else ""))
    if w == "ffn":
        cfg = psi_synth.FFN
        return (f"paged FFN: X {cfg.N}x{cfg.d}, W1 {cfg.h}x{cfg.d}, W2 {cfg.d}x{cfg.h}, "
                f"{cfg.slice}-wide hidden slices, {cfg.slots}-slice arena, streamed")
    if w == "linear":
        cfg = psi_synth.LINEAR
        return (f"single paged linear: X {cfg.N}x{cfg.K}, W {cfg.M}x{cfg.K}, "
                f"{cfg.page_rows}-row pages, {cfg.slots}-page arena (latency-bound)")
    if w == "attention":
        cfg = psi_synth.ATTN
        if args.key_block:
            cfg = dataclasses.replace(cfg, key_block=args.key_block)
        return (f"partitioned attention: Q,K,V {cfg.heads}x{cfg.N}x{cfg.dh}, scale "
                f"1/sqrt({cfg.dh}), key blocks of {cfg.key_block}, FP32 online softmax")
    raise SystemExit(f"unknown workload {w}")


class BlockWorkload(Workload):
    def __init__(self, torch, dev, blocks=1, arena_mib=80, resident=False, prenorm=False,
                 branches=1, journal=False):
        import psi_synth
        from weight_streamed_bf16_gb300.block import BlockRunner, BlockShape, BlockWeights
        from weight_streamed_bf16_gb300.torch_io import Arena, pinned_like
        cfg = psi_synth.BLOCK
        self.torch = torch
        self.prenorm = prenorm
        self.shape = BlockShape(d=cfg.d, N=cfg.N, heads=cfg.heads, dh=cfg.dh,
                                hidden=cfg.hidden, slice=cfg.slice, page_bytes=cfg.page_bytes,
                                prenorm=prenorm, eps=cfg.eps)
        self.blocks = []
        for b in range(blocks):
            w = psi_synth.block_weights(cfg, block=b, device=dev)  # drawn on the GPU
            # projection weights are streamed straight from pinned copies; the
            # FFN weights are packed into a pinned page image by BlockWeights
            w = {k: (pinned_like(v.cpu()) if k in ("Wqkv", "Wo") else
                     (v.cpu() if v.dim() == 2 else v)) for k, v in w.items()}
            if prenorm:
                w["gamma1"], w["gamma2"] = psi_synth.norm_gains(cfg, block=b, device=dev)
            self.blocks.append(BlockWeights(w, self.shape, resident=resident, device=dev))
            del w
        slots = arena_mib * MiB // cfg.page_bytes
        self.arena = Arena(cfg.page_bytes, slots, device=dev)
        self.runner = BlockRunner(self.shape, self.arena, device=dev,
                                  rope=psi_synth.rope_table(cfg.N, cfg.dh) if prenorm else None)
        self.branches = branches
        self.journal = None
        X0 = psi_synth.block_input(cfg, device=dev)
        if branches > 1 or journal:
            # branch r's input: the block input scaled by 2^-r (distinct bytes)
            self.X = torch.stack([X0 * (0.5 ** r) for r in range(branches)])
        else:
            self.X = X0
        self.Y = torch.empty_like(self.X)
        self.tmp = torch.empty_like(X0)
        if journal:
            from weight_streamed_bf16_gb300.torch_io import Journal
            self.journal = Journal(self.arena, cfg.N * cfg.d * 2, 2 * branches)
        self.flags = 1 if resident else 0
        self.flops = float(cfg.flops) * blocks * branches
        self.linear_flops = float(cfg.linear_flops) * blocks * branches
        self.weight_h2d = 0 if resident else cfg.weight_bytes * blocks * branches
        self.name = (("pre-norm (RMSNorm, split RoPE on Q/K) " if prenorm else "") +
                     f"synthetic transformer block x{blocks}: d_model {cfg.d}, {cfg.N} tokens, "
                     f"{cfg.heads} heads x {cfg.dh}, QKV {cfg.qkv_rows}x{cfg.d} + out "
                     f"{cfg.d}x{cfg.d} + FFN {cfg.d}->{cfg.hidden}->{cfg.d} tanh-GELU, "
                     f"{cfg.page_bytes // MiB} MiB pages, {arena_mib} MiB arena "
                     f"({slots} slots), weights {'resident' if resident else 'streamed from pinned host'}" +
                     (f", {branches} branch states" if branches > 1 or journal else "") +
                     (" kept in the host journal (3 device state buffers)" if journal else ""))

    @property
    def stream(self):
        return self.arena.compute

    def step(self, X=None, Y=None, marks=None):
        X = self.X if X is None else X
        Y = self.Y if Y is None else Y
        if self.journal is not None:
            # branch inputs read from X[r], outputs written to Y[r]; every
            # intermediate state lives in the host journal
            self.runner.run_branches(self.blocks, self.journal, self.branches, self.flags,
                                     inputs=[X[r] for r in range(self.branches)],
                                     outputs=[Y[r] for r in range(self.branches)])
        elif X.dim() == 3:
            for r in range(X.shape[0]):
                self.runner.stack(X[r], self.blocks, Y[r], self.tmp, self.flags)
        elif len(self.blocks) == 1:
            self.runner.forward(X, self.blocks[0], Y, self.flags, marks)
        else:
            self.runner.stack(X, self.blocks, Y, self.tmp, self.flags)

    def managed_bytes(self):
        """Device bytes of the block step by the terms of Eq.(1): the page
        arena (W + 2P in the paper's notation, here all slots), live state
        (activations of one step) and bounded workspace; the library itself
        allocates none."""
        r = self.runner
        nb = lambda t: t.numel() * t.element_size()  # noqa: E731
        live = [self.X, self.Y, r.h, r.att, r.x1] + ([r.xn] if r.xn is not None else [])
        if hasattr(r, "states"):
            live += r.states
        work = [r.hid, r.acc, r.attn_ws]
        out = {"arena": self.arena.buf.numel(), "live_state": sum(nb(t) for t in live),
               "workspace": sum(nb(t) for t in work), "library_allocations": 0}
        out["total"] = out["arena"] + out["live_state"] + out["workspace"]
        return out

    @property
    def phase_names(self):
        """Operator phases one step marks (a single block without a journal)."""
        if len(self.blocks) != 1 or self.X.dim() == 3 or self.journal is not None:
            return None
        return (["norm1", "qkv_rope", "attention", "out_proj", "norm2", "ffn"] if self.prenorm
                else ["qkv", "attention", "out_proj", "ffn"])

    def phase_split(self, steps=5):
        """Per-operator time of a single block on the compute stream (ms):
        QKV projection, attention, out-projection, FFN (median of steps)."""
        torch = self.torch
        names = self.phase_names
        if names is None:
            return None
        per = [[] for _ in names]
        for _ in range(steps):
            marks = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
            with torch.cuda.stream(self.stream):
                self.step(marks=marks)
            marks[-1].synchronize()
            for i in range(len(names)):
                per[i].append(marks[i].elapsed_time(marks[i + 1]))
        # median per phase: one step delayed by the host does not skew it
        return {k: sorted(v)[len(v) // 2] for k, v in zip(names, per)}

    def io(self):
        return self.X, self.Y


class ShardedBlockWorkload(Workload):
    """The block split by output columns over the job's ranks (one part per
    GPU): each rank streams its own pages (its heads' Q, K, V rows, its rows
    of Wo, all of U with its rows of V) through its own 80 MiB arena, and
    the attention output, x1 and y are all-gathered by columns between the
    phases (NCCL).  One step is one block forward of the whole job, so the
    algorithmic FLOPs per step are one block's (strong scaling)."""

    def __init__(self, torch, dev, arena_mib=80, dist=None):
        import psi_synth
        from weight_streamed_bf16_gb300.block import BlockShape
        from weight_streamed_bf16_gb300.shard import (ShardBuffers, ShardPlan, ShardRunner,
                                                      ShardWeights)
        from weight_streamed_bf16_gb300.torch_io import Arena
        cfg = psi_synth.BLOCK
        self.torch, self.dist = torch, dist
        world = dist.get_world_size() if dist is not None else 1
        rank = dist.get_rank() if dist is not None else 0
        self.shape = BlockShape(d=cfg.d, N=cfg.N, heads=cfg.heads, dh=cfg.dh,
                                hidden=cfg.hidden, slice=cfg.slice, page_bytes=cfg.page_bytes)
        self.plan = ShardPlan(self.shape, world, rank)
        w = psi_synth.block_weights(cfg, block=0, device=dev)
        w = {k: v.cpu() for k, v in w.items()}
        self.w = ShardWeights(w, self.plan, device=dev)
        del w
        self.arena = Arena(cfg.page_bytes, arena_mib * MiB // cfg.page_bytes, device=dev)
        self.bufs = ShardBuffers(self.shape, device=dev)
        self.runner = ShardRunner(self.plan, self.arena, self.bufs, device=dev,
                                  attn_tail_split=True)
        self.X = psi_synth.block_input(cfg, device=dev)
        self.Y = torch.empty_like(self.X)
        self.flops = float(cfg.flops)
        self.world_factor = 1            # the job does one block per step in total
        self.weight_h2d = self.w.host_bytes
        self.name = (f"synthetic transformer block x1 split by output columns over {world} "
                     f"GPU(s): d_model {cfg.d}, {cfg.N} tokens, {cfg.heads} heads x {cfg.dh}, "
                     f"QKV {cfg.qkv_rows}x{cfg.d} + out {cfg.d}x{cfg.d} + FFN "
                     f"{cfg.d}->{cfg.hidden}->{cfg.d} tanh-GELU, {cfg.page_bytes // MiB} MiB "
                     f"pages, {arena_mib} MiB arena per GPU, weights streamed from pinned host, "
                     f"columns all-gathered between phases")

    @property
    def stream(self):
        return self.arena.compute

    def step(self, X=None, Y=None):
        from weight_streamed_bf16_gb300.shard import forward_parts_in_turn, forward_sharded
        X = self.X if X is None else X
        Y = self.Y if Y is None else Y
        if self.dist is not None:
            forward_sharded(self.runner, X, self.w, Y, 0)
        else:
            forward_parts_in_turn([self.runner], X, [self.w], Y, 0)

    def io(self):
        return self.X, self.Y


class FfnWorkload(Workload):
    def __init__(self, torch, dev):
        import psi_synth
        from weight_streamed_bf16_gb300.torch_io import Arena, FfnWeight, ffn_workspace
        cfg = psi_synth.FFN
        self.cfg = cfg
        X, U, V, a, b = psi_synth.ffn_inputs(cfg)
        self.w = FfnWeight(U, V, cfg.slice)
        self.arena = Arena(cfg.page_bytes, cfg.slots, device=dev)
        self.X, self.a, self.b = X.to(dev), a.to(dev), b.to(dev)
        self.Y = torch.empty(cfg.N, cfg.r, dtype=torch.bfloat16, device=dev)
        self.hid, self.acc = ffn_workspace(cfg.N, cfg.r, cfg.slice, dev)
        self.flops = float(cfg.flops)
        self.weight_h2d = (cfg.h // cfg.slice) * cfg.page_bytes
        self.name = (f"paged FFN: X {cfg.N}x{cfg.d}, W1 {cfg.h}x{cfg.d}, W2 {cfg.d}x{cfg.h}, "
                     f"{cfg.slice}-wide hidden slices, {cfg.slots}-slice arena, streamed")

    @property
    def stream(self):
        return self.arena.compute

    def step(self, X=None, Y=None):
        from weight_streamed_bf16_gb300 import psi
        X = self.X if X is None else X
        Y = self.Y if Y is None else Y
        psi.psi_ffn_paged(self.arena.handle, X.data_ptr(), self.cfg.N, self.w.desc(),
                          self.a.data_ptr(), self.b.data_ptr(), self.hid.data_ptr(),
                          self.acc.data_ptr(), None, Y.data_ptr(), 0)

    def io(self):
        return self.X, self.Y


class LinearWorkload(Workload):
    def __init__(self, torch, dev):
        import psi_synth
        from weight_streamed_bf16_gb300.torch_io import Arena, LinearWeight
        cfg = psi_synth.LINEAR
        self.cfg = cfg
        X, W, b = psi_synth.linear_inputs(cfg)
        self.w = LinearWeight(W, cfg.page_bytes, page_rows=cfg.page_rows)
        self.arena = Arena(cfg.page_bytes, cfg.slots, device=dev)
        self.X, self.b = X.to(dev), b.to(dev)
        self.Y = torch.empty(cfg.N, cfg.M, dtype=torch.bfloat16, device=dev)
        self.flops = float(cfg.flops)
        self.weight_h2d = cfg.M * cfg.K * 2
        self.name = (f"single paged linear: X {cfg.N}x{cfg.K}, W {cfg.M}x{cfg.K}, "
                     f"{cfg.page_rows}-row pages, {cfg.slots}-page arena (latency-bound)")

    @property
    def stream(self):
        return self.arena.compute

    def step(self, X=None, Y=None):
        from weight_streamed_bf16_gb300 import psi
        X = self.X if X is None else X
        Y = self.Y if Y is None else Y
        psi.psi_linear_paged(self.arena.handle, X.data_ptr(), self.cfg.N, self.cfg.K,
                             self.w.desc(), self.b.data_ptr(), None, Y.data_ptr(), self.cfg.M, 0)

    def io(self):
        return self.X, self.Y


class AttentionWorkload(Workload):
    timed_alone = True

    def __init__(self, torch, dev, key_block=None):
        import dataclasses

        import psi_synth
        cfg = psi_synth.ATTN
        if key_block:
            cfg = dataclasses.replace(cfg, key_block=key_block)
        self.cfg = cfg
        self.torch = torch
        self.Q, self.K, self.V = psi_synth.attn_inputs(cfg, device=dev)
        self.O = torch.empty_like(self.Q)
        from weight_streamed_bf16_gb300 import psi
        nws = psi.psi_attn_workspace_size(cfg.key_block)
        self.ws = torch.empty(nws // 4, dtype=torch.float32, device=dev)
        self._stream = torch.cuda.current_stream(dev)
        self.flops = float(cfg.flops)
        self.weight_h2d = 0
        self.name = (f"partitioned attention: Q,K,V {cfg.heads}x{cfg.N}x{cfg.dh}, scale "
                     f"1/sqrt({cfg.dh}), key blocks of {cfg.key_block}, FP32 online softmax")

    @property
    def stream(self):
        return self._stream

    def step(self, X=None, Y=None):
        from weight_streamed_bf16_gb300 import psi
        from weight_streamed_bf16_gb300.torch_io import heads_view
        Q = self.Q if X is None else X
        O = self.O if Y is None else Y
        psi.psi_attn_partitioned_ws(heads_view(Q), heads_view(self.K), heads_view(self.V),
                                    heads_view(O), self.cfg.heads, self.cfg.N, self.cfg.N,
                                    self.cfg.dh, self.cfg.scale, self.cfg.key_block,
                                    self.ws.data_ptr(), self.ws.numel() * 4,
                                    self._stream.cuda_stream, 0)

    def io(self):
        return self.Q, self.O


def stack_sweep_runs(torch, dev, blocks: int, steps: int):
    """The stack configuration's transport control: one stack of `blocks`
    blocks (weights in pinned host memory, plus a device-resident copy) run
    streamed through arenas of 32, 80 and 256 MiB, resident, and streamed
    with the copies on the compute stream (no prefetch: the scheduling
    comparison of Table IV); the arena sweep is the Table V analog.  Each
    run times `steps` stacks after one warm-up stack with one event pair
    over all of them (a stack moves 19 GB of weights, far more than L2),
    and compares its output with the first run's bit for bit."""
    from weight_streamed_bf16_gb300 import psi
    from weight_streamed_bf16_gb300.block import BlockRunner
    from weight_streamed_bf16_gb300.torch_io import Arena
    t0 = time.perf_counter()
    wl = BlockWorkload(torch, dev, blocks, 80, resident=True)
    setup_s = time.perf_counter() - t0
    wl.arena.close()
    runs = []
    ref = None
    for mib, flags in [(32, 0), (80, 0), (256, 0), (80, psi.PSI_RESIDENT),
                       (80, psi.PSI_SYNC_COPY)]:
        arena = Arena(wl.shape.page_bytes, mib * MiB // wl.shape.page_bytes, device=dev)
        runner = BlockRunner(wl.shape, arena, device=dev)
        Y = torch.empty_like(wl.X)
        tmp = torch.empty_like(wl.X)
        with torch.cuda.stream(arena.compute):
            runner.stack(wl.X, wl.blocks, Y, tmp, flags)           # warm-up
        arena.sync(600000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(arena.compute):
            e0.record(arena.compute)
            for _ in range(steps):
                runner.stack(wl.X, wl.blocks, Y, tmp, flags)
            e1.record(arena.compute)
        arena.sync(600000)
        ms = e0.elapsed_time(e1) / steps
        st = arena.stats()
        same = None
        if ref is None:
            ref = Y.clone()
        else:
            same = bool(torch.equal(ref.view(torch.int16), Y.view(torch.int16)))
        runs.append({"arena_mib": mib, "slots": arena.slots,
                     "mode": ("resident" if flags & psi.PSI_RESIDENT else
                              "streamed, copies on the compute stream" if flags else "streamed"),
                     "ms_per_stack": ms, "tflops": wl.flops / (ms * 1e-3) / 1e12,
                     "ingest_gbs": (0 if flags & psi.PSI_RESIDENT else
                                    len(wl.blocks) * psi_weight_bytes()) /
                                   (ms * 1e-3) / 1e9,
                     "bitwise_equal_to_first": same, "pages": st["pages_streamed"]})
        arena.close()
        del runner, Y, tmp
    out = {"workload": f"stack of {blocks} synthetic blocks ({len(wl.blocks) * psi_weight_bytes()} "
                       f"bytes of weights in pinned host memory), transport control",
           "stacks_per_run": steps, "runs": runs, "setup_s": setup_s,
           "all_bitwise_equal": all(r["bitwise_equal_to_first"] in (None, True) for r in runs)}
    del wl
    torch.cuda.empty_cache()
    return out


def stack_sweep(args):
    """--sweep: the stack transport control alone, as its own JSON line."""
    import torch
    from weight_streamed_bf16_gb300 import build, psi
    build.build()
    psi.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    link_gbs = h2d_probe(torch, dev)
    out = stack_sweep_runs(torch, dev, args.blocks, args.steps)
    out.update({"metric": METRIC, "unit": "TFLOP/s", "steps": args.steps,
                "link_probe_gbs": link_gbs, "peaks": peaks})
    print(json.dumps(out))
    return 0


def time_config(torch, wl, flush, steps: int, warmup: int = 3):
    """One of the other configurations timed as the headline is: warm-up
    iterations of the timed body, then `steps` steps each after an L2 flush,
    one event pair over the loop and one per step; the whole loop when the
    workload streams weights, else the sum of the steps."""
    s = wl.stream
    n = warmup + steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for i in range(n):
            if i == warmup:
                l0.record(s)
            flush.fill_(i & 0xFF)
            ev[i][0].record(s)
            wl.step()
            ev[i][1].record(s)
        l1.record(s)
    torch.cuda.synchronize()
    step_sum = sum(a.elapsed_time(b) for a, b in ev[warmup:]) / steps
    loop = l0.elapsed_time(l1) / steps
    ms = loop if wl.weight_h2d else step_sum
    return {"workload": wl.name, "ms_per_step": ms,
            "ms_per_step_from": "whole loop" if wl.weight_h2d else "sum of steps",
            "tflops": wl.flops / (ms * 1e-3) / 1e12,
            "weight_gbs": wl.weight_h2d / (ms * 1e-3) / 1e9 if wl.weight_h2d else 0.0}


def other_configs(torch, dev, flush, peaks, link_gbs, steps: int, stack_blocks: int):
    """The other four configurations of the study, for the same JSON line:
    the single paged linear (latency-bound), the paged FFN (bound by its
    weight copies), partitioned attention with key blocks of 256 (tensor
    cores, burst peak) and the stack's transport control."""
    out = {}
    lw = LinearWorkload(torch, dev)
    out["linear"] = time_config(torch, lw, flush, steps)
    out["linear"]["bound"] = "latency (8 page launches, 8 copies of 64 KiB)"
    lw.arena.close()
    fw = FfnWorkload(torch, dev)
    r = time_config(torch, fw, flush, steps)
    r.update({"bound": "host link", "frac_of_link": r["weight_gbs"] / link_gbs,
              "link_probe_gbs": link_gbs})
    out["ffn"] = r
    fw.arena.close()
    aw = AttentionWorkload(torch, dev)
    r = time_config(torch, aw, flush, steps)
    r.update({"bound": "tensor", "frac_of_burst_peak": r["tflops"] / peaks["bf16_tflops"]})
    out["attention"] = r
    del aw
    if stack_blocks > 0:
        out["stack"] = stack_sweep_runs(torch, dev, stack_blocks, 1)
    return out


def psi_weight_bytes():
    import psi_synth
    return psi_synth.BLOCK.weight_bytes


def make_workload(torch, dev, args, dist=None):
    if args.shard:
        if args.workload != "block":
            raise SystemExit("--shard applies to the block workload")
        return ShardedBlockWorkload(torch, dev, args.arena_mib, dist)
    if args.workload == "block":
        return BlockWorkload(torch, dev, 1, args.arena_mib, args.resident, args.prenorm)
    if args.workload == "stack":
        return BlockWorkload(torch, dev, args.blocks, args.arena_mib, args.resident, args.prenorm,
                             args.branches, args.journal)
    if args.workload == "ffn":
        return FfnWorkload(torch, dev)
    if args.workload == "linear":
        return LinearWorkload(torch, dev)
    if args.workload == "attention":
        return AttentionWorkload(torch, dev, args.key_block)
    raise SystemExit(f"unknown workload {args.workload}")


# ------------------------------------------------------------ CPU oracle --
class OracleSample:
    """The CPU oracle on a bounded sample of a workload.  Inputs are drawn
    once (untimed); ``run(rows)`` times the oracle on `rows` token (query)
    rows of every operator and returns (algorithmic FLOPs, seconds, text)."""

    def __init__(self, workload: str):
        import numpy as np
        import torch

        import psi_synth
        from oracle import bf16

        def f64(t):
            return bf16.decode(t.contiguous().view(torch.int16).numpy().view(np.uint16))

        self.workload = workload
        self.np = np
        if workload in ("block", "stack"):
            cfg = psi_synth.BLOCK
            w = psi_synth.block_weights(cfg, block=0)
            self.cfg = cfg
            self.w = {k: f64(v) for k, v in w.items()}
            self.X = f64(psi_synth.normal_bf16((1024, cfg.d), 1.0, cfg.seed, 90001))
            self.KV = f64(psi_synth.normal_bf16((2, cfg.N, cfg.dh), 1.0, cfg.seed, 90002))
        elif workload == "ffn":
            cfg = psi_synth.FFN
            self.cfg = cfg
            self.t = [f64(t) for t in psi_synth.ffn_inputs(cfg)]
        elif workload == "linear":
            cfg = psi_synth.LINEAR
            self.cfg = cfg
            self.t = [f64(t) for t in psi_synth.linear_inputs(cfg)]
        else:
            cfg = psi_synth.ATTN
            self.cfg = cfg
            self.t = [f64(t) for t in psi_synth.attn_inputs(cfg)]

    def run(self, rows: int):
        from oracle import ops
        np, cfg = self.np, self.cfg
        fl = 0.0
        t0 = time.perf_counter()
        if self.workload in ("block", "stack"):
            w = self.w
            rows = min(rows, self.X.shape[0])
            X = self.X[:rows]
            h = ops.linear(X, w["Wqkv"], w["bqkv"]).y
            fl += 2.0 * rows * cfg.d * cfg.qkv_rows
            att = np.empty((rows, cfg.heads * cfg.dh))
            for hd in range(cfg.heads):
                q = h[:, hd * cfg.dh:(hd + 1) * cfg.dh]
                att[:, hd * cfg.dh:(hd + 1) * cfg.dh] = ops.attention(
                    q, self.KV[0], self.KV[1], 1 / math.sqrt(cfg.dh)).y
            fl += 4.0 * rows * cfg.N * cfg.dh * cfg.heads
            x1 = ops.linear(att, w["Wo"], w["bo"], residual=X).y
            fl += 2.0 * rows * cfg.d * cfg.d
            ops.ffn(x1, w["W1"], w["W2"], w["a1"], w["b1"], residual=x1)
            fl += 4.0 * rows * cfg.d * cfg.hidden
            desc = (f"oracle on {rows} token rows of every block operator (QKV, attention of "
                    f"all {cfg.heads} heads against {cfg.N} keys, out-proj, FFN), float64 numpy")
        elif self.workload == "ffn":
            X, U, V, a, b = self.t
            rows = min(rows, X.shape[0])
            ops.ffn(X[:rows], U, V, a, b)
            fl = 4.0 * rows * cfg.d * cfg.h
            desc = f"oracle FFN on {rows} of {cfg.N} token rows"
        elif self.workload == "linear":
            X, W, b = self.t
            n = 0
            while time.perf_counter() - t0 < 1.0:
                ops.linear(X, W, b)
                n += 1
            fl = float(cfg.flops) * n
            desc = f"oracle linear, whole configuration, {n} repetitions"
        else:
            Q, K, V = self.t
            rows = min(rows, Q.shape[1])
            for hd in range(cfg.heads):
                ops.attention(Q[hd, :rows], K[hd], V[hd], cfg.scale)
            fl = 4.0 * cfg.heads * rows * cfg.N * cfg.dh
            desc = f"oracle attention on {rows} of {cfg.N} query rows of all {cfg.heads} heads"
        return fl, time.perf_counter() - t0, desc


def reference_arm(args):
    """--impl reference: the oracle timed on the host cores (rank 0 only)."""
    rank, world, _ = env_rank()
    if rank != 0:
        return 0
    rows = {"block": 64, "stack": 64, "ffn": 64, "linear": 0, "attention": 16}[args.workload]
    sample = OracleSample(args.workload)
    for _ in range(args.warmup):
        sample.run(max(1, rows // 8))
    tot_fl, tot_s, desc = 0.0, 0.0, ""
    for _ in range(args.steps):
        fl, sec, desc = sample.run(rows)
        tot_fl += fl
        tot_s += sec
    v = tot_fl / tot_s / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_s / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(args), "sample": desc},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))
    return 0


# ------------------------------------------------------------------- main --
def busy_ms(records, kind, lo, hi):
    """Length of the union of the `kind` records' intervals clipped to
    [lo, hi] (records of the page trace, times in ms)."""
    iv = sorted((max(r["start_ms"], lo), min(r["end_ms"], hi)) for r in records
                if r["kind"] == kind and r["end_ms"] > lo and r["start_ms"] < hi)
    tot, end = 0.0, -1e300
    for a, b in iv:
        if b > end:
            tot += b - max(a, end)
            end = b
    return tot


def write_trace(path, wl, arena, stream, flush, torch):
    """Page timeline of two steps after the measured ones (not timed): one
    record per page copy and page GEMM from the library, the operator phase
    marks of each step where the workload has them, and per-step sums of
    copy and GEMM busy time.  Written to `path`; nothing is printed."""
    from weight_streamed_bf16_gb300 import psi
    origin = torch.cuda.Event(enable_timing=True)
    origin.record(stream)          # creates the event (torch creates it on first record)
    arena.sync()
    torch.cuda.synchronize()
    # The library's origin and this one are recorded behind a short device
    # delay on the same stream, so both take the timestamp of its end; on an
    # idle stream each would take the host time of its record call, and
    # marks and page records would be offset by the host time in between.
    with torch.cuda.stream(stream):
        torch.cuda._sleep(1 << 21)
    psi.psi_arena_trace_begin(arena.handle, 1 << 14)
    origin.record(stream)
    names = getattr(wl, "phase_names", None)
    marks = []
    with torch.cuda.stream(stream):
        for k in range(2):
            flush.fill_(k & 0xFF)
            if names:
                m = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
                wl.step(marks=m)
                marks.append(m)
            else:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                wl.step()
                e1.record(stream)
                marks.append([e0, e1])
    arena.sync()
    torch.cuda.synchronize()
    rec = psi.psi_arena_trace_get(arena.handle)
    psi.psi_arena_set_timing(arena.handle, False)
    steps = []
    for m in marks:
        t = [origin.elapsed_time(e) for e in m]
        lo, hi = t[0], t[-1]

        steps.append({"start_ms": lo, "end_ms": hi,
                      "phases": ({n: [t[i], t[i + 1]] for i, n in enumerate(names)}
                                 if names else None),
                      "copy_busy_ms": busy_ms(rec, "copy", lo, hi),
                      "gemm_busy_ms": busy_ms(rec, "gemm", lo, hi)})
    with open(path, "w") as f:
        json.dump({"workload": wl.name, "steps": steps, "records": rec}, f)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="psi", choices=["psi", "reference"])
    ap.add_argument("--workload", default="block",
                    choices=["block", "stack", "ffn", "linear", "attention"])
    ap.add_argument("--blocks", type=int, default=48, help="stack depth (workload stack)")
    ap.add_argument("--arena-mib", type=int, default=80)
    ap.add_argument("--resident", action="store_true", help="weights resident (no streaming)")
    ap.add_argument("--key-block", type=int, default=None,
                    help="attention workload: keys per online-softmax block (default 256)")
    ap.add_argument("--prenorm", action="store_true",
                    help="block/stack: pre-norm block (RMSNorm before QKV and FFN, split RoPE)")
    ap.add_argument("--branches", type=int, default=1,
                    help="stack: independent branch states run through every block")
    ap.add_argument("--journal", action="store_true",
                    help="stack: keep branch states in the host journal (3 device buffers)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="stack workload: arena sweep 32/80/256 MiB + resident, bitwise control")
    ap.add_argument("--cpu-rows", type=int, default=1024,
                    help="token (query) rows of the oracle sample for cpu_baseline "
                         "(the block sample holds 1024)")
    ap.add_argument("--no-configs", action="store_true",
                    help="block: skip the other configurations (linear, FFN, attention, "
                         "stack transport control) after the headline measurement")
    ap.add_argument("--stack-blocks", type=int, default=48,
                    help="blocks of the stack in the default line's transport control "
                         "(0: none)")
    ap.add_argument("--shard", action="store_true",
                    help="block: split every operator by output columns over the ranks "
                         "(NCCL column gathers between phases; strong scaling) instead of "
                         "running one independent block per rank")
    ap.add_argument("--trace", default=None, metavar="PATH",
                    help="after the measurements, write the page timeline of two more "
                         "steps (copies, page GEMMs, phase marks) to PATH as JSON")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.impl == "reference":
        return reference_arm(args)
    if args.sweep:
        return stack_sweep(args)

    import torch
    rank, world, local = env_rank()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    from weight_streamed_bf16_gb300 import build, psi
    build.build()
    psi.load()

    peaks = load_peaks()
    link_gbs = h2d_probe(torch, dev)
    link2_gbs = h2d_probe(torch, dev, streams=2)
    link4_gbs = h2d_probe(torch, dev, streams=4)
    wl = make_workload(torch, dev, args, dist)
    stream = wl.stream
    arena = getattr(wl, "arena", None)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed_loop(n, ev, loop0=None, loop1=None):
        """n steps, each after an L2 flush (a write larger than L2) and
        bracketed by its own event pair; loop0/loop1 span the whole loop."""
        with torch.cuda.stream(stream):
            if loop0 is not None:
                loop0.record(stream)
            for i in range(n):
                flush.fill_(i & 0xFF)
                ev[i][0].record(stream)
                wl.step()
                ev[i][1].record(stream)
            if loop1 is not None:
                loop1.record(stream)

    # warm-up: the timed loop's own body (the first pass through it is
    # slower on the host than the ones after it)
    warm = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.warmup)]
    timed_loop(args.warmup, warm)
    barrier()
    j0 = wl.journal.stats() if getattr(wl, "journal", None) is not None else None
    k0 = psi.psi_kernel_launches()

    # ------------------------------------------------ device-timed region --
    # One event pair spans the whole loop, the L2 flushes between steps
    # included: ms_per_step = that time / steps, so every copy and kernel of
    # every step is inside the interval (a step's first page copies can
    # start during the flush before it).  The per-step pairs give the sum
    # without the flushes.  No per-launch timing inside the library here
    # (its event pairs around every page GEMM and copy cost about 5 % of the
    # step); it is taken in a separate pass below.
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    clocks = ClockSampler(gpu_id)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    loop0, loop1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    clocks.start()
    t_wall = time.perf_counter()
    timed_loop(args.steps, ev, loop0, loop1)
    barrier()
    k1 = psi.psi_kernel_launches()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    step_sum_ms = sum(step_ms)
    loop_ms = loop0.elapsed_time(loop1)
    # with streamed weights a step's first page copies may start before its
    # start event (during the flush), so the whole loop is the honest time;
    # without a copy stream every operation of a step lies between its two
    # events and the per-step sum leaves out only the flushes
    timing = "whole loop" if wl.weight_h2d else "sum of steps"
    total_ms = loop_ms if wl.weight_h2d else step_sum_ms
    # the same steps again with the library's per-launch event pairs, for the
    # in-step page-GEMM and copy figures (not for `value`)
    st = None
    timed_ms = None
    if arena is not None:
        psi.psi_arena_reset_stats(arena.handle)
        psi.psi_arena_set_timing(arena.handle, True)
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        timed_loop(args.steps, ev2)
        barrier()
        timed_ms = sum(a.elapsed_time(b) for a, b in ev2) / args.steps
        st = psi.psi_arena_stats(arena.handle)
        psi.psi_arena_set_timing(arena.handle, False)
    jst = None
    if getattr(wl, "journal", None) is not None:
        js = wl.journal.stats()
        jst = {k: (js[k] - j0[k]) / args.steps
               for k in ("commits", "reloads", "d2h_bytes", "h2d_bytes", "host_waits",
                         "hazard_waits")}
        jst["per"] = "step"
        js = {k: js[k] - j0[k] for k in ("d2h_bytes", "h2d_bytes")}
        jst["d2h_gbs_per_step_time"] = js["d2h_bytes"] / (total_ms * 1e-3) / 1e9
        jst["h2d_gbs_per_step_time"] = js["h2d_bytes"] / (total_ms * 1e-3) / 1e9
    # the library's own count of the kernels it launched in the timed region
    gpu_launches = k1 - k0
    wf = getattr(wl, "world_factor", world)  # ranks whose work a step counts
    total_ms, ms_per_step, value = aggregate_ranks(dist, dev, total_ms, wl.flops, args.steps,
                                                   world, wf)

    phases = wl.phase_split() if hasattr(wl, "phase_split") else None

    # ------------------------------------------------------------ e2e ---
    # Every step moves its input X from pinned host memory and its output Y
    # back, through the same public calls.  The copies run on their own
    # streams with two device buffers each, so step k's D2H overlaps step
    # k+1 (the other link direction) and step k+1's H2D overlaps step k;
    # every dependency is an event.  The region runs from the first H2D to
    # the last D2H; L2 is flushed before every step, as in the device-timed
    # region.
    Xd, Yd = wl.io()
    Xh = torch.empty(Xd.shape, dtype=Xd.dtype, pin_memory=True)
    Xh.copy_(Xd)
    Yh = torch.empty(Yd.shape, dtype=Yd.dtype, pin_memory=True)
    Xe = [torch.empty_like(Xd) for _ in range(2)]
    Ye = [torch.empty_like(Yd) for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(n, t0=None, t1=None):
        ev = lambda: torch.cuda.Event()  # noqa: E731
        step_done, out_done = [], []
        if t0 is not None:
            t0.record(h2d_s)
        for k in range(n):
            b = k & 1
            if k >= 2:
                h2d_s.wait_event(step_done[k - 2])   # step k-2 has read Xe[b]
            with torch.cuda.stream(h2d_s):
                Xe[b].copy_(Xh, non_blocking=True)
            e_in = ev()
            e_in.record(h2d_s)
            stream.wait_event(e_in)
            if k >= 2:
                stream.wait_event(out_done[k - 2])   # Ye[b] has been read back
            with torch.cuda.stream(stream):
                flush.fill_(k & 0xFF)
                wl.step(Xe[b], Ye[b])
            e_s = ev()
            e_s.record(stream)
            step_done.append(e_s)
            d2h_s.wait_event(e_s)
            with torch.cuda.stream(d2h_s):
                Yh.copy_(Ye[b], non_blocking=True)
            e_o = ev()
            e_o.record(d2h_s)
            out_done.append(e_o)
        if t1 is not None:
            d2h_s.wait_event(step_done[-1])
            t1.record(d2h_s)

    e2e_run(max(3, args.warmup))
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(args.steps, t0, t1)
    barrier()
    e2e_ms = t0.elapsed_time(t1)
    e2e_ms, _, e2e_value = aggregate_ranks(dist, dev, e2e_ms, wl.flops, args.steps, world, wf)
    in_bytes = Xh.numel() * Xh.element_size()
    out_bytes = Yh.numel() * Yh.element_size()

    if args.trace and arena is not None and rank == 0:
        write_trace(args.trace, wl, arena, stream, flush, torch)

    # ------------------------------------------------ roofline (page GEMM) --
    digest = source_digest("page_gemm.cu", "page_gemm_pair.cu", "gemm_epilogue.cuh", "ptx.cuh")
    roof = None
    peak_s = peaks["bf16_tflops_sustained"]
    if st and st["timed_gemms"]:
        avg_ms = st["gemm_ms"] / st["timed_gemms"]
        fl_launch = st["gemm_flops"] / st["timed_gemms"]
        ach = fl_launch / (avg_ms * 1e-3) / 1e12
        busy = st["gemm_flops"] / (st["gemm_busy_ms"] * 1e-3) / 1e12 if st["gemm_busy_ms"] else None
        in_step = {
            "achieved": ach, "peak": peak_s, "unit": "TFLOP/s", "frac": ach / peak_s,
            "peak_kind": f"sustained bf16, of {peaks['source']}",
            "launches": st["timed_gemms"], "avg_launch_ms": avg_ms,
            "flops_per_launch": fl_launch,
            # consecutive page GEMMs overlap on two streams, which stretches
            # each launch's event interval; FLOPs over the union of the
            # intervals is the throughput while any page GEMM runs
            "achieved_busy": busy, "frac_busy": busy / peak_s if busy else None,
            "ms_per_step_with_launch_events": timed_ms}
        roof = {"kernel": "page_gemm (tcgen05, all epilogues)", "bound": "tensor",
                "in_step": in_step}
        if isinstance(wl, BlockWorkload):
            # the compute-bound figure: one resident QKV page timed alone
            ga = gemm_alone(torch, dev, wl, peaks, flush)
            pg = ga["page"]
            roof.update({"achieved": pg["achieved"], "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": pg["frac"],
                         "peak_kind": f"burst bf16, of {peaks['source']}",
                         "measured": "one resident 6144x2048x4096 QKV page launch per event "
                                     "pair, L2 flushed before each (median of 20)",
                         "avg_launch_ms": pg["ms"], "flops_per_launch": pg["flops"],
                         "qkv_resident": ga["qkv_resident"],
                         "cublas_same_shape": ga["cublas_same_shape"],
                         "traffic": profile_traffic("page_gemm_block_traffic.txt", digest)})
        else:
            roof.update({k: in_step[k] for k in ("achieved", "peak", "unit", "frac",
                                                 "peak_kind", "avg_launch_ms",
                                                 "flops_per_launch")})
            roof["traffic"] = None
    elif isinstance(wl, AttentionWorkload):
        ach = wl.flops / (ms_per_step * 1e-3) / 1e12
        roof = {"kernel": "attn_partitioned (tcgen05)", "bound": "tensor", "achieved": ach,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16_tflops"],
                "peak_kind": f"burst bf16, of {peaks['source']}",
                "traffic": profile_traffic("attention_traffic.txt",
                                           source_digest("attention.cu", "ptx.cuh"))}

    norm_roof = None
    if getattr(wl, "prenorm", False) and wl.X.dim() == 2:
        # the RMSNorm kernel timed alone: rounds of four back-to-back launches
        # on four input/output pairs (400 MB together, so each launch reads
        # X from DRAM: the other three evicted it from L2), one event pair per
        # round, so launch latency overlaps the previous launch as in a step;
        # and, for reference, single launches with L2 flushed before each.
        # Algorithmic bytes = read X + write Y + gamma.
        import psi_synth
        c = psi_synth.BLOCK
        nb = 2 * c.N * c.d * 2 + 2 * c.d
        r = wl.runner
        gam = wl.blocks[0].gamma1.data_ptr()
        xs = [wl.X] + [torch.randn(c.N, c.d, device=dev).to(torch.bfloat16) for _ in range(3)]
        ys = [torch.empty_like(wl.X) for _ in range(4)]

        def norm(i):
            psi.psi_rmsnorm(xs[i].data_ptr(), c.d, c.N, c.d, gam, c.eps, ys[i].data_ptr(), c.d,
                            stream.cuda_stream)
        rounds = 10
        with torch.cuda.stream(stream):
            for i in range(4):
                norm(i)                           # warm-up
            evr = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(rounds)]
            for e0, e1 in evr:
                e0.record(stream)
                for i in range(4):
                    norm(i)
                e1.record(stream)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(rounds)]
            for e0, e1 in evs:
                flush.fill_(1)
                e0.record(stream)
                norm(0)
                e1.record(stream)
        evs[-1][1].synchronize()
        us = sum(a.elapsed_time(b) for a, b in evr) * 1e3 / (4 * rounds)
        us1 = sum(a.elapsed_time(b) for a, b in evs) * 1e3 / rounds
        g = nb / (us * 1e-6) / 1e9
        norm_roof = {"kernel": "rmsnorm", "bound": "hbm", "avg_launch_us": us, "achieved": g,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": g / peaks["hbm_gbs"],
                     "bytes_per_launch": nb, "single_launch_us": us1,
                     "timing": "rounds of 4 back-to-back launches on 4 inputs (400 MB > L2)"}
        del xs, ys

    ingest = None
    if st and st["timed_copies"]:
        ce = st["copy_bytes"] / (st["copy_ms"] * 1e-3) / 1e9
        eff = wl.weight_h2d / (ms_per_step * 1e-3) / 1e9
        ce_busy = (st["copy_bytes"] / (st["copy_busy_ms"] * 1e-3) / 1e9
                   if st["copy_busy_ms"] else None)
        ingest = {"unit": "GB/s", "copy_engine_gbs": ce, "copy_busy_gbs": ce_busy,
                  "effective_gbs": eff,
                  "link_probe_gbs": link_gbs, "copy_frac_of_link": ce / link_gbs,
                  "link_probe_two_streams_gbs": link2_gbs,
                  "link_probe_four_streams_gbs": link4_gbs,
                  "weight_bytes_per_step": wl.weight_h2d,
                  "pages_per_step": st["pages_streamed"] / args.steps}
        if isinstance(wl, BlockWorkload):
            # the transfer-bound figure: the streamed FFN configuration
            ingest["transfer_bound"] = ingest_alone(torch, dev, link_gbs, flush)
    step_bound_ms = max(wl.flops / (peaks["bf16_tflops_sustained"] * 1e12),
                        wl.weight_h2d / (link_gbs * 1e9)) * 1e3

    configs = None
    if (rank == 0 and world == 1 and args.workload == "block" and not args.shard and
            not args.prenorm and not args.resident and not args.no_configs):
        # the study's other configurations, measured after the headline's
        # timed region (they do not enter `value`)
        configs = other_configs(torch, dev, flush, peaks, link_gbs, 10, args.stack_blocks)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        fl, sec, desc = OracleSample(args.workload).run(args.cpu_rows)
        cpu = {"value": fl / sec / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
               "kind": "oracle", "sample": desc, "seconds": sec}

    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "strong" if args.shard else "weak",
            "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded, N(0,1/fan_in) weights)",
            "config": {"workload": wl.name, "l2": "flushed between steps (256 MiB write)",
                       "parallelism": (f"output columns x{world}" if args.shard else
                                       f"replicas x{world}" if world > 1 else "single GPU"),
                       "flops_per_step": wl.flops, "wall_s_timed": t_wall,
                       # the sum of the per-step event pairs (flushes
                       # excluded) and the whole timed loop (one event pair,
                       # flushes included), each over the steps
                       "step_sum_ms_per_step": step_sum_ms / args.steps,
                       "loop_ms_per_step": loop_ms / args.steps,
                       "ms_per_step_from": timing,
                       "step_roofline_ms": step_bound_ms,
                       "phase_ms": phases, "rmsnorm_roofline": norm_roof,
                       "managed_device_bytes": (wl.managed_bytes()
                                                if hasattr(wl, "managed_bytes") else None),
                       "frac_of_step_roofline": step_bound_ms / ms_per_step},
            "roofline": roof, "ingest": ingest, "journal": jst, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step":
                    in_bytes + wl.weight_h2d, "d2h_bytes_per_step": out_bytes,
                    "ms_per_step": e2e_ms / args.steps},
            "gpu_launches": gpu_launches, "clocks": clk,
            "peaks": peaks, "configs": configs,
        }
        print(json.dumps(out))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
