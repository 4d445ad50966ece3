"""The N > 1 host path of bench.py on CPU: two gloo ranks run independent
replicas (no data-path collective) and the job time is the maximum over
ranks; the job value counts every rank's work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r took 10 * (r + 1) ms for 5 steps of 2 TFLOP each
    total, per_step, value = bench.aggregate_ranks(dist, torch.device("cpu"),
                                                   10.0 * (rank + 1), 2e12, 5, world)
    out[rank] = (total, per_step, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_max_time_and_weak_scaling_value():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    for r in range(2):
        total, per_step, value = out[r]
        assert total == 20.0                 # the slower rank's time
        assert per_step == 4.0
        assert value == pytest.approx(2 * 2e12 / 4e-3 / 1e12)   # both ranks' work


def test_single_rank_needs_no_process_group():
    import bench
    total, per_step, value = bench.aggregate_ranks(None, torch.device("cpu"), 8.0, 1e12, 4, 1)
    assert (total, per_step) == (8.0, 2.0)
    assert value == pytest.approx(1e12 / 2e-3 / 1e12)


def test_trace_busy_time_is_the_union_of_intervals():
    """The page-timeline summary counts overlapping records once and clips
    them to the step."""
    import bench
    rec = [{"kind": "copy", "start_ms": 0.0, "end_ms": 1.0},
           {"kind": "copy", "start_ms": 0.5, "end_ms": 1.5},    # overlaps the first
           {"kind": "copy", "start_ms": 2.0, "end_ms": 2.25},
           {"kind": "gemm", "start_ms": 0.0, "end_ms": 9.0},
           {"kind": "copy", "start_ms": 2.9, "end_ms": 3.4}]    # clipped at 3.0
    assert abs(bench.busy_ms(rec, "copy", 0.0, 3.0) - 1.85) < 1e-12
    assert abs(bench.busy_ms(rec, "copy", 0.75, 3.0) - (0.75 + 0.25 + 0.1)) < 1e-12
    assert bench.busy_ms(rec, "gemm", 1.0, 2.0) == 1.0
    assert bench.busy_ms(rec, "copy", 5.0, 6.0) == 0.0


def test_profile_traffic_is_gated_by_the_source_digest(tmp_path, monkeypatch):
    """DRAM traffic from a committed ncu summary is reported only while the
    summary's source digest matches the kernel sources it was taken on."""
    import bench
    src = tmp_path / "weight_streamed_bf16_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k.cu").write_text("kernel v1\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d1 = bench.source_digest("k.cu")
    (tmp_path / "profiles" / "k_traffic.txt").write_text(
        "a description without a separator\ncommand: ncu ...\n"
        f"source_digest: {d1}\ntraffic_bytes_per_launch: 12345\n")
    assert bench.profile_traffic("k_traffic.txt", d1) == 12345.0
    (src / "k.cu").write_text("kernel v2\n")             # the source changed
    d2 = bench.source_digest("k.cu")
    assert d2 != d1 and bench.profile_traffic("k_traffic.txt", d2) is None
    assert bench.profile_traffic("missing.txt", d1) is None
