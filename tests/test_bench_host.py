"""Host-side checks of bench.py: the reference arm's JSON line, the launch
count, and the multi-rank timing (max over ranks) with world size 2 on gloo."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

import synthetic

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "1", "--workload", "stage0"],
                         capture_output=True, text=True, timeout=300, check=True)
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["cores"] <= bench_host_cores()
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["steps"] == 2 and d["higher_is_better"] is True


def bench_host_cores():
    sys.path.insert(0, ROOT)
    import bench

    return bench.host_cores()


def test_cpu_baseline_single_and_all_cores():
    """cpu_baseline times the oracle on one thread and, on the same sample,
    on every host core (one frame per job); the per-frame jobs compute
    exactly what the single pass computes."""
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    import oracle
    import synthetic

    w = synthetic.WORKLOADS["stage0"]
    line = bench.cpu_baseline(w, 0.5)
    assert line["cores"] == 1 and line["value"] > 0
    assert line["all_cores"]["cores"] == bench.host_cores() and line["all_cores"]["value"] > 0
    q, _ = synthetic.qk(w)
    q = q.reshape(-1)
    tabs = oracle.tables(w.T, w.H, w.W, w.split, w.base)
    full = oracle.rope3d(q, (w.B, w.T, w.H, w.W, w.heads, w.head_dim), w.split, tabs)
    per_frame = w.H * w.W * w.heads * w.head_dim
    (ct, st), th, tw = tabs
    frames = [oracle.rope3d(q[i * per_frame:(i + 1) * per_frame], (1, 1, w.H, w.W, w.heads, w.head_dim),
                            w.split, ((ct[i:i + 1], st[i:i + 1]), th, tw)) for i in range(w.T)]
    assert np.array_equal(np.concatenate(frames), full.reshape(-1))


def test_launch_count():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.launches_per_call(synthetic.WORKLOADS["large"], 1) == 1
    assert bench.launches_per_call(synthetic.WORKLOADS["tiny"], 2) == 1


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.max_over_ranks(float(rank + 1) * 1.5, dist, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, slowest))


def test_max_over_ranks_gloo_world_2():
    torch = pytest.importorskip("torch")
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 3.0, 1: 3.0}


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0", "--workload", "tiny"],
                         capture_output=True, text=True, timeout=120, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_na3d_traffic_only_for_the_captured_kernel_and_workload(monkeypatch):
    """The attention line's traffic is the recorded capture's DRAM bytes only
    while the kernel source and the workload are the captured ones."""
    sys.path.insert(0, ROOT)
    import bench

    rec = bench.NA3D_TRAFFIC_RECORD
    c = dict(bench.NA3D)
    monkeypatch.setitem(rec, "kernel_source", bench.kernel_source_hash(bench.NA3D_KERNEL_SOURCES))
    assert bench.na3d_traffic_per_launch(c) == rec["dram_read_bytes"] + rec["dram_write_bytes"]
    assert bench.na3d_traffic_per_launch(dict(c, W=32)) is None
    assert bench.na3d_traffic_per_launch(dict(c, kernel=(1, 7, 7))) is None
    monkeypatch.setitem(rec, "kernel_source", "0" * 16)
    assert bench.na3d_traffic_per_launch(c) is None
