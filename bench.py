#!/usr/bin/env python3
"""Benchmark of the fused paired 3D RoPE (Q and K) on GB300.

One step is one rotation of Q and K (one rope3d_apply_pair call, one kernel
launch) over the largest single-GPU workload: B=2, T=24, H=96, W=96
(221,184 tokens per batch), 24 heads, head_dim 128, split (32, 48, 48),
base 10000, bf16 values N(0, 1) from seed 4. Each step moves 10.87 GB
(read Q and K, write Q_out and K_out, read the tables once): far more than
the 129 MB L2, so no flush is needed between steps.

Metric: achieved HBM GB/s from algorithmic bytes (and the fraction of the
measured peak), plus tokens*heads per second. Printed as one JSON line.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference]

--impl reference times the CPU oracle (single thread, as it stands) on a
bounded sample of the same workload: each step rotates Q and K of the first
frame(s) of batch 0.
Under torchrun (N > 1) every rank runs its own replica on its own GPU (the
rotation needs no exchange): the value is all ranks' bytes over the slowest
rank's time.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = "fused 3D RoPE Q+K: achieved HBM GB/s and % of GB300 peak; bit-exact vs oracle"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = [os.path.join(ROOT, "rope_rope3d_apply_gb300", "csrc", "rope3d_kernels.cu")]

# DRAM traffic of one launch of the contiguous bf16 vector kernel, from one
# ncu capture (dram__bytes_read.sum, dram__bytes_write.sum; one launch, 2 GB
# on the device) of the stage-5 tile, 1,073,768,448 algorithmic bytes:
#   python bench.py --workload stage5 --steps 2 --warmup 3 --no-e2e --no-cpu-baseline
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum
#       --clock-control none -k regex:rope3d_vec16_kernel -s 4 -c 1 (the same command)
# Valid while the kernel source hashes to `kernel_source`; a launch of another
# size gets the same bytes per algorithmic byte (scaled by the units it moves).
TRAFFIC_RECORD = {
    "kernel_source": "ae41e94be201bd5f",
    "workload": "stage5",
    "algorithmic_bytes": 1_073_768_448,
    "dram_read_bytes": 536_930_304,
    "dram_write_bytes": 485_344_256,
}


# DRAM traffic of one launch of the tensor-core attention rotating its Q tiles
# (rope3d_na3d_tc_kernel<2>, the larger of the two kernels of the rotate-once
# step) on the NA3D workload, from one ncu capture (--set full, one launch,
# 1.07 GB on the device):
#   python bench.py --op na3d --steps 3 --warmup 3
#   ncu --set full --clock-control none -k regex:rope3d_na3d_tc_kernel -s 9 -c 1 (the same command)
# Valid while the attention source hashes to `kernel_source` and the workload
# is the recorded one.
NA3D_KERNEL_SOURCES = [os.path.join(ROOT, "rope_rope3d_apply_gb300", "csrc", "rope3d_na3d.cu")]
NA3D_TRAFFIC_RECORD = {
    "kernel_source": "3beb48028a0ef549",
    "kernel": "rope3d_na3d_tc_kernel<2>",
    "workload": {"B": 1, "T": 16, "H": 64, "W": 64, "heads": 16, "kernel": (3, 7, 7)},
    "dram_read_bytes": 805_516_544,
    "dram_write_bytes": 248_363_264,
}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="large", choices=sorted(synthetic.WORKLOADS))
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--variant", default="contiguous", choices=["contiguous", "f16", "qkv_inplace"],
                   help="contiguous Q/K (default); the same in fp16; or Q and K as views of a "
                        "fused [B, N, 3, heads, head_dim] QKV buffer rotated in place")
    p.add_argument("--op", default="rope", choices=["rope", "patchify", "neox", "na3d"],
                   help="rope: the fused 3D RoPE (default); patchify: the decoder's "
                        "space-to-depth layout kernel and its inverse")
    p.add_argument("--na3d-kernel", type=int, default=0, choices=[0, 1, 2],
                   help="--op na3d: 0 the library's choice, 1 the tensor-core (tcgen05) "
                        "attention, 2 the warp-MMA attention")
    p.add_argument("--graph", action="store_true",
                   help="capture one step's calls in a CUDA graph and time its replays")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def workload_config(w: synthetic.Workload) -> dict:
    return {
        "workload": (f"{w.name}: B={w.B}, T={w.T}, H={w.H}, W={w.W} (N={w.N}), heads={w.heads}, "
                     f"head_dim={w.head_dim}, split={tuple(w.split)}, base={w.base:g}, "
                     f"{w.dtype} N(0,{w.sigma:g}) seed {w.seed}"),
        "B": w.B, "T": w.T, "H": w.H, "W": w.W, "heads": w.heads, "head_dim": w.head_dim,
        "split": list(w.split), "io_dtype": w.dtype,
        "bytes_per_call": w.bytes_per_call,
        "calls_per_step": w.repeat,
        "bytes_per_step": w.bytes_per_call * w.repeat,
        "token_heads_per_step": w.token_heads * w.repeat,
        "l2": ("no flush: each step reads and writes %.2f GB in distinct buffers, more than "
               "the 129 MB L2" % (w.bytes_per_call * w.repeat / 1e9))
              if w.bytes_per_call * w.repeat > 1 << 30 else
              "inputs smaller than L2: numbers include L2 reuse",
    }


def host_link_gbs(torch, dev, h_in, h_out, d_in, d_out, reps=5):
    """`reps` rounds of raw copies: the pinned host inputs to device buffers on
    one stream while the device outputs go to pinned host buffers on another;
    per round, bytes moved both ways over the round's time (GB/s)."""
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    nbytes = sum(t.numel() * t.element_size() for t in h_in) + sum(t.numel() * t.element_size() for t in h_out)
    rounds = []
    for _ in range(reps):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        with torch.cuda.stream(s_in):
            for h, d in zip(h_in, d_in):
                d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s_out):
            for h, d in zip(h_out, d_out):
                h.copy_(d, non_blocking=True)
        torch.cuda.synchronize(dev)
        rounds.append(nbytes / (time.perf_counter() - t0) / 1e9)
    return rounds


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for p in sources or KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def na3d_traffic_per_launch(c) -> int | None:
    """DRAM bytes of one launch of the recorded attention kernel, while its
    source and the workload are the captured ones; otherwise None."""
    rec = NA3D_TRAFFIC_RECORD
    w = rec["workload"]
    same = all(c[key] == w[key] for key in ("B", "T", "H", "W", "heads")) and tuple(c["kernel"]) == w["kernel"]
    if not same or kernel_source_hash(NA3D_KERNEL_SOURCES) != rec["kernel_source"]:
        return None
    return rec["dram_read_bytes"] + rec["dram_write_bytes"]


def traffic_per_launch(w: synthetic.Workload):
    """DRAM bytes of one launch: the recorded capture's bytes per algorithmic
    byte times this launch's algorithmic bytes, while the kernel source is the
    one captured (bf16 contiguous calls only); otherwise None."""
    rec = TRAFFIC_RECORD
    if w.dtype != "bf16" or kernel_source_hash() != rec["kernel_source"]:
        return None
    per_byte = (rec["dram_read_bytes"] + rec["dram_write_bytes"]) / rec["algorithmic_bytes"]
    return int(per_byte * w.bytes_per_call)


class NvmlClocks:
    """Read-only NVML queries (SM clock, its maximum, the clock-event reasons)
    through the driver's libnvidia-ml, for one GPU given by PCI bus id."""

    SM = 1  # NVML_CLOCK_SM
    # reason bits of nvmlDeviceGetCurrentClocksEventReasons, by the names the
    # nvidia-smi query uses (hw_slowdown includes the power-brake slowdown)
    REASONS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8 | 0x80),
               ("sw_thermal_slowdown", 0x20), ("hw_thermal_slowdown", 0x40))

    def __init__(self, pci_bus_id: str):
        import ctypes

        self.c = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h)) != 0:
            raise OSError(f"no NVML device at {pci_bus_id}")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM, ctypes.byref(mx)) != 0:
            raise OSError("nvmlDeviceGetMaxClockInfo failed")
        self.max_mhz = float(mx.value)

    def read(self):
        c = self.c
        clk, bits = c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, c.byref(clk)) != 0:
            return None
        if self.reasons_fn(self.h, c.byref(bits)) != 0:
            return None
        reasons = [n for n, b in self.REASONS if bits.value & b]
        return float(clk.value), self.max_mhz, reasons


class ClockSampler:
    """SM clocks and throttle reasons while running: NVML every 5 ms (several
    samples even inside a timed region of a few tens of milliseconds), else
    nvidia-smi every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_S = 0.005

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.samples = []  # (time, sm_mhz, max_mhz, reasons)
        self.source = None
        self._proc = None
        self._thread = None
        self._stop = threading.Event()

    def start(self):
        try:
            nvml = NvmlClocks(self.gpu)
        except (OSError, AttributeError):
            nvml = None
        if nvml is not None and nvml.read() is not None:
            self.source = "nvml, every 5 ms"
            self._thread = threading.Thread(target=self._poll, args=(nvml,), daemon=True)
            self._thread.start()
            return
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self._proc = None
            return
        self.source = "nvidia-smi, every 100 ms"
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()

    def _poll(self, nvml):
        while not self._stop.is_set():
            s = nvml.read()
            if s is not None:
                self.samples.append((time.time(), *s))
            self._stop.wait(self.PERIOD_S)

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self._proc.stdout:
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = [n for n, v in zip(names, parts[5:9]) if v.lower().startswith("active")]
            self.samples.append((time.time(), sm, mx, reasons))

    def stop(self):
        self._stop.set()
        if self._proc:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread:
            self._thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        used = inside
        if not used and self.samples:
            # the timed region was shorter than the sampling period: nearest sample
            mid = 0.5 * (t0 + t1)
            used = [min(self.samples, key=lambda s: abs(s[0] - mid))]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": self.source}
        reasons = sorted({r for s in used for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in used),
                "sm_max_mhz": max(s[2] for s in used), "reasons": reasons,
                "samples": len(used), "samples_in_window": len(inside), "source": self.source}


def same_box_copy_gbs(torch, dev, sustained_s: float = 1.0):
    """A torch copy of 1 Gi bf16 elements on this GPU (read + write bytes, CUDA
    events): the best of 10 single copies, the way the measured peak was
    taken (how this GPU compares with the one the peak was measured on), and
    the average of back-to-back copies over about `sustained_s` seconds, timed
    like the kernel's own steps (the like-for-like ratio)."""
    x = torch.empty(1 << 30, dtype=torch.bfloat16, device=dev)
    y = torch.empty_like(x)
    nbytes = 2 * x.numel() * 2
    best = 0.0
    for _ in range(11):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        y.copy_(x)
        b.record()
        torch.cuda.synchronize(dev)
        best = max(best, nbytes / (a.elapsed_time(b) / 1e3) / 1e9)
    reps = max(10, int(sustained_s * best * 1e9 / nbytes))
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        y.copy_(x)
    b.record()
    torch.cuda.synchronize(dev)
    sustained = reps * nbytes / (a.elapsed_time(b) / 1e3) / 1e9
    del x, y
    return best, sustained


def launches_per_call(w: synthetic.Workload, kernel: int) -> int:
    """Kernel launches of one call: one per 2^30 work units (16-byte vectors or
    pairs), whole rows per launch."""
    per_unit = (16 // w.elem_bytes) if kernel == 1 else 2
    units_per_row = w.heads * w.head_dim // per_unit
    rows_per_launch = max(1, (1 << 30) // units_per_row)
    rows = w.B * w.N
    return -(-rows // rows_per_launch)


def max_over_ranks(value: float, dist, device) -> float:
    """The slowest rank's time (a no-op on one process)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def smi_gpu_id(local: int) -> str:
    """nvidia-smi --id for CUDA device `local` (by PCI bus id when known)."""
    try:
        import torch

        p = torch.cuda.get_device_properties(local)
        return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v for v in vis.split(",") if v.strip()]
        return ids[local] if local < len(ids) else str(local)


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def oracle_sample_step(w: synthetic.Workload, frames: int, rows: int, cache: dict, pool=None,
                       jobs: int = 1):
    """One oracle pass over Q and K of a leading sub-grid of batch 0: the first
    `rows` rows (h) of frame 0 when frames == 1, else the first `frames` whole
    frames. Those tokens use the same table rows as in the full workload, so
    the sub-grid is the same computation as that part of the workload. With a
    thread pool, frame 0's rows are cut into `jobs` blocks (each with its rows
    of the H table, so positions are unchanged) that run concurrently.
    Returns the algorithmic bytes of the pass."""
    import oracle

    key = (frames, rows)
    if key not in cache:
        shape = (1, frames, rows, w.W, w.heads, w.head_dim)
        n = int(np.prod(shape))
        q = synthetic.normal(n, w.sigma, w.seed, 0, w.dtype)
        k = synthetic.normal(n, w.sigma, w.seed, 1, w.dtype)
        tabs = oracle.tables(frames, rows, w.W, w.split, w.base)
        cache[key] = (shape, q, k, tabs)
    shape, q, k, tabs = cache[key]
    if pool is None or frames != 1 or jobs <= 1:
        oracle.rope3d(q, shape, w.split, tabs)
        oracle.rope3d(k, shape, w.split, tabs)
    else:
        per_row = w.W * w.heads * w.head_dim
        (tt, (ch, sh), tw) = tabs
        bounds = np.linspace(0, rows, min(jobs, rows) + 1).astype(int)

        def job(i):
            r0, r1 = int(bounds[i]), int(bounds[i + 1])
            sub = (tt, (ch[r0:r1], sh[r0:r1]), tw)
            shp = (1, 1, r1 - r0, w.W, w.heads, w.head_dim)
            oracle.rope3d(q[r0 * per_row:r1 * per_row], shp, w.split, sub)
            oracle.rope3d(k[r0 * per_row:r1 * per_row], shp, w.split, sub)

        list(pool.map(job, range(len(bounds) - 1)))
    return 4 * q.size * w.elem_bytes + sum(8 * n * (d // 2) for n, d in zip(shape[1:4], w.split))


def cpu_baseline(w: synthetic.Workload, seconds: float, q=None, k=None) -> dict:
    """The oracle as it stands, single-threaded, on a leading part of the
    workload sized to about `seconds` of CPU work: whole batches when one fits,
    else the first frames of batch 0 (the same table rows as the full run).
    q, k: the workload's host inputs when the caller has them (else drawn)."""
    import oracle

    per_frame = w.H * w.W * w.heads * w.head_dim
    if q is None or k is None:
        q, k = synthetic.qk(w)
    q, k = q.reshape(-1), k.reshape(-1)
    tabs = oracle.tables(w.T, w.H, w.W, w.split, w.base)
    t0 = time.perf_counter()
    oracle.rope3d(q[:per_frame], (1, 1, w.H, w.W, w.heads, w.head_dim), w.split, tabs)
    one = time.perf_counter() - t0          # one frame of Q, to size the sample
    frames_fit = seconds / max(2 * one, 1e-6)
    if frames_fit >= w.T:
        b, t = int(min(w.B, frames_fit // w.T)), w.T
    else:
        b, t = 1, int(max(1, frames_fit))
    shape = (b, t, w.H, w.W, w.heads, w.head_dim)
    n = b * t * per_frame
    sub = oracle.tables(t, w.H, w.W, w.split, w.base)
    t0 = time.perf_counter()
    oracle.rope3d(q[:n], shape, w.split, sub if b == 1 else tabs)
    oracle.rope3d(k[:n], shape, w.split, sub if b == 1 else tabs)
    dt = time.perf_counter() - t0
    moved = 4 * n * w.elem_bytes + sum(8 * m * (d // 2) for m, d in zip((t, w.H, w.W), w.split))
    what = (f"the whole workload ({b} x {t} frames)" if (b, t) == (w.B, w.T)
            else f"{b} whole batch(es)" if t == w.T else f"frames 0..{t - 1} of batch 0")
    line = {"value": moved / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"{what}: {b * t * w.H * w.W} tokens x {w.heads} heads, Q and K, "
                       f"{moved / 1e9:.3f} GB algorithmic, in {dt:.2f} s on one thread")}
    # The same sample on every host core: the unchanged oracle, one frame per
    # job (its T-table row sliced, so positions are those of the full grid);
    # the C oracle runs without the interpreter lock.
    from concurrent.futures import ThreadPoolExecutor

    cores = host_cores()
    (ct, st), th, tw = tabs
    one_frame = (1, 1, w.H, w.W, w.heads, w.head_dim)

    def frame_job(i):
        bi, ti = divmod(i, t)
        base = (bi * w.T + ti) * per_frame
        ft = ((ct[ti:ti + 1], st[ti:ti + 1]), th, tw)
        oracle.rope3d(q[base:base + per_frame], one_frame, w.split, ft)
        oracle.rope3d(k[base:base + per_frame], one_frame, w.split, ft)

    with ThreadPoolExecutor(max_workers=cores) as ex:
        t0 = time.perf_counter()
        list(ex.map(frame_job, range(b * t)))
        dt_all = time.perf_counter() - t0
    line["all_cores"] = {"value": moved / dt_all / 1e9, "unit": UNIT, "cores": cores,
                         "sample": f"the same sample, one frame per job, {cores} threads, "
                                   f"in {dt_all:.2f} s"}
    return line


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle
# ---------------------------------------------------------------------------

def run_reference(args, w):
    """The oracle timed on the host cores; each step a bounded sample (leading
    rows of frame 0 of batch 0) sized so that warm-up and timed steps together
    take about two minutes."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from concurrent.futures import ThreadPoolExecutor

    cores = host_cores()
    cache = {}
    oracle_sample_step(w, 1, 1, cache)  # inputs drawn once, outside the estimate
    t0 = time.perf_counter()
    oracle_sample_step(w, 1, 1, cache)
    per_row = time.perf_counter() - t0
    budget = 120.0 / max(1, args.steps + args.warmup)
    # rows per step: about the budget's worth of work across the cores
    rows = int(max(1, min(w.H, cores * budget / max(per_row, 1e-6))))
    with ThreadPoolExecutor(max_workers=cores) as pool:
        for _ in range(max(args.warmup, 0)):
            oracle_sample_step(w, 1, rows, cache, pool, cores)
        t0 = time.perf_counter()
        moved = 0
        for _ in range(args.steps):
            moved += oracle_sample_step(w, 1, rows, cache, pool, cores)
        dt = time.perf_counter() - t0
    value = moved / dt / 1e9
    used = min(cores, rows)
    sample = (f"each step: rows h=0..{rows - 1} of frame 0 of batch 0 ({rows * w.W} tokens x "
              f"{w.heads} heads, Q and K), oracle in {used} concurrent row blocks")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, w):
    import torch

    import rope_rope3d_apply_gb300 as r

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    r.load_library()

    # inputs: pinned host buffers (also the end-to-end inputs), then device copies
    np_dt = np.float32 if w.dtype == "f32" else np.uint16
    t_dtype = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[w.dtype]
    shp = (w.B, w.N, w.heads, w.head_dim)
    host = [torch.empty(w.numel * w.elem_bytes, dtype=torch.uint8).pin_memory() for _ in range(4)]
    hq, hk, hqo, hko = (h.numpy().view(np_dt).reshape(shp) for h in host)
    synthetic.qk(w, hq.reshape(-1), hk.reshape(-1))
    tabs = r.rope3d_build_tables(w.T, w.H, w.W, w.split, w.base)
    stream = torch.cuda.current_stream(dev)
    if args.variant == "qkv_inplace":
        qkv = torch.zeros((w.B, w.N, 3, w.heads, w.head_dim), dtype=t_dtype, device=dev)
        q, k = qkv[:, :, 0], qkv[:, :, 1]
        q.copy_(host[0].to(dev).view(t_dtype).view(shp))
        k.copy_(host[1].to(dev).view(t_dtype).view(shp))

        def step():
            r.rope3d_apply_pair_strided(q, k, tabs, q, k, stream=stream)
    else:
        # one buffer set per call of a step (the stage-4 tile runs 24 attention
        # blocks, each with its own Q and K, sharing one table set)
        sets = []
        for _ in range(w.repeat):
            q = host[0].to(dev).view(t_dtype).view(shp)
            k = host[1].to(dev).view(t_dtype).view(shp)
            sets.append((q, k, torch.empty_like(q), torch.empty_like(k)))

        def step():
            for q, k, qo, ko in sets:
                r.rope3d_apply_pair(q, k, tabs, qo, ko, stream=stream)

    # warm-up (the first call also runs the library's bit-exact gate)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if args.graph:
        # capture one step's calls in a CUDA graph (the gate has verified this
        # configuration during warm-up, so no call synchronises) and replay it
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            stream = torch.cuda.current_stream(dev)
            step()
        stream = torch.cuda.current_stream(dev)

        def step():
            graph.replay()
        for _ in range(3):
            step()
        torch.cuda.synchronize(dev)
    dt_code = {"bf16": r.BF16, "f16": r.F16, "f32": r.F32}[w.dtype]
    verdict = (r.rope3d_gate_verdict(w.B, w.T, w.H, w.W, w.heads, w.head_dim, w.split, w.base, dt_code)
               if args.variant != "qkv_inplace" else 1)  # a strided call that returned was verified
    launch = r.rope3d_last_launch()
    calls = w.repeat if args.variant != "qkv_inplace" else 1
    launches_per_step = calls * launches_per_call(w, launch["kernel"])

    # timed region: exactly K steps, per-launch events on the launching stream
    clocks = ClockSampler(smi_gpu_id(local))
    clocks.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    for i in range(args.steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    total_ms = starts[0].elapsed_time(ends[-1])
    per_launch = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    time.sleep(0.25)
    clocks.stop()
    clk = clocks.summary(t_wall0, t_wall1)

    total_ms = max_over_ranks(total_ms, dist, dev)

    box_copy, box_copy_sustained = same_box_copy_gbs(torch, dev)
    bytes_step = w.bytes_per_call * calls
    value = world * args.steps * bytes_step / (total_ms / 1e3) / 1e9
    kernel_ms = statistics.fmean(per_launch) / calls   # per call (one launch per call)
    achieved = w.bytes_per_call / (kernel_ms / 1e3) / 1e9
    peak, peak_kind = measured_peak()

    # end to end through the host-buffer entry point (copies inside the timed region)
    e2e = None
    if not args.no_e2e and args.variant != "qkv_inplace" and w.repeat == 1:
        r.rope3d_apply_pair_host(hq, hk, hqo, hko, tabs)  # warm-up: staging allocation
        if dist:
            dist.barrier()
        stamps = [time.perf_counter()]
        for _ in range(args.e2e_steps):
            r.rope3d_apply_pair_host(hq, hk, hqo, hko, tabs)
            stamps.append(time.perf_counter())
        e2e_s = max_over_ranks(stamps[-1] - stamps[0], dist, dev)
        step_gbs = sorted(world * bytes_step / (b - a) / 1e9 for a, b in zip(stamps, stamps[1:]))
        e2e = {"value": world * args.e2e_steps * bytes_step / e2e_s / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": 2 * w.numel * w.elem_bytes,
               "d2h_bytes_per_step": 2 * w.numel * w.elem_bytes,
               "steps": args.e2e_steps, "api": "rope3d_apply_pair_host (pinned host buffers)",
               "step_values": {"min": step_gbs[0], "median": statistics.median(step_gbs),
                               "max": step_gbs[-1]}}
        r.rope3d_release_scratch()
        # The host link right after (it stalls at random moments on some boxes):
        # raw concurrent copies of the same bytes, Q and K in, both outputs out.
        dq, dk, dqo, dko = (t.view(torch.uint8).reshape(-1) for t in sets[0])
        link = sorted(host_link_gbs(torch, dev, host[:2], host[2:], (dq, dk), (dqo, dko)))
        copied = e2e["h2d_bytes_per_step"] + e2e["d2h_bytes_per_step"]
        e2e["host_link_gbs"] = {"min": link[0], "median": statistics.median(link), "max": link[-1],
                                "rounds": len(link)}
        # copies of the median step against the link's median round
        e2e["frac_of_host_link"] = (statistics.median(step_gbs) / world * copied / bytes_step
                                    / statistics.median(link))

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": dict(workload_config(w), variant=args.variant,
                           parallelism=f"replicas x{world}" if world > 1 else "1 GPU"),
            "token_heads_per_s": world * args.steps * calls * w.token_heads / (total_ms / 1e3),
            "calls_per_step": calls, "cuda_graph": bool(args.graph),
            "pct_of_peak_hbm": 100.0 * achieved / peak,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic_per_launch(w),
                         "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth)",
                         "kernel_ms": kernel_ms,
                         "same_box_copy_gbs": box_copy,
                         "frac_of_same_box_copy": achieved / box_copy if box_copy else None,
                         "same_box_copy_sustained_gbs": box_copy_sustained,
                         "frac_of_same_box_copy_sustained":
                             achieved / box_copy_sustained if box_copy_sustained else None},
            "clocks": clk,
            "gpu_launches": args.steps * launches_per_step,
            "kernel": {"variant": {1: "vec16", 2: "pair"}.get(launch["kernel"], "?"),
                       "grid": launch["grid"], "block": launch["block"]},
            "gate_verdict": {0: "unseen", 1: "verified", 2: "refused"}[verdict],
            "e2e": e2e,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, hq, hk)
        print(json.dumps(line), flush=True)
    tabs.close()
    if dist:
        dist.destroy_process_group()
    return 0


# The patchify workload: a stand-in for the decoder's pixel-space volume (the
# page gives neither the patch size nor the shape): bf16, 268 MB each way.
PATCHIFY = dict(B=1, C=32, F=16, H=512, W=512, p=4)


def run_patchify(args):
    """Time rope3d_patchify (the step) and rope3d_unpatchify on PATCHIFY."""
    import torch

    import rope_rope3d_apply_gb300 as r

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    r.load_library()
    c = PATCHIFY
    shape = (c["B"], c["C"], c["F"], c["H"], c["W"])
    n = int(np.prod(shape))
    host = torch.empty(n * 2, dtype=torch.uint8).pin_memory()
    synthetic.normal(n, 1.0, 9, 0, "bf16", out=host.numpy().view(np.uint16))
    x = host.to(dev).view(torch.bfloat16).view(shape)
    p = c["p"]
    y = torch.empty((c["B"], c["C"] * p * p, c["F"], c["H"] // p, c["W"] // p),
                    dtype=x.dtype, device=dev)
    x2 = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        r.rope3d_patchify(x, p, y, stream=stream)
        r.rope3d_unpatchify(y, p, x2, stream=stream)
    torch.cuda.synchronize(dev)
    assert torch.equal(x2.view(torch.int16), x.view(torch.int16))
    kernel = r.rope3d_patchify_last_kernel()

    def timed(fn):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a.record(stream)
        for _ in range(args.steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / args.steps

    clocks = ClockSampler(smi_gpu_id(dev.index))
    clocks.start()
    time.sleep(0.3)
    t0 = time.time()
    ms_fwd = timed(lambda: r.rope3d_patchify(x, p, y, stream=stream))
    t1 = time.time()
    ms_inv = timed(lambda: r.rope3d_unpatchify(y, p, x2, stream=stream))
    time.sleep(0.25)
    clocks.stop()
    moved = 2 * n * 2
    peak, peak_kind = measured_peak()
    achieved = moved / (ms_fwd / 1e3) / 1e9
    line = {
        "op": "patchify", "metric": "patchify (space-to-depth) achieved HBM GB/s", "value": achieved,
        "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_fwd,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "patchify: x (B=%d, C=%d, F=%d, H=%d, W=%d) bf16, p=%d" % (
            c["B"], c["C"], c["F"], c["H"], c["W"], p), "bytes_per_step": moved,
            "l2": "no flush: 0.54 GB read and written per step, more than the 129 MB L2"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth)", "kernel_ms": ms_fwd},
        "unpatchify": {"ms": ms_inv, "GBps": moved / (ms_inv / 1e3) / 1e9,
                       "frac": moved / (ms_inv / 1e3) / 1e9 / peak},
        "kernel": {1: "vector", 2: "element"}.get(kernel, "?"),
        "clocks": clocks.summary(t0, t1), "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


# The NeoX workload: a Gemma3-like prefill (the page gives no sizes): 65,536
# tokens, 8 query heads and 4 key heads of 256 channels, bf16, positions
# 0..65535 into a 131,072-row cache.
NEOX = dict(tokens=65536, q_heads=8, k_heads=4, head_dim=256, max_position=131072)


def run_neox(args):
    """Time rope3d_apply_neox on NEOX (one launch per step)."""
    import torch

    import rope_rope3d_apply_gb300 as r

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    r.load_library()
    c = NEOX
    t, qh, kh, hd = c["tokens"], c["q_heads"], c["k_heads"], c["head_dim"]
    q = torch.from_numpy(synthetic.normal(t * qh * hd, 1.0, 11, 0, "bf16").view(np.int16)) \
        .view(torch.bfloat16).reshape(t, qh, hd).to(dev)
    k = torch.from_numpy(synthetic.normal(t * kh * hd, 1.0, 11, 1, "bf16").view(np.int16)) \
        .view(torch.bfloat16).reshape(t, kh, hd).to(dev)
    pos = torch.arange(t, dtype=torch.int64, device=dev)
    cache = torch.from_numpy(r.rope3d_neox_cache_host(c["max_position"], hd)).to(dev)
    qo, ko = torch.empty_like(q), torch.empty_like(k)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        r.rope3d_apply_neox(q, k, pos, cache, qo, ko, stream=stream)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(smi_gpu_id(dev.index))
    clocks.start()
    time.sleep(0.3)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    a.record(stream)
    for _ in range(args.steps):
        r.rope3d_apply_neox(q, k, pos, cache, qo, ko, stream=stream)
    b.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    time.sleep(0.25)
    clocks.stop()
    ms = a.elapsed_time(b) / args.steps
    moved = (qh + kh) * hd * 2 * 2 * t + t * hd * 4 + t * 8
    peak, peak_kind = measured_peak()
    achieved = moved / (ms / 1e3) / 1e9
    line = {
        "op": "neox", "metric": "NeoX RoPE (Q+K) achieved HBM GB/s", "value": achieved, "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "neox: %d tokens, %d/%d heads x %d, cache %d rows, positions 0..%d" % (
            t, qh, kh, hd, c["max_position"], t - 1), "bytes_per_step": moved,
            "l2": "no flush: %.2f GB per step, more than the 129 MB L2" % (moved / 1e9)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth)", "kernel_ms": ms},
        "kernel": {1: "vector", 2: "pair"}.get(r.rope3d_neox_last_kernel(), "?"),
        "clocks": clocks.summary(t0, t1), "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


# The fused attention workload: the stage-5 tile geometry (1 x 16 x 64 x 64
# tokens, 16 heads x 128, bf16) with a 3 x 7 x 7 neighbourhood (the pages give
# no window size).
NA3D = dict(B=1, T=16, H=64, W=64, heads=16, split=(32, 48, 48), kernel=(3, 7, 7))


def na3d_tc_mma_flops(B, T, H, W, heads, kernel, chunk_keys=112):
    """The tensor-core attention's issued MMA work: per 2 x 8 x 8 query block,
    S = Q K^T and O += P V over every chunk of its key region (whole region
    rows of one frame, rwb = min(W, k_w + 7) keys each, chunk_keys // rwb rows
    a chunk, the chunk's keys rounded up to 16), 4 * 128 * 128 * N flops a
    chunk of N keys."""
    kt, kh, kw = kernel

    def start(i, L, k):
        s0 = max(i - k // 2, 0)
        return L - k if s0 + k > L else s0

    rwb = min(W, kw + 7)
    chb = chunk_keys // rwb
    total = 0
    for t0 in range(0, T, 2):
        frames = start(min(t0 + 1, T - 1), T, kt) + kt - start(t0, T, kt)
        for h0 in range(0, H, 8):
            rh0 = start(h0, H, kh)
            RH = start(min(h0 + 7, H - 1), H, kh) + kh - rh0
            keys = sum(((min(chb, RH - r0) * rwb + 15) // 16) * 16 for r0 in range(0, RH, chb))
            total += frames * keys * ((W + 7) // 8)
    return 4.0 * 128 * 128 * total * B * heads


def run_na3d(args):
    """The RoPE fused with the neighbourhood attention, each element of Q and
    K rotated once (rope3d_na3d_rotate_once: the step), against the per-CTA
    fused form (rope3d_na3d rotating every K tile it copies) and the unfused
    pair (rope3d_apply_pair, then rope3d_na3d on the rotated Q and K)."""
    import torch

    import rope_rope3d_apply_gb300 as r

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    r.load_library()
    c = NA3D
    N = c["T"] * c["H"] * c["W"]
    shp = (c["B"], N, c["heads"], 128)
    n = int(np.prod(shp))
    q, k, v = (torch.from_numpy(synthetic.normal(n, 1.0, 12, i, "bf16").view(np.int16))
               .view(torch.bfloat16).reshape(shp).to(dev) for i in range(3))
    tabs = r.rope3d_build_tables(c["T"], c["H"], c["W"], c["split"])
    r.rope3d_testing_na3d_kernel(args.na3d_kernel)
    out = torch.empty_like(q)
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    stream = torch.cuda.current_stream(dev)

    def once():
        r.rope3d_na3d_rotate_once(q, k, v, tabs, c["kernel"], out, k_rot=kr, stream=stream)

    def fused():   # K rotated once into the library's pooled scratch
        r.rope3d_na3d(q, k, v, tabs, c["kernel"], out, stream=stream)

    def fused_per_cta():   # Q and every K tile rotated inside each CTA
        r.rope3d_testing_na3d_per_cta(True)
        try:
            r.rope3d_na3d(q, k, v, tabs, c["kernel"], out, stream=stream)
        finally:
            r.rope3d_testing_na3d_per_cta(False)

    def unfused():
        r.rope3d_apply_pair(q, k, tabs, qr, kr, stream=stream)
        r.rope3d_na3d(qr, kr, v, tabs, c["kernel"], out, apply_rope=False, stream=stream)

    def attention_only():
        r.rope3d_na3d(qr, kr, v, tabs, c["kernel"], out, apply_rope=False, stream=stream)

    def timed(fn, steps):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / steps

    clocks = ClockSampler(smi_gpu_id(dev.index))
    clocks.start()
    time.sleep(0.3)
    t0 = time.time()
    ms_once = timed(once, args.steps)
    t1 = time.time()
    ms_fused = timed(fused, args.steps)
    ms_per_cta = timed(fused_per_cta, args.steps)
    ms_unfused = timed(unfused, args.steps)
    ms_attention = timed(attention_only, args.steps)
    time.sleep(0.25)
    clocks.stop()
    kt, kh, kw = c["kernel"]
    window = kt * kh * kw
    flops = 4.0 * 128 * window * N * c["heads"] * c["B"]           # q.k and p.v over each window
    mma_flops = na3d_tc_mma_flops(c["B"], c["T"], c["H"], c["W"], c["heads"], c["kernel"])
    tflops = flops / (ms_once / 1e3) / 1e12
    peak = 1898.6
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)["bf16_tflops"])
        kind = "measured"
    except (OSError, KeyError, ValueError):
        kind = "fallback"
    line = {
        "op": "na3d", "metric": "fused RoPE + 3D neighbourhood attention, useful TFLOP/s",
        "value": tflops, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": ms_once, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "na3d: B=%d, T=%d, H=%d, W=%d, heads=%d x 128, window %dx%dx%d" % (
            c["B"], c["T"], c["H"], c["W"], c["heads"], kt, kh, kw), "useful_flops": flops},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops / peak, "traffic": na3d_traffic_per_launch(c),
                     "traffic_kernel": NA3D_TRAFFIC_RECORD["kernel"],
                     "peak_source": f"{kind} bf16_tflops (cuBLAS burst)", "kernel_ms": ms_once},
        "step": "rope3d_na3d_rotate_once (K pass + attention rotating its Q tiles)",
        "attention_kernel": {1: "tcgen05 (tensor memory)", 2: "warp-level mma.sync"}.get(
            r.rope3d_testing_na3d_last_kernel(), "?"),
        "unfused_ms": ms_unfused, "fusion_saving_ms": ms_unfused - ms_once,
        "fused_ms": ms_fused, "fused_per_cta_ms": ms_per_cta,
        "attention_only_ms": ms_attention,
        "attention_only_tflops": flops / (ms_attention / 1e3) / 1e12,
        # the tensor cores' issued work (the whole key region of each query
        # block), against the same peak: how busy the MMAs are
        "attention_only_mma_issued_tflops": mma_flops / (ms_attention / 1e3) / 1e12,
        "attention_only_mma_issued_frac": mma_flops / (ms_attention / 1e3) / 1e12 / peak,
        "clocks": clocks.summary(t0, t1), "gpu_launches": 2 * args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.op == "na3d":
        return run_na3d(args)
    if args.op == "patchify":
        return run_patchify(args)
    if args.op == "neox":
        return run_neox(args)
    w = synthetic.WORKLOADS[args.workload]
    if args.variant == "f16":
        w = dataclasses.replace(w, dtype="f16")
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
