"""Seeded synthetic inputs and the workload shapes, shared by the tests, the
smoke check and the benchmark.

This module holds no RoPE arithmetic: it only draws Q and K. Values are
i.i.d. normal N(0, sigma) drawn in float32 with numpy's PCG64 and, for bf16
inputs, rounded to the nearest bfloat16 (ties to even) by bit manipulation
here. The stream is split into fixed chunks of ``CHUNK`` elements; chunk i of
tensor ``which`` (0 = Q, 1 = K) of seed s uses SeedSequence([s, which, i]),
so the values do not depend on the thread count.

The decoder geometries follow the LTX-2.5 decoder stages the sglang PR #35698
review measures ("功能与动机": stage 0, stage 4 tile, stage 5 tile); the page
does not print their shapes, so the sizes below are the workload definitions of
this project (tiny, stage-0-like, stage-4-tile-like, stage-5-tile-like with an
odd-width variant, and a large bandwidth sweep).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

CHUNK = 1 << 22


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    W: int
    heads: int
    head_dim: int
    split: tuple
    base: float = 10000.0
    sigma: float = 1.0
    seed: int = 0
    dtype: str = "bf16"          # "bf16", "f16" or "f32"
    repeat: int = 1              # calls per step sharing one table set
    note: str = field(default="", compare=False)

    @property
    def N(self) -> int:
        return self.T * self.H * self.W

    @property
    def shape6(self) -> tuple:
        return (self.B, self.T, self.H, self.W, self.heads, self.head_dim)

    @property
    def numel(self) -> int:
        return self.B * self.N * self.heads * self.head_dim

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def table_bytes(self) -> int:
        # cos and sin, fp32, [L_X, d_X / 2] per axis
        return sum(8 * n * (d // 2) for n, d in zip((self.T, self.H, self.W), self.split))

    @property
    def bytes_per_call(self) -> int:
        """Algorithmic bytes: read Q and K, write Q_out and K_out, read the tables once."""
        return 4 * self.numel * self.elem_bytes + self.table_bytes

    @property
    def token_heads(self) -> int:
        return self.B * self.N * self.heads


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", 1, 2, 4, 4, 2, 48, (16, 16, 16), sigma=1.0, seed=0),
        Workload("stage0", 1, 4, 16, 16, 16, 64, (16, 24, 24), sigma=1.0, seed=1),
        Workload("stage0_f32", 1, 4, 16, 16, 16, 64, (16, 24, 24), sigma=1.0, seed=1, dtype="f32"),
        Workload("stage4", 1, 8, 32, 32, 16, 128, (32, 48, 48), sigma=1.0, seed=2, repeat=24),
        Workload("stage5", 1, 16, 64, 64, 16, 128, (32, 48, 48), sigma=2.0, seed=3),
        Workload("stage5_w63", 1, 16, 64, 63, 16, 128, (32, 48, 48), sigma=2.0, seed=3),
        Workload("large", 2, 24, 96, 96, 24, 128, (32, 48, 48), sigma=1.0, seed=4),
    ]
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Nearest bfloat16 (ties to even) of finite float32 values, as uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def _chunk(seed: int, which: int, i: int, n: int, sigma: float, dtype: str) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, which, i])))
    v = g.standard_normal(n, dtype=np.float32)
    if sigma != 1.0:
        v *= np.float32(sigma)
    if dtype == "bf16":
        return f32_to_bf16_bits(v)
    if dtype == "f16":
        return v.astype(np.float16).view(np.uint16)   # nearest binary16, ties to even
    return v


def normal(numel: int, sigma: float, seed: int, which: int, dtype: str = "bf16",
           out: np.ndarray | None = None, threads: int | None = None) -> np.ndarray:
    """numel values (uint16 bf16 / binary16 bits, or float32) of tensor
    ``which`` of ``seed``.

    ``out`` may be a preallocated 1-D array (for instance a view of pinned host
    memory) of the right dtype; it is filled in place.
    """
    np_dtype = np.float32 if dtype == "f32" else np.uint16
    if out is None:
        out = np.empty(numel, dtype=np_dtype)
    if out.dtype != np_dtype or out.size != numel:
        raise ValueError("out has the wrong dtype or size")
    nchunks = (numel + CHUNK - 1) // CHUNK

    def fill(i):
        lo = i * CHUNK
        hi = min(numel, lo + CHUNK)
        out[lo:hi] = _chunk(seed, which, i, hi - lo, sigma, dtype)

    threads = threads or min(32, os.cpu_count() or 1)
    if nchunks <= 1 or threads <= 1:
        for i in range(nchunks):
            fill(i)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def qk(w: Workload, out_q: np.ndarray | None = None, out_k: np.ndarray | None = None):
    """Q then K for a workload (Q is tensor 0, K tensor 1 of the workload's seed)."""
    q = normal(w.numel, w.sigma, w.seed, 0, w.dtype, out=out_q)
    k = normal(w.numel, w.sigma, w.seed, 1, w.dtype, out=out_k)
    return q, k


def sample_indices(numel: int, count: int, seed: int, head_dim: int) -> np.ndarray:
    """Sorted flat indices to check at full size: ``count`` random ones plus
    the first and last head rows (the edges of the tensor)."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 99])))
    r = g.integers(0, numel, size=count, dtype=np.int64)
    edges = np.concatenate([np.arange(min(head_dim, numel)),
                            np.arange(max(0, numel - head_dim), numel)]).astype(np.int64)
    return np.unique(np.concatenate([r, edges]))
