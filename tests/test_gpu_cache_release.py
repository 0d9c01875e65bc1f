"""Stream-ordered release of cached tables.

A 17th grid evicts the oldest cache entry (the table cache of the sglang PR
#35698 review, "实现拆解" step 1: first-in-first-out, capped at 16). When a
launch that reads the evicted tables is still queued on another stream, the
evicting call must neither wait for that stream nor free the tables under it:
the buffer is retired and freed only after the launch completes. The queued
rotation is then compared with the oracle bit for bit, which it can only
match if its tables were still intact when it ran.
"""
from __future__ import annotations

import time

import numpy as np
import pytest

import oracle
import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU hosts
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import rope_rope3d_apply_gb300 as r  # noqa: E402

DEV = torch.device("cuda:0")
SLEEP_S = 0.6  # how long the side stream stays busy before the rotation


def _to_device(a, shp):
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).reshape(shp).to(DEV)


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16).reshape(-1)


def _busy(stream, seconds):
    """A spin kernel of a fixed number of clock cycles (about `seconds` at
    2 GHz; it always ends) on `stream`."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(seconds * 2.0e9))


@pytest.fixture(autouse=True)
def _gate_off():
    # with the gate on, the first call of a configuration waits for its kernel
    r.rope3d_gate_set_mode(r.GATE_OFF)
    r.rope3d_cache_clear()
    yield
    r.rope3d_cache_clear()
    r.rope3d_gate_set_mode(r.GATE_FIRST)


def _setup():
    w = synthetic.WORKLOADS["stage0"]
    q_np, k_np = synthetic.qk(w)
    shp = (w.B, w.N, w.heads, w.head_dim)
    q, k = _to_device(q_np, shp), _to_device(k_np, shp)
    otabs = oracle.tables(w.T, w.H, w.W, w.split, w.base)
    want = (oracle.rope3d(q_np, w.shape6, w.split, otabs), oracle.rope3d(k_np, w.shape6, w.split, otabs))
    # The first launch of a kernel in a process loads it (CUDA loads modules
    # lazily), which waits for the device: launch once before any stream is
    # made busy. Then clear the cache so the scenario starts from nothing.
    with r.rope3d_build_tables(w.T, w.H, w.W, w.split, w.base) as t:
        r.rope3d_apply_pair(q, k, t)
    torch.cuda.synchronize()
    r.rope3d_cache_clear()
    assert r.rope3d_cache_retired() == 0
    return w, q, k, want


def test_eviction_does_not_wait_for_a_busy_stream_and_keeps_its_tables():
    w, q, k, want = _setup()
    qo, ko = torch.empty_like(q), torch.empty_like(k)
    first = r.rope3d_build_tables(w.T, w.H, w.W, w.split, w.base)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    _busy(side, SLEEP_S)
    r.rope3d_apply_pair(q, k, first, qo, ko, stream=side)   # queued behind the spin
    first.close()                                           # the cache holds the last reference
    t0 = time.perf_counter()
    others = [r.rope3d_build_tables(w.T, w.H, w.W + 1 + i, w.split, w.base) for i in range(16)]
    evict_s = time.perf_counter() - t0
    assert r.rope3d_cache_stats()["evictions"] == 1
    waiting = r.rope3d_cache_retired()
    still_busy = not side.query()
    assert still_busy, "the spin ended before the evictions were checked"
    assert waiting == 1, "the evicted tables were freed while a launch still reads them"
    assert evict_s < SLEEP_S / 2, f"building 16 grids took {evict_s:.3f} s: it waited for the side stream"
    side.synchronize()
    assert r.rope3d_cache_retired() == 0
    assert np.array_equal(_bits(qo), want[0])
    assert np.array_equal(_bits(ko), want[1])
    for t in others:
        t.close()


def test_release_after_eviction_does_not_wait_and_keeps_its_tables():
    w, q, k, want = _setup()
    qo, ko = torch.empty_like(q), torch.empty_like(k)
    first = r.rope3d_build_tables(w.T, w.H, w.W, w.split, w.base)
    others = [r.rope3d_build_tables(w.T, w.H, w.W + 1 + i, w.split, w.base) for i in range(16)]
    assert r.rope3d_cache_stats()["evictions"] == 1          # `first` is held by the caller only
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    _busy(side, SLEEP_S)
    r.rope3d_apply_pair(q, k, first, qo, ko, stream=side)
    t0 = time.perf_counter()
    first.close()                                            # the last reference
    release_s = time.perf_counter() - t0
    assert not side.query()
    assert r.rope3d_cache_retired() == 1
    assert release_s < SLEEP_S / 2
    side.synchronize()
    assert r.rope3d_cache_retired() == 0
    assert np.array_equal(_bits(qo), want[0])
    assert np.array_equal(_bits(ko), want[1])
    for t in others:
        t.close()


def test_released_tables_used_by_attention_wait_for_it():
    """The fused attention entry points read the tables too (K pass and Q
    rotation): a release while they are queued must wait for them."""
    T, H, W, heads = 3, 8, 8, 2
    shp = (1, T * H * W, heads, 128)
    n = int(np.prod(shp))
    qkv = [torch.from_numpy(synthetic.normal(n, 1.0, 60, i, "bf16").view(np.int16))
           .view(torch.bfloat16).reshape(shp).to(DEV) for i in range(3)]
    split, kernel = (32, 48, 48), (3, 7, 7)
    ref_tabs = r.rope3d_build_tables(T, H, W, split)
    want, _ = r.rope3d_na3d_rotate_once(*qkv, ref_tabs, kernel)   # also loads the kernels
    torch.cuda.synchronize()
    want_bits = want.cpu().view(torch.int16).clone()
    ref_tabs.close()
    r.rope3d_cache_clear()                                   # the next build allocates afresh
    tabs = r.rope3d_build_tables(T, H, W, split)
    r.rope3d_cache_clear()                                   # the caller holds the only reference
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    _busy(side, SLEEP_S)
    out, k_rot = torch.empty_like(qkv[0]), torch.empty_like(qkv[1])
    r.rope3d_na3d_rotate_once(*qkv, tabs, kernel, out, k_rot=k_rot, stream=side)
    tabs.close()
    assert not side.query()
    assert r.rope3d_cache_retired() == 1
    side.synchronize()
    assert r.rope3d_cache_retired() == 0
    assert torch.equal(out.cpu().view(torch.int16), want_bits)
