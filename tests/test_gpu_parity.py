"""GPU parity: the CUDA path through the C ABI against the CPU oracle,
element by element, on seeded inputs.

The bar is bit-exactness (sglang PR #35698 review, "实现拆解" step 4 and
"评论区精华": the fused output must equal the eager order bit for bit; every
test there asserts with torch.equal). The one allowance: where both sides give
a NaN, any NaN payload is accepted (the pages do not fix NaN payloads).
"""
from __future__ import annotations

import os

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


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def to_device(a: np.ndarray, shape, dtype: str):
    if dtype == "bf16":
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    return t.reshape(shape).to(DEV)


def to_numpy(t) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return t.numpy().reshape(-1)


def assert_bit_exact(got: np.ndarray, want: np.ndarray, what=""):
    """Equal bit patterns, or NaN on both sides."""
    assert got.shape == want.shape and got.dtype == want.dtype
    if got.dtype == np.uint16:
        g, w = got, want
        nan = lambda b: (b & 0x7FFF) > 0x7F80  # noqa: E731
    else:
        g, w = got.view(np.uint32), want.view(np.uint32)
        nan = lambda b: (b & 0x7FFFFFFF) > 0x7F800000  # noqa: E731
    bad = (g != w) & ~(nan(g) & nan(w))
    if bad.any():
        i = np.flatnonzero(bad)
        pytest.fail(f"{what}: {i.size} mismatches, first at {i[:5]}: got {g[i[:5]]} want {w[i[:5]]}")


def run_gpu(q_np, k_np, shape6, split, dtype, base=10000.0, offset_elems=0, layout4=True):
    """Upload, rotate through rope3d_apply_pair, return host outputs."""
    B, T, H, W, heads, hd = shape6
    shp = (B, T * H * W, heads, hd) if layout4 else shape6
    q = to_device(q_np, shp, dtype)
    k = to_device(k_np, shp, dtype)
    if offset_elems:
        # sub-views that start offset_elems into a larger buffer (4-byte aligned,
        # not 16-byte aligned)
        def shifted(t):
            big = torch.empty(t.numel() + offset_elems, dtype=t.dtype, device=DEV)
            v = big[offset_elems:].view(shp)
            v.copy_(t)
            return v
        q, k = shifted(q), shifted(k)
        qo = torch.empty(q.numel() + offset_elems, dtype=q.dtype, device=DEV)[offset_elems:].view(shp)
        ko = torch.empty(q.numel() + offset_elems, dtype=q.dtype, device=DEV)[offset_elems:].view(shp)
    else:
        qo, ko = None, None
    tabs = r.rope3d_build_tables(T, H, W, split, base)
    qo, ko = r.rope3d_apply_pair(q, k, tabs, qo, ko)
    torch.cuda.synchronize()
    info = r.rope3d_last_launch()
    tabs.close()
    return to_numpy(qo), to_numpy(ko), info


def oracle_full(q_np, k_np, shape6, split, base=10000.0):
    tabs = oracle.tables(*shape6[1:4], split, base)
    return oracle.rope3d(q_np, shape6, split, tabs), oracle.rope3d(k_np, shape6, split, tabs)


@pytest.fixture(autouse=True)
def _fresh_gate():
    r.rope3d_gate_reset()
    r.rope3d_gate_set_mode(r.GATE_FIRST)
    r.rope3d_testing_max_units_per_launch(0)
    yield
    r.rope3d_gate_reset()
    r.rope3d_testing_max_units_per_launch(0)


# ---------------------------------------------------------------------------
# the workloads, full comparison
# ---------------------------------------------------------------------------

FULL = ["tiny", "stage0", "stage0_f32", "stage4", "stage5", "stage5_w63"]


@pytest.mark.parametrize("name", FULL)
def test_workload_bit_exact(name):
    w = synthetic.WORKLOADS[name]
    q_np, k_np = synthetic.qk(w)
    got_q, got_k, info = run_gpu(q_np, k_np, w.shape6, w.split, w.dtype, w.base)
    assert info["kernel"] == 1, info  # these shapes take the 16-byte vector kernel
    want_q, want_k = oracle_full(q_np, k_np, w.shape6, w.split, w.base)
    assert_bit_exact(got_q, want_q, f"{name} Q")
    assert_bit_exact(got_k, want_k, f"{name} K")
    # the first call of the configuration was verified by the library's gate too
    dt = r.BF16 if w.dtype == "bf16" else r.F32
    assert r.rope3d_gate_verdict(w.B, w.T, w.H, w.W, w.heads, w.head_dim, w.split, w.base, dt) == 1


def test_large_full_bit_exact():
    """The largest workload (2 x 24 x 96 x 96 tokens, 24 heads, head_dim 128,
    2.7 GB per tensor), in the launch configuration the benchmark times:
    every element of Q_out and K_out compared with the oracle. The outputs
    come back whole; the oracle runs one frame per job on every host core (each
    job with its row of the T table, so positions are those of the full grid),
    and each frame is compared as it finishes."""
    from concurrent.futures import ThreadPoolExecutor

    w = synthetic.WORKLOADS["large"]
    q_np, k_np = synthetic.qk(w)
    shp = (w.B, w.N, w.heads, w.head_dim)
    q = to_device(q_np, shp, "bf16")
    k = to_device(k_np, shp, "bf16")
    tabs = r.rope3d_build_tables(w.T, w.H, w.W, w.split, w.base)
    qo, ko = r.rope3d_apply_pair(q, k, tabs)  # the first call also runs the library's gate
    torch.cuda.synchronize()
    assert r.rope3d_last_launch()["kernel"] == 1
    assert r.rope3d_gate_verdict(w.B, w.T, w.H, w.W, w.heads, w.head_dim, w.split, w.base, r.BF16) == 1
    # a second call (gate already verified) gives the same bits
    qo2, ko2 = r.rope3d_apply_pair(q, k, tabs)
    torch.cuda.synchronize()
    assert torch.equal(qo2.view(torch.int16), qo.view(torch.int16))
    assert torch.equal(ko2.view(torch.int16), ko.view(torch.int16))
    del qo2, ko2, q, k
    got = {"Q": to_numpy(qo), "K": to_numpy(ko)}
    del qo, ko
    tabs.close()
    src = {"Q": q_np.reshape(-1), "K": k_np.reshape(-1)}
    (ct, st), th, tw = oracle.tables(w.T, w.H, w.W, w.split, w.base)
    per_frame = w.H * w.W * w.heads * w.head_dim
    one_frame = (1, 1, w.H, w.W, w.heads, w.head_dim)

    def frame_mismatches(job):
        name, b, t = job
        base = (b * w.T + t) * per_frame
        ft = ((ct[t:t + 1], st[t:t + 1]), th, tw)
        want = oracle.rope3d(src[name][base:base + per_frame], one_frame, w.split, ft)
        return int(np.count_nonzero(got[name][base:base + per_frame] != want))

    jobs = [(name, b, t) for name in ("Q", "K") for b in range(w.B) for t in range(w.T)]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    with ThreadPoolExecutor(max_workers=cores) as ex:
        bad = dict(zip(jobs, ex.map(frame_mismatches, jobs)))
    compared = len(jobs) * per_frame
    assert compared == 2 * w.numel == 2 * 1_358_954_496
    wrong = {j: n for j, n in bad.items() if n}
    assert not wrong, f"mismatching elements per (tensor, batch, frame): {wrong}"


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

EDGE = [
    # (B, T, H, W, heads, head_dim), split, dtype, expected kernel
    ((3, 1, 1, 1, 2, 48), (16, 16, 16), "bf16", 1),        # a 1x1x1 grid, batches wrap
    ((2, 5, 1, 7, 3, 48), (16, 16, 16), "bf16", 1),        # H = 1
    ((1, 3, 5, 7, 3, 24), (6, 8, 10), "bf16", 2),          # chunks not multiples of 8
    ((2, 3, 5, 7, 3, 18), (4, 6, 8), "f32", 2),            # fp32, chunks not multiples of 4
    ((2, 3, 5, 7, 3, 24), (4, 8, 12), "f32", 1),           # fp32 16-byte path, 2 pairs/vector
    ((1, 2, 3, 3, 1, 4096), (1024, 1536, 1536), "bf16", 1),  # the largest head_dim
    ((1, 1, 1, 257, 1, 2 + 2 + 2), (2, 2, 2), "bf16", 2),  # minimal chunks, long W
    ((1, 7, 9, 11, 5, 40), (8, 16, 16), "bf16", 1),        # odd grid, ragged tail
    ((4, 2, 2, 2, 1, 8), (8 - 4, 2, 2), "f32", 2),         # tiny rows
]


@pytest.mark.parametrize("case", EDGE, ids=[f"{c[0]}-{c[1]}-{c[2]}" for c in EDGE])
def test_edge_shapes(case):
    shape6, split, dtype, kernel = case
    n = int(np.prod(shape6))
    q_np = synthetic.normal(n, 1.0, 50, 0, dtype)
    k_np = synthetic.normal(n, 1.0, 50, 1, dtype)
    got_q, got_k, info = run_gpu(q_np, k_np, shape6, split, dtype)
    assert info["kernel"] == kernel, info
    want_q, want_k = oracle_full(q_np, k_np, shape6, split)
    assert_bit_exact(got_q, want_q, "Q")
    assert_bit_exact(got_k, want_k, "K")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_unaligned_pointers_take_pair_kernel(dtype):
    """4-byte aligned but not 16-byte aligned buffers."""
    w = synthetic.WORKLOADS["stage0"]
    q_np = synthetic.normal(w.numel, 1.0, 51, 0, dtype)
    k_np = synthetic.normal(w.numel, 1.0, 51, 1, dtype)
    off = 2 if dtype == "bf16" else 1
    got_q, got_k, info = run_gpu(q_np, k_np, w.shape6, w.split, dtype, offset_elems=off)
    assert info["kernel"] == 2, info
    want_q, want_k = oracle_full(q_np, k_np, w.shape6, w.split)
    assert_bit_exact(got_q, want_q, "Q")
    assert_bit_exact(got_k, want_k, "K")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_special_values(dtype):
    """Signed zeros, subnormals, the largest finite values, infinities and
    NaNs, mixed into normal data."""
    shape6, split = (2, 3, 4, 5, 2, 32), (8, 8, 16)
    n = int(np.prod(shape6))
    x = synthetic.normal(n, 1.0, 52, 0, "f32")
    g = np.random.Generator(np.random.PCG64(52))
    pool = np.array([0.0, -0.0, 2.0 ** -130, -(2.0 ** -133), 2.0 ** -149, 1e-39,
                     3.3e38, -3.38e38, np.inf, -np.inf, np.nan, 1.0, -1.0], np.float32)
    pick = g.integers(0, n, n // 4)
    x[pick] = pool[g.integers(0, pool.size, pick.size)]
    # tiny magnitudes so that products underflow into subnormals
    x[g.integers(0, n, n // 8)] *= np.float32(2.0 ** -120)
    if dtype == "bf16":
        u = x.view(np.uint32)
        q_np = (u >> np.uint32(16)).astype(np.uint16)  # truncation keeps NaN/inf/zero classes
        k_np = q_np[::-1].copy()
    else:
        q_np = x
        k_np = x[::-1].copy()
    got_q, got_k, _ = run_gpu(q_np, k_np, shape6, split, dtype)
    want_q, want_k = oracle_full(q_np, k_np, shape6, split)
    assert_bit_exact(got_q, want_q, "Q")
    assert_bit_exact(got_k, want_k, "K")


def test_multi_launch_split_matches():
    """With the per-launch cap lowered, a workload runs as several launches
    (each with its own first row); the result is unchanged."""
    w = synthetic.WORKLOADS["stage0"]
    q_np, k_np = synthetic.qk(w)
    want_q, want_k = oracle_full(q_np, k_np, w.shape6, w.split)
    for cap in (1000, 4096, 77):
        r.rope3d_testing_max_units_per_launch(cap)
        got_q, got_k, _ = run_gpu(q_np, k_np, w.shape6, w.split, "bf16")
        assert_bit_exact(got_q, want_q, f"cap {cap} Q")
        assert_bit_exact(got_k, want_k, f"cap {cap} K")
    r.rope3d_testing_max_units_per_launch(0)


def test_six_d_layout_and_guard_bytes():
    """6-D tensors are the same memory as [B, N, heads, head_dim]; writes stay
    inside the outputs (guard bytes around them are untouched)."""
    shape6, split = (2, 3, 5, 7, 3, 24), (8, 8, 8)
    n = int(np.prod(shape6))
    q_np = synthetic.normal(n, 1.0, 53, 0, "bf16")
    k_np = synthetic.normal(n, 1.0, 53, 1, "bf16")
    q = to_device(q_np, shape6, "bf16")
    k = to_device(k_np, shape6, "bf16")
    guard = 4096
    bq = torch.full((n + 2 * guard,), -7.0, dtype=torch.bfloat16, device=DEV)
    bk = torch.full((n + 2 * guard,), -7.0, dtype=torch.bfloat16, device=DEV)
    qo = bq[guard:guard + n].view(shape6)
    ko = bk[guard:guard + n].view(shape6)
    tabs = r.rope3d_build_tables(3, 5, 7, split)
    r.rope3d_apply_pair(q, k, tabs, qo, ko)
    torch.cuda.synchronize()
    for b in (bq, bk):
        assert torch.all(b[:guard] == -7.0) and torch.all(b[-guard:] == -7.0)
    want_q, want_k = oracle_full(q_np, k_np, shape6, split)
    assert_bit_exact(to_numpy(qo), want_q, "Q")
    assert_bit_exact(to_numpy(ko), want_k, "K")
    tabs.close()


# ---------------------------------------------------------------------------
# preflight on the device
# ---------------------------------------------------------------------------

def test_rejections_leave_outputs_untouched():
    w = synthetic.WORKLOADS["tiny"]
    shp = (w.B, w.N, w.heads, w.head_dim)
    q = torch.randn(shp, device=DEV).to(torch.bfloat16)
    k = torch.randn(shp, device=DEV).to(torch.bfloat16)
    qo = torch.full(shp, 3.0, dtype=torch.bfloat16, device=DEV)
    ko = torch.full(shp, 3.0, dtype=torch.bfloat16, device=DEV)
    tabs = r.rope3d_build_tables(w.T, w.H, w.W, w.split)
    lib = r.load_library()
    sp = (r.ctypes.c_int32 * 3)(*w.split)
    args = lambda **kw: dict(dict(q=q.data_ptr(), k=k.data_ptr(), qo=qo.data_ptr(),  # noqa: E731
                                  ko=ko.data_ptr(), B=w.B, heads=w.heads, hd=w.head_dim,
                                  dt=r.BF16), **kw)
    cases = {
        "ERR_SHAPE": args(B=0),
        "ERR_DTYPE": args(dt=5),
        "ERR_ALIGN": args(q=q.data_ptr() + 2),
        "ERR_ALIAS": args(qo=q.data_ptr()),
        "ERR_NULL": args(k=0),
    }
    for want, a in cases.items():
        rc = lib.rope3d_apply_pair(a["q"], a["k"], a["qo"], a["ko"], tabs.handle, a["B"], w.T, w.H,
                                   w.W, a["heads"], a["hd"], sp, a["dt"], 0)
        assert r.STATUS[rc] == want, (want, r.STATUS[rc])
    # host memory given to the device entry point
    host = torch.empty(shp, dtype=torch.bfloat16)
    rc = lib.rope3d_apply_pair(host.data_ptr(), k.data_ptr(), qo.data_ptr(), ko.data_ptr(),
                               tabs.handle, w.B, w.T, w.H, w.W, w.heads, w.head_dim, sp, r.BF16, 0)
    assert r.STATUS[rc] == "ERR_DEVICE"
    # tables of another grid
    other = r.rope3d_build_tables(w.T, w.H, w.W + 1, w.split)
    rc = lib.rope3d_apply_pair(q.data_ptr(), k.data_ptr(), qo.data_ptr(), ko.data_ptr(),
                               other.handle, w.B, w.T, w.H, w.W, w.heads, w.head_dim, sp, r.BF16, 0)
    assert r.STATUS[rc] == "ERR_TABLES"
    torch.cuda.synchronize()
    assert torch.all(qo == 3.0) and torch.all(ko == 3.0)
    with pytest.raises(ValueError):
        r.rope3d_apply_pair(q.transpose(1, 2), k.transpose(1, 2), tabs)  # not contiguous
    tabs.close()
    other.close()


# ---------------------------------------------------------------------------
# the gate, the table cache, streams
# ---------------------------------------------------------------------------

def test_gate_verifies_then_trusts_and_refuses_on_mismatch():
    w = synthetic.WORKLOADS["stage0"]
    q_np, k_np = synthetic.qk(w)
    shp = (w.B, w.N, w.heads, w.head_dim)
    q, k = to_device(q_np, shp, "bf16"), to_device(k_np, shp, "bf16")
    tabs = r.rope3d_build_tables(w.T, w.H, w.W, w.split)
    key = (w.B, w.T, w.H, w.W, w.heads, w.head_dim, w.split, w.base)
    assert r.rope3d_gate_verdict(*key, r.BF16) == 0
    r.rope3d_apply_pair(q, k, tabs)
    assert r.rope3d_gate_verdict(*key, r.BF16) == 1
    # a planted one-bit difference in the host copy makes the gate refuse
    r.rope3d_gate_reset()
    r.rope3d_testing_corrupt_gate(1)
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_apply_pair(q, k, tabs)
    assert e.value.name == "ERR_PARITY"
    assert r.rope3d_gate_verdict(*key, r.BF16) == 2
    # refused for good: later calls fail before launching
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_apply_pair(q, k, tabs)
    assert e.value.name == "ERR_PARITY"
    # other configurations are unaffected
    w0 = synthetic.WORKLOADS["tiny"]
    qt = torch.randn((w0.B, w0.N, w0.heads, w0.head_dim), device=DEV).to(torch.bfloat16)
    t0 = r.rope3d_build_tables(w0.T, w0.H, w0.W, w0.split)
    r.rope3d_apply_pair(qt, qt.clone(), t0)
    # reset forgets the refusal; with the gate off nothing is recorded
    r.rope3d_gate_reset()
    r.rope3d_gate_set_mode(r.GATE_OFF)
    r.rope3d_apply_pair(q, k, tabs)
    assert r.rope3d_gate_verdict(*key, r.BF16) == 0
    r.rope3d_gate_set_mode(r.GATE_FIRST)
    tabs.close()
    t0.close()


def test_tables_shared_across_24_blocks():
    """Stage-4 tile: 24 attention blocks share one cached table set
    ("实现拆解" step 1); every block's call gives the same bits."""
    r.rope3d_cache_clear()
    w = synthetic.WORKLOADS["stage4"]
    q_np, k_np = synthetic.qk(w)
    shp = (w.B, w.N, w.heads, w.head_dim)
    q, k = to_device(q_np, shp, "bf16"), to_device(k_np, shp, "bf16")
    handles, outs = [], []
    for _ in range(24):
        t = r.rope3d_build_tables(w.T, w.H, w.W, w.split, w.base)
        handles.append(t)
        outs.append(r.rope3d_apply_pair(q, k, t))
    torch.cuda.synchronize()
    st = r.rope3d_cache_stats()
    assert st["misses"] == 1 and st["hits"] == 23 and st["entries"] == 1
    assert len({h.handle for h in handles}) == 1
    for qo, ko in outs[1:]:
        assert torch.equal(qo.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(ko.view(torch.int16), outs[0][1].view(torch.int16))
    otabs = oracle.tables(w.T, w.H, w.W, w.split)
    for axis in range(3):
        c, s = r.rope3d_tables_read(handles[0], axis, from_device=True)
        assert np.array_equal(c.view(np.uint32), otabs[axis][0].view(np.uint32))
        assert np.array_equal(s.view(np.uint32), otabs[axis][1].view(np.uint32))
    for h in handles:
        h.close()


def test_evicted_tables_stay_usable():
    r.rope3d_cache_clear()
    first = r.rope3d_build_tables(2, 4, 4, (16, 16, 16))
    others = [r.rope3d_build_tables(2, 4, 5 + i, (16, 16, 16)) for i in range(16)]
    assert r.rope3d_cache_stats()["evictions"] == 1
    w = synthetic.WORKLOADS["tiny"]
    q_np, k_np = synthetic.qk(w)
    shp = (w.B, w.N, w.heads, w.head_dim)
    qo, ko = r.rope3d_apply_pair(to_device(q_np, shp, "bf16"), to_device(k_np, shp, "bf16"), first)
    want_q, want_k = oracle_full(q_np, k_np, w.shape6, w.split)
    assert_bit_exact(to_numpy(qo), want_q, "Q")
    assert_bit_exact(to_numpy(ko), want_k, "K")
    for t in [first] + others:
        t.close()


def test_runs_on_a_side_stream():
    w = synthetic.WORKLOADS["stage0"]
    q_np, k_np = synthetic.qk(w)
    shp = (w.B, w.N, w.heads, w.head_dim)
    tabs = r.rope3d_build_tables(w.T, w.H, w.W, w.split)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        q, k = to_device(q_np, shp, "bf16"), to_device(k_np, shp, "bf16")
        qo, ko = r.rope3d_apply_pair(q, k, tabs)  # launches on the current (side) stream
        res_q, res_k = to_numpy(qo), to_numpy(ko)
    want_q, want_k = oracle_full(q_np, k_np, w.shape6, w.split)
    assert_bit_exact(res_q, want_q, "Q")
    assert_bit_exact(res_k, want_k, "K")
    tabs.close()


# ---------------------------------------------------------------------------
# host buffers
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,pinned", [("stage5_w63", True), ("stage0_f32", False), ("tiny", True)])
def test_host_buffers_bit_exact(name, pinned):
    w = synthetic.WORKLOADS[name]
    np_dt = np.uint16 if w.dtype == "bf16" else np.float32
    if pinned:
        bufs = [torch.empty(w.numel * w.elem_bytes, dtype=torch.uint8).pin_memory() for _ in range(4)]
        q_np, k_np, qo_np, ko_np = (b.numpy().view(np_dt) for b in bufs)
        synthetic.qk(w, q_np, k_np)
    else:
        q_np, k_np = synthetic.qk(w)
        qo_np, ko_np = np.empty_like(q_np), np.empty_like(k_np)
    shp = (w.B, w.N, w.heads, w.head_dim)
    tabs = r.rope3d_build_tables(w.T, w.H, w.W, w.split)
    r.rope3d_apply_pair_host(q_np.reshape(shp), k_np.reshape(shp), qo_np.reshape(shp),
                             ko_np.reshape(shp), tabs)
    dt = r.BF16 if w.dtype == "bf16" else r.F32
    assert r.rope3d_gate_verdict(w.B, w.T, w.H, w.W, w.heads, w.head_dim, w.split, w.base, dt) == 1
    want_q, want_k = oracle_full(q_np, k_np, w.shape6, w.split)
    assert_bit_exact(qo_np, want_q, "Q")
    assert_bit_exact(ko_np, want_k, "K")
    # device memory is refused by the host entry point
    qd = to_device(q_np, shp, w.dtype)
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_apply_pair_host(qd, qd, torch.empty_like(qd), torch.empty_like(qd), tabs)
    assert e.value.name == "ERR_DEVICE"
    tabs.close()
