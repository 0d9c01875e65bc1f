"""Host-side tests of the library that need no GPU: the C ABI exports, the
table builder (bitwise against the oracle), the index-decode division, the
preflight rules, the table cache's FIFO and reference counting, and the gate's
bookkeeping."""
from __future__ import annotations

import ctypes
import json
import os
import re

import numpy as np
import pytest

import oracle
import rope_rope3d_apply_gb300 as r

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from rope_rope3d_apply_gb300 import build

    build.build()
    return r.load_library()


@pytest.fixture
def host_tables(lib):
    """The cache in its host-memory test mode (no GPU needed)."""
    r.rope3d_cache_clear()
    r.rope3d_testing_host_tables(True)
    yield
    r.rope3d_cache_clear()
    r.rope3d_testing_host_tables(False)


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(rope3d_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 20
    raw = ctypes.CDLL(r.LIB_PATH)
    missing = [n for n in names if not hasattr(raw, n)]
    assert not missing, missing
    assert lib.rope3d_abi_version() == 1


def test_status_strings(lib):
    for code, name in r.STATUS.items():
        s = r.rope3d_status_string(code)
        assert name in s.replace("ROPE3D_", ""), (code, s)
    assert "unknown" in r.rope3d_status_string(-99)


@pytest.mark.parametrize("length,dim,base", [
    (2, 16, 10000.0), (4, 16, 10000.0), (16, 24, 10000.0), (24, 32, 10000.0),
    (96, 48, 10000.0), (64, 48, 10000.0), (63, 48, 10000.0), (1, 2, 10000.0),
    (1000, 128, 10000.0), (7, 10, 3.5), (50, 64, 1e6),
])
def test_axis_table_matches_oracle_bitwise(lib, length, dim, base):
    c, s = r.rope3d_axis_table_host(length, dim, base)
    oc, os_ = oracle.axis_table(length, dim, base)
    assert np.array_equal(c.view(np.uint32), oc.view(np.uint32))
    assert np.array_equal(s.view(np.uint32), os_.view(np.uint32))


def test_axis_table_rejects(lib):
    for length, dim, base in [(0, 16, 1e4), (4, 15, 1e4), (4, 0, 1e4)]:
        with pytest.raises(r.Rope3dError) as e:
            r.rope3d_axis_table_host(length, dim, base)
        assert e.value.name == "ERR_SHAPE"
    for base in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(r.Rope3dError) as e:
            r.rope3d_axis_table_host(4, 16, base)
        assert e.value.name == "ERR_ARG"


def test_fastdiv_is_exact(lib):
    g = np.random.Generator(np.random.PCG64(7))
    divisors = [1, 2, 3, 5, 7, 16, 48, 63, 64, 96, 384, 9216, 65536, 221184, 442368,
                (1 << 31) - 1, (1 << 30) + 1, 1 << 30]
    divisors += [int(d) for d in g.integers(1, 1 << 31, 200)]
    for d in divisors:
        ns = [0, 1, d - 1, d, d + 1, (1 << 31) - 1, (1 << 31) - 2, 2 * d - 1, 2 * d]
        ns += [int(n) for n in g.integers(0, 1 << 31, 200)]
        for n in ns:
            if 0 <= n < (1 << 31):
                assert r.rope3d_testing_fastdiv(n, d) == n // d, (n, d)
    assert r.rope3d_testing_fastdiv(1 << 31, 3) == -1
    assert r.rope3d_testing_fastdiv(5, 0) == -1


def _preflight_case(case, base, handles):
    cfg = dict(base)
    cfg.update(case["changes"])
    elem = 4 if cfg["dtype"] == 1 else 2
    numel = max(0, cfg["B"] * cfg["T"] * cfg["H"] * cfg["W"] * cfg["heads"] * cfg["head_dim"])
    span = max(numel * elem, 1) + (1 << 20)
    ptrs = {"q": 1 << 32, "k": (1 << 32) + span, "q_out": (1 << 32) + 2 * span,
            "k_out": (1 << 32) + 3 * span}
    for name in ("q", "k", "q_out", "k_out"):
        v = case["changes"].get(name, "keep")
        if v is None:
            ptrs[name] = 0
        elif isinstance(v, str) and v != "keep":
            ref, _, off = v.partition("+")
            ptrs[name] = ptrs[ref] + int(off or 0)
        ptrs[name] += case["changes"].get(name + "_offset", 0)
    tab = cfg.get("tables")
    handle = None if tab is None else handles[(tab[0], tab[1], tab[2], tuple(tab[3]))]
    return r.rope3d_preflight(ptrs["q"], ptrs["k"], ptrs["q_out"], ptrs["k_out"], handle,
                              cfg["B"], cfg["T"], cfg["H"], cfg["W"], cfg["heads"],
                              cfg["head_dim"], cfg["split"], cfg["dtype"], check_device=False)


def test_preflight_rules_from_the_pages(lib, host_tables):
    spec = json.load(open(os.path.join(ROOT, "tests", "golden", "preflight_cases.json")))
    handles = {}
    for case in [spec["base_case"]] + [dict(spec["base_case"], **c["changes"]) for c in spec["cases"]]:
        tab = case.get("tables")
        if tab is not None:
            key = (tab[0], tab[1], tab[2], tuple(tab[3]))
            if key not in handles:
                handles[key] = r.rope3d_build_tables(*key[:3], key[3], 10000.0)
    for case in spec["cases"]:
        got = _preflight_case(case, spec["base_case"], handles)
        assert r.STATUS[got] == case["status"], (case["name"], r.STATUS[got])
    for h in handles.values():
        h.close()


def test_cache_fifo_refcount_and_key(lib, host_tables):
    split = (16, 16, 16)
    first = r.rope3d_build_tables(1, 1, 1, split)
    held = [first]
    for i in range(2, 17):
        held.append(r.rope3d_build_tables(i, 1, 1, split))
    st = r.rope3d_cache_stats()
    assert st == {"entries": 16, "hits": 0, "misses": 16, "evictions": 0}
    # a hit returns the same entry and does not refresh its age
    again = r.rope3d_build_tables(1, 1, 1, split)
    assert again.handle == first.handle
    assert r.rope3d_cache_stats()["hits"] == 1
    # the 17th entry evicts the oldest (grid 1x1x1) ...
    held.append(r.rope3d_build_tables(17, 1, 1, split))
    st = r.rope3d_cache_stats()
    assert st["entries"] == 16 and st["evictions"] == 1
    # ... whose handles stay valid while held
    c, s = r.rope3d_tables_read(first, 0, from_device=True)
    assert c.shape == (1, 8) and np.all(c == 1.0) and np.all(s == 0.0)
    # building it again is a miss and a different entry
    fresh = r.rope3d_build_tables(1, 1, 1, split)
    assert fresh.handle != first.handle
    assert r.rope3d_cache_stats()["misses"] == 18
    # the key includes the split and the base
    a = r.rope3d_build_tables(2, 4, 4, (16, 16, 16), 10000.0)
    b = r.rope3d_build_tables(2, 4, 4, (16, 8, 24), 10000.0)
    c_ = r.rope3d_build_tables(2, 4, 4, (16, 16, 16), 500.0)
    assert len({a.handle, b.handle, c_.handle}) == 3
    for t in held + [again, fresh, a, b, c_]:
        t.close()


def test_cached_tables_match_oracle(lib, host_tables):
    for T, H, W, split in [(24, 96, 96, (32, 48, 48)), (16, 64, 63, (32, 48, 48)), (3, 5, 7, (4, 6, 8))]:
        t = r.rope3d_build_tables(T, H, W, split)
        otabs = oracle.tables(T, H, W, split)
        for axis in range(3):
            for dev in (False, True):
                c, s = r.rope3d_tables_read(t, axis, from_device=dev)
                assert np.array_equal(c.view(np.uint32), otabs[axis][0].view(np.uint32))
                assert np.array_equal(s.view(np.uint32), otabs[axis][1].view(np.uint32))
        t.close()


def test_gate_bookkeeping_without_gpu(lib, host_tables):
    r.rope3d_gate_reset()
    assert r.rope3d_gate_get_mode() == r.GATE_FIRST
    assert r.rope3d_gate_verdict(1, 2, 4, 4, 2, 48, (16, 16, 16), 10000.0, r.BF16) == 0
    r.rope3d_gate_set_mode(r.GATE_OFF)
    assert r.rope3d_gate_get_mode() == r.GATE_OFF
    r.rope3d_gate_set_mode(r.GATE_FIRST)
    with pytest.raises(r.Rope3dError):
        r.rope3d_gate_set_mode(7)
    with pytest.raises(r.Rope3dError):
        r.rope3d_testing_corrupt_gate(-1)


def test_build_tables_rejects(lib, host_tables):
    for args, name in [((0, 4, 4, (16, 16, 16)), "ERR_SHAPE"), ((2, 4, 4, (15, 17, 16)), "ERR_SHAPE"),
                       ((2, 4, 4, (0, 24, 24)), "ERR_SHAPE"), ((1 << 20, 1 << 11, 2, (2, 2, 2)), "ERR_SHAPE")]:
        with pytest.raises(r.Rope3dError) as e:
            r.rope3d_build_tables(*args)
        assert e.value.name == name
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_build_tables(2, 4, 4, (16, 16, 16), -1.0)
    assert e.value.name == "ERR_ARG"


# ---------------------------------------------------------------------------
# strided views: the overlap analysis of rope3d_apply_pair_strided
# ---------------------------------------------------------------------------

def _contig_strides(B, T, H, W, heads, hd):
    return (T * H * W * heads * hd, H * W * heads * hd, W * heads * hd, heads * hd, hd)


def _status(ptrs, strides, tables, dims, split=(16, 16, 16), dtype=0):
    B, T, H, W, heads, hd = dims
    return r.STATUS[r.rope3d_preflight_strided(ptrs, strides, tables, B, T, H, W, heads, hd,
                                               split, dtype, check_device=False)]


def test_strided_fused_qkv_layouts(lib, host_tables):
    dims = (2, 2, 4, 4, 3, 48)
    B, T, H, W, heads, hd = dims
    N = T * H * W
    tabs = r.rope3d_build_tables(T, H, W, (16, 16, 16))
    base = 1 << 32
    far = 1 << 40
    out = _contig_strides(*dims)
    # [B, N, 3, heads, hd]: Q, K, V thirds
    s3 = (N * 3 * heads * hd, H * W * 3 * heads * hd, W * 3 * heads * hd, 3 * heads * hd, hd)
    q, k, v = base, base + 2 * heads * hd, base + 4 * heads * hd
    assert _status((q, k, far, far + (1 << 30)), (s3, s3, out, out), tabs, dims) == "OK"
    assert _status((q, k, q, k), (s3, s3, s3, s3), tabs, dims) == "OK"            # in place
    assert _status((q, k, v, far), (s3, s3, s3, out), tabs, dims) == "OK"         # Q_out into V
    assert _status((q, k, k, far), (s3, s3, s3, out), tabs, dims) == "ERR_ALIAS"  # Q_out onto K
    assert _status((q, k, v, v), (s3, s3, s3, s3), tabs, dims) == "ERR_ALIAS"     # outputs collide
    assert _status((q, k, q + 4, k), (s3, s3, s3, s3), tabs, dims) == "ERR_ALIAS"  # off by two elements
    # [B, N, heads, 3, hd]: interleaved per head
    si = (N * heads * 3 * hd, H * W * heads * 3 * hd, W * heads * 3 * hd, heads * 3 * hd, 3 * hd)
    q, k = base, base + 2 * hd
    assert _status((q, k, q, k), (si, si, si, si), tabs, dims) == "OK"
    assert _status((q, k, k, q), (si, si, si, si), tabs, dims) == "ERR_ALIAS"     # swapped
    tabs.close()


def test_strided_rejections(lib, host_tables):
    dims = (1, 2, 4, 4, 2, 48)
    tabs = r.rope3d_build_tables(2, 4, 4, (16, 16, 16))
    c = _contig_strides(*dims)
    p = (1 << 32, 1 << 34, 1 << 36, 1 << 38)
    assert _status(p, (c, c, c, c), tabs, dims) == "OK"
    bcast = (c[0], c[1], c[2], c[3], 0)  # two heads written to one place
    assert _status(p, (c, c, bcast, c), tabs, dims) == "ERR_ALIAS"
    assert _status(p, (c, c, c, (c[0], c[1], -c[2], c[3], c[4])), tabs, dims) == "ERR_SHAPE"
    odd = (c[0], c[1], c[2], c[3], 49)
    assert _status(p, (odd, c, c, c), tabs, dims) == "ERR_ALIGN"
    assert _status(p, (odd, c, c, c), tabs, dims, dtype=1) == "OK"  # fp32 pairs need no even stride
    assert _status(p, (None, c, c, c), tabs, dims) == "ERR_NULL"
    assert _status((p[0] + 2, p[1], p[2], p[3]), (c, c, c, c), tabs, dims) == "ERR_ALIGN"
    # a crop of a larger grid, and another crop of the same buffer
    big = (1 * 4 * 8 * 8 * 2 * 48, 8 * 8 * 2 * 48, 8 * 2 * 48, 2 * 48, 48)
    b0 = 1 << 32
    crop_a = b0
    crop_b = b0 + 2 * (4 * 2 * 48)             # 4 columns to the right: disjoint
    crop_c = b0 + 2 * (2 * 2 * 48)             # 2 columns to the right: overlaps crop_a
    assert _status((crop_a, p[1], crop_b, p[3]), (big, c, big, c), tabs, dims) == "OK"
    assert _status((crop_a, p[1], crop_c, p[3]), (big, c, big, c), tabs, dims) == "ERR_ALIAS"
    tabs.close()


def _elements(base, shape, strides):
    idx = np.indices(shape).reshape(len(shape), -1)
    return set((base + (idx * np.array(strides)[:, None]).sum(axis=0)).tolist())


def test_strided_overlap_matches_brute_force(lib, host_tables):
    """For outputs with identical strides, ERR_ALIAS exactly when the two
    views share an element (enumerated)."""
    g = np.random.Generator(np.random.PCG64(21))
    tabs = {}
    checked = alias = 0
    while checked < 300:
        B, T, H, W, heads = (int(v) for v in g.integers(1, 4, 5))
        hd = int(g.choice([6, 12]))
        split = (2, 2, hd - 4)
        key = (T, H, W, split)
        if key not in tabs:
            tabs[key] = r.rope3d_build_tables(T, H, W, split)
        shape = (B, T, H, W, heads, hd)
        strides = tuple(int(v) * 2 for v in g.integers(0, 40, 5)) + (1,)
        # only non-self-overlapping output views (else the call is refused anyway)
        if len(_elements(0, shape, strides)) != int(np.prod(shape)):
            continue
        off = int(g.integers(-300, 300)) * 2
        ob = 1 << 32
        st5 = strides[:5]
        got = _status((1 << 44, 1 << 45, ob, ob + 2 * off), ((0,) * 4 + (hd,), (0,) * 4 + (hd,), st5, st5),
                      tabs[key], shape, split)
        want = "ERR_ALIAS" if _elements(0, shape, strides) & _elements(off, shape, strides) else "OK"
        assert got == want, (shape, strides, off)
        checked += 1
        alias += want == "ERR_ALIAS"
    assert 30 < alias < 270  # both outcomes exercised
    for t in tabs.values():
        t.close()


def test_patchify_host_checks(lib):
    P = 1 << 32
    Q = 1 << 36
    ok = (P, Q, 1, 3, 2, 8, 8, 4, 2)
    assert r.rope3d_patchify_check(*ok) == "OK"
    cases = {
        "ERR_NULL": (0, Q, 1, 3, 2, 8, 8, 4, 2),
        "ERR_DTYPE": (P, Q, 1, 3, 2, 8, 8, 4, 3),
        "ERR_SHAPE": (P, Q, 1, 3, 2, 8, 6, 4, 2),      # W not a multiple of p
        "ERR_ALIGN": (P + 1, Q, 1, 3, 2, 8, 8, 4, 2),
        "ERR_ALIAS": (P, P + 64, 1, 3, 2, 8, 8, 4, 2),
    }
    for want, args in cases.items():
        assert r.rope3d_patchify_check(*args) == want, want
    assert r.rope3d_patchify_check(P, Q, 1, 3, 2, 8, 8, 0, 2) == "ERR_SHAPE"
    assert r.rope3d_patchify_check(P, Q, 1, 3, 2, 9, 9, 3, 1) == "OK"


def test_na3d_host_checks(lib, host_tables):
    """The argument checks of rope3d_na3d and rope3d_na3d_rotate_once without
    a GPU: tables in host memory, addresses that are never dereferenced."""
    T, H, W, heads = 3, 8, 8, 2
    tabs = r.rope3d_build_tables(T, H, W, (32, 48, 48))
    base, step = 1 << 32, 1 << 24     # tensors of 98,304 bytes, far apart
    q, k, v, kr, out = (base + i * step for i in range(5))

    def chk(*a, **kw):
        return r.rope3d_na3d_preflight(*a, check_device=False, **kw)

    args = (tabs, 1, T, H, W, heads, (3, 3, 3))
    assert chk(q, k, v, None, out, *args) == "OK"
    assert chk(q, k, v, kr, out, *args) == "OK"
    assert chk(q, k, v, k, out, *args) == "OK"                      # K rotated in place
    assert chk(q, k, v, None, out, None, 1, T, H, W, heads, (3, 3, 3), apply_rope=False) == "OK"
    # pointers
    assert chk(0, k, v, None, out, *args) == "ERR_NULL"
    assert chk(q, k, v, None, 0, *args) == "ERR_NULL"
    assert chk(q, k, v, None, out, None, 1, T, H, W, heads, (3, 3, 3),
               split=(32, 48, 48)) == "ERR_NULL"                   # rotation without tables
    assert chk(q + 8, k, v, None, out, *args) == "ERR_ALIGN"
    assert chk(q, k, v, kr + 8, out, *args) == "ERR_ALIGN"
    # overlaps: out with an input; k_rot with anything but exactly k
    assert chk(q, k, v, None, q + 4096, *args) == "ERR_ALIAS"
    for bad in (q, v, out, k + 4096, k - 4096):
        assert chk(q, k, v, bad, out, *args) == "ERR_ALIAS", bad - base
    # Q may share K's memory (both only read), but not when K is rotated in place
    assert chk(k, k, v, kr, out, *args) == "OK"
    assert chk(k, k, v, None, out, *args) == "OK"
    assert chk(k, k, v, k, out, *args) == "ERR_ALIAS"
    assert chk(k + 4096, k, v, k, out, *args) == "ERR_ALIAS"
    assert chk(q, k, k + 4096, k, out, *args) == "ERR_ALIAS"     # V inside K, K rotated in place
    # windows and sizes
    assert chk(q, k, v, None, out, tabs, 1, T, H, W, heads, (2, 3, 3)) == "ERR_SHAPE"   # even
    assert chk(q, k, v, None, out, tabs, 1, T, H, W, heads, (5, 3, 3)) == "ERR_SHAPE"   # > T
    assert chk(q, k, v, None, out, *args, head_dim=64) == "ERR_SHAPE"
    # the tables' key, and chunks the kernel's 16-byte vectors cannot take
    assert chk(q, k, v, None, out, tabs, 1, T, H + 1, W, heads, (3, 3, 3)) == "ERR_TABLES"
    odd = r.rope3d_build_tables(T, H, W, (36, 44, 48))
    assert chk(q, k, v, kr, out, odd, 1, T, H, W, heads, (3, 3, 3)) == "ERR_SHAPE"
    odd.close()
    tabs.close()


def test_neox_cache_matches_oracle_bitwise(lib):
    for max_pos, d, base in [(64, 16, 10000.0), (4096, 256, 10000.0), (33, 6, 1e6)]:
        got = r.rope3d_neox_cache_host(max_pos, d, base)
        want = oracle.neox_cache(max_pos, d, base)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_neox_host_checks(lib):
    base = 1 << 32
    step = 1 << 28
    ptrs = [base + i * step for i in range(7)]
    ok = (4096, 100, 8, 4, 256, r.BF16)
    assert r.rope3d_neox_check(ptrs, *ok) == "OK"
    inplace = ptrs[:2] + ptrs[:2] + ptrs[4:]
    assert r.rope3d_neox_check(inplace, *ok) == "OK"
    swapped = ptrs[:2] + [ptrs[1], ptrs[0]] + ptrs[4:]
    assert r.rope3d_neox_check(swapped, *ok) == "ERR_ALIAS"
    onto_cache = ptrs[:2] + [ptrs[5], ptrs[3]] + ptrs[4:]
    assert r.rope3d_neox_check(onto_cache, *ok) == "ERR_ALIAS"
    # Q and K may share memory (both only read) unless one is rotated in place
    same = [ptrs[0], ptrs[0]] + ptrs[2:]
    assert r.rope3d_neox_check(same, 4096, 100, 8, 8, 256, r.BF16) == "OK"
    q_in_place_over_k = [ptrs[0], ptrs[0], ptrs[0]] + ptrs[3:]
    assert r.rope3d_neox_check(q_in_place_over_k, 4096, 100, 8, 8, 256, r.BF16) == "ERR_ALIAS"
    k_in_place_over_q = [ptrs[0], ptrs[0], ptrs[2], ptrs[0]] + ptrs[4:]
    assert r.rope3d_neox_check(k_in_place_over_q, 4096, 100, 8, 8, 256, r.BF16) == "ERR_ALIAS"
    assert r.rope3d_neox_check(ptrs, 4096, 100, 8, 4, 255, r.BF16) == "ERR_SHAPE"
    assert r.rope3d_neox_check(ptrs, 4096, 0, 8, 4, 256, r.BF16) == "ERR_SHAPE"
    assert r.rope3d_neox_check(ptrs, 4096, 100, 8, 4, 256, 7) == "ERR_DTYPE"
    bad = list(ptrs)
    bad[4] += 4    # positions must be 8-byte aligned
    assert r.rope3d_neox_check(bad, *ok) == "ERR_ALIGN"
    nul = list(ptrs)
    nul[5] = 0
    assert r.rope3d_neox_check(nul, *ok) == "ERR_NULL"
    no_counter = ptrs[:6] + [0]
    assert r.rope3d_neox_check(no_counter, *ok) == "OK"


def test_normal_build_has_no_bound_checks(lib):
    """The normal build compiles the debug bounds checks away and says so."""
    if os.environ.get("ROPE3D_LIB"):
        pytest.skip("a different build was named")
    assert r.rope3d_debug_bounds() == (False, 0)


def test_noalloc_binding_checks_extents_and_dtypes_before_the_call(lib):
    """The C ABI takes bare pointers, so the binding's checks are what keep a
    call inside the caller's buffers: a grid that does not match the buffers'
    shape, or an output dtype other than q's, raises before any library call."""
    shp6 = (1, 2, 4, 4, 2, 48)
    q = np.zeros(shp6, np.uint16)
    k, qo, ko = q.copy(), q.copy(), q.copy()
    with pytest.raises(ValueError):
        r.rope3d_apply_pair_noalloc(q, k, qo, ko, 2, 4, 8, (16, 16, 16))
    with pytest.raises(ValueError):
        r.rope3d_apply_pair_noalloc(q.reshape(1, 32, 2, 48), k.reshape(1, 32, 2, 48),
                                    qo.reshape(1, 32, 2, 48), ko.reshape(1, 32, 2, 48),
                                    2, 4, 2, (16, 16, 16))
    with pytest.raises(TypeError):
        r.rope3d_apply_pair_noalloc(q.astype(np.float32), k.astype(np.float32), qo, ko,
                                    2, 4, 4, (16, 16, 16))
    with pytest.raises(ValueError):
        r.rope3d_apply_pair_noalloc(q, k, qo[:, :1], ko, 2, 4, 4, (16, 16, 16))


@pytest.mark.parametrize("double_precision", [True, False])
@pytest.mark.parametrize("dim,elems,theta", [
    (4096, 6, 10000.0), (2048, 2, 10000.0), (128, 6, 10000.0), (3072, 6, 10000.0),
    (96, 6, 1.0e6), (60, 6, 2.5), (12, 6, 10000.0), (6, 6, 10000.0), (7, 6, 10000.0),
    (1 << 20, 6, 10000.0), (60, 6, 1.0),
])
def test_dit_freqs_match_oracle_bitwise(lib, dim, elems, theta, double_precision):
    got = r.rope3d_dit_freqs_host(dim, elems, theta, double_precision)
    want = oracle.dit_rope_freqs(dim, elems, theta, double_precision)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_dit_freqs_rejects(lib):
    for args, name in [((5, 6, 1e4), "ERR_SHAPE"), ((12, 0, 1e4), "ERR_SHAPE"),
                       ((12, 6, 0.0), "ERR_ARG"), ((12, 6, float("nan")), "ERR_ARG"),
                       ((12, 6, -3.0), "ERR_ARG")]:
        with pytest.raises((r.Rope3dError, ValueError)) as e:
            r.rope3d_dit_freqs_host(*args)
        if isinstance(e.value, r.Rope3dError):
            assert e.value.name == name, args
    assert lib.rope3d_dit_freqs_host(12, 6, 1e4, 1, None) == -1


def test_released_host_tables_are_freed_at_once(lib, host_tables):
    """Host-memory test tables have no launches to wait for: eviction and
    release free them on the spot."""
    first = r.rope3d_build_tables(2, 4, 4, (16, 16, 16))
    others = [r.rope3d_build_tables(2, 4, 5 + i, (16, 16, 16)) for i in range(16)]
    assert r.rope3d_cache_stats()["evictions"] == 1
    first.close()
    assert r.rope3d_cache_retired() == 0
    for t in others:
        t.close()
    r.rope3d_cache_clear()
    assert r.rope3d_cache_retired() == 0
