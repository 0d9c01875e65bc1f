"""Pins for the neighbourhood-attention oracle: a pure-Python loop written
from the published definition (window centred on the query, shifted inside
the grid), the closed forms of the two extreme windows (a 1x1x1 window
returns V; a window as large as the grid is full softmax attention), the
border rule on a hand example, and the one-query-at-a-time form against the
full pass. The last test plants mistakes in a copy of the oracle and checks
that some pin catches each one."""
from __future__ import annotations

import importlib.util
import itertools
import math
import os

import numpy as np
import pytest

import oracle


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def loop_na3d(q, k, v, shape, kernel):
    B, T, H, W, heads, d = shape
    out = np.zeros(shape)
    for b, t, h, w, e in itertools.product(range(B), range(T), range(H), range(W), range(heads)):
        lo = []
        for i, L, kk in ((t, T, kernel[0]), (h, H, kernel[1]), (w, W, kernel[2])):
            s = i - kk // 2
            s = 0 if s < 0 else s
            s = L - kk if s + kk > L else s
            lo.append(s)
        keys = [(a, bb, c) for a in range(lo[0], lo[0] + kernel[0])
                for bb in range(lo[1], lo[1] + kernel[1]) for c in range(lo[2], lo[2] + kernel[2])]
        sc = [sum(q[b, t, h, w, e, x] * k[b, a, bb, c, e, x] for x in range(d)) / math.sqrt(d)
              for a, bb, c in keys]
        m = max(sc)
        ex = [math.exp(s - m) for s in sc]
        z = sum(ex)
        for x in range(d):
            out[b, t, h, w, e, x] = sum(p * v[b, a, bb, c, e, x] for p, (a, bb, c) in zip(ex, keys)) / z
    return out


LOOP_CASES = [((1, 3, 4, 5, 2, 4), (3, 3, 3)), ((2, 2, 5, 3, 1, 6), (1, 3, 3)),
              ((1, 4, 3, 6, 1, 2), (3, 1, 5))]


# The pins as functions of an oracle module, so that the planted-mistake test
# can run them against a mutated copy.
def pin_na_matches_loop(o):
    for shape, kernel in LOOP_CASES:
        g = _rng(sum(shape))
        q, k, v = (g.standard_normal(shape) for _ in range(3))
        assert np.allclose(o.na3d(q, k, v, shape, kernel), loop_na3d(q, k, v, shape, kernel),
                           rtol=1e-12, atol=1e-12)


def pin_na_extreme_windows(o):
    shape = (2, 3, 5, 5, 2, 8)
    g = _rng(7)
    q, k, v = (g.standard_normal(shape) for _ in range(3))
    # a single-key window: each query returns its own V
    assert np.array_equal(o.na3d(q, k, v, shape, (1, 1, 1)), v)
    # a window as large as the grid: full softmax attention per (batch, head)
    full = o.na3d(q, k, v, shape, (3, 5, 5))
    N = 3 * 5 * 5
    for b in range(2):
        for e in range(2):
            Q = q[b, ..., e, :].reshape(N, 8)
            K = k[b, ..., e, :].reshape(N, 8)
            V = v[b, ..., e, :].reshape(N, 8)
            S = Q @ K.T / math.sqrt(8)
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            assert np.allclose(full[b, ..., e, :].reshape(N, 8), P @ V, rtol=1e-12, atol=1e-12)


def pin_na_border_rule(o):
    # length 6, kernel 3: starts 0,0,1,2,3,3 (shifted inward at both ends)
    assert o.na_window_starts(6, 3).tolist() == [0, 0, 1, 2, 3, 3]
    # length 5, kernel 5: the window is the whole axis for every query
    assert o.na_window_starts(5, 5).tolist() == [0, 0, 0, 0, 0]
    with pytest.raises(ValueError):
        o.na3d(np.zeros(24), np.zeros(24), np.zeros(24), (1, 2, 3, 4, 1, 1), (3, 3, 3))


def pin_na_single_query(o, shape=(2, 3, 6, 7, 2, 16), nq=None):
    """rope_na3d_at (one query at a time, element-by-element rotation) gives
    the full pass's outputs, and its |v| sums are the full pass on |v|; so the
    sampled checks at full size rest on the same pins as the full pass."""
    B, T, H, W, heads, d = shape
    split, kernel = (4, 6, 6), (3, 3, 5)
    g = _rng(11)
    n = int(np.prod(shape))
    to_bits = lambda a: (a.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)  # noqa: E731
    q, k, v = (to_bits(g.normal(size=n)) for _ in range(3))
    lib = oracle.load()
    tabs = oracle.tables(T, H, W, split)
    full = o.rope_na3d(q, k, v, shape, split, tabs, kernel, lib=lib)
    qr = oracle.rope3d(q, shape, split, tabs)
    kr = oracle.rope3d(k, shape, split, tabs)
    to64 = lambda b: (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)  # noqa: E731
    full_abs = o.na3d(to64(qr), to64(kr), np.abs(to64(v)), shape, kernel)
    queries = list(itertools.product(range(B), range(T), range(H), range(W), range(heads)))[:nq]
    out, absv = o.rope_na3d_at(q, k, v, shape, split, tabs, kernel, queries, lib=lib)
    ref = np.array([full[b, t, h, w, e] for b, t, h, w, e in queries])
    ref_abs = np.array([full_abs[b, t, h, w, e] for b, t, h, w, e in queries])
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-14)
    assert np.allclose(absv, ref_abs, rtol=1e-12, atol=1e-14)
    # without the rotation it is plain neighbourhood attention
    out0, _ = o.rope_na3d_at(q, k, v, shape, split, tabs, kernel, queries[:40], rope=False, lib=lib)
    plain = o.na3d(to64(q), to64(k), to64(v), shape, kernel)
    assert np.allclose(out0, [plain[x] for x in queries[:40]], rtol=1e-12, atol=1e-14)
    # the full pass against the loop written from the definition
    assert np.allclose(full, loop_na3d(to64(qr).reshape(shape), to64(kr).reshape(shape),
                                       to64(v).reshape(shape), shape, kernel),
                       rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shape,kernel", LOOP_CASES)
def test_na3d_matches_loop(shape, kernel):
    g = _rng(sum(shape))
    q, k, v = (g.standard_normal(shape) for _ in range(3))
    assert np.allclose(oracle.na3d(q, k, v, shape, kernel), loop_na3d(q, k, v, shape, kernel),
                       rtol=1e-12, atol=1e-12)


def test_na3d_extreme_windows():
    pin_na_extreme_windows(oracle)


def test_border_rule_hand_example():
    pin_na_border_rule(oracle)


def test_single_query_oracle_equals_full_pass():
    pin_na_single_query(oracle)


# planted mistakes: each mutation of the oracle's attention code must fail a pin
MUTATIONS = {
    "window_off_centre": ("np.minimum(np.maximum(i - k // 2, 0), length - k)",
                          "np.minimum(np.maximum(i - k // 2 + 1, 0), length - k)"),
    "no_score_scale": ("    scale = 1.0 / np.sqrt(d)\n", "    scale = 1.0\n"),
    "softmax_shift_over_heads": ("s = s - s.max(axis=-1, keepdims=True)",
                                 "s = s - s.max(axis=-2, keepdims=True)"),
    "values_from_keys": ("vv = v[b][kt_idx, kh_idx, kw_idx]", "vv = k[b][kt_idx, kh_idx, kw_idx]"),
    "key_frame_fixed": ("kt_idx = st[:, None, None, None] + dt.reshape(1, 1, 1, -1)",
                        "kt_idx = st[:, None, None, None] + 0 * dt.reshape(1, 1, 1, -1)"),
    "single_query_no_scale": ("s = to64(kv).reshape(len(keys), d) @ to64(qv) / np.sqrt(d)",
                              "s = to64(kv).reshape(len(keys), d) @ to64(qv)"),
    "single_query_drops_a_key": ("for ww in range(sw[w], sw[w] + kw)]",
                                 "for ww in range(sw[w], sw[w] + kw - 1)]"),
}

PINS = [pin_na_matches_loop, pin_na_extreme_windows, pin_na_border_rule,
        lambda o: pin_na_single_query(o, shape=(1, 3, 5, 6, 1, 16), nq=30)]


def _copy_of_oracle(tmp_path, name, old="", new=""):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "__init__.py")).read()
    if old:
        assert src.count(old) == 1, name
        src = src.replace(old, new)
    path = tmp_path / "oracle_copy.py"
    path.write_text(src)
    spec = importlib.util.spec_from_file_location(f"oracle_copy_{name}", path)
    module = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(module)
    return module


def test_pins_pass_on_an_unmutated_copy(tmp_path):
    """The harness itself: an unchanged copy, loaded the same way, passes every pin."""
    copy = _copy_of_oracle(tmp_path, "unmutated")
    for pin in PINS:
        pin(copy)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_na3d_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    mutant = _copy_of_oracle(tmp_path, name, old, new)
    failed = 0
    for pin in PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, IndexError, pytest.fail.Exception):
            failed += 1
    assert failed, f"no pin caught mutation {name}"
