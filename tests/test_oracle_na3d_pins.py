"""Pins for the neighbourhood-attention oracle: a pure-Python loop written
from the published definition (window centred on the query, shifted inside
the grid), the closed forms of the two extreme windows (a 1x1x1 window
returns V; a window as large as the grid is full softmax attention), and the
border rule on a hand example."""
from __future__ import annotations

import itertools
import math

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


@pytest.mark.parametrize("shape,kernel", [((1, 3, 4, 5, 2, 4), (3, 3, 3)), ((2, 2, 5, 3, 1, 6), (1, 3, 3)),
                                          ((1, 4, 3, 6, 1, 2), (3, 1, 5))])
def test_na3d_matches_loop(shape, kernel):
    g = _rng(sum(shape))
    q, k, v = (g.standard_normal(shape) for _ in range(3))
    assert np.allclose(oracle.na3d(q, k, v, shape, kernel), loop_na3d(q, k, v, shape, kernel),
                       rtol=1e-12, atol=1e-12)


def test_na3d_extreme_windows():
    shape = (2, 3, 5, 5, 2, 8)
    g = _rng(7)
    q, k, v = (g.standard_normal(shape) for _ in range(3))
    # a single-key window: each query returns its own V
    assert np.array_equal(oracle.na3d(q, k, v, shape, (1, 1, 1)), v)
    # a window as large as the grid: full softmax attention per (batch, head)
    full = oracle.na3d(q, k, v, shape, (3, 5, 5))
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


def test_border_rule_hand_example():
    # length 6, kernel 3: starts 0,0,1,2,3,3 (shifted inward at both ends)
    assert oracle.na_window_starts(6, 3).tolist() == [0, 0, 1, 2, 3, 3]
    # length 5, kernel 5: the window is the whole axis for every query
    assert oracle.na_window_starts(5, 5).tolist() == [0, 0, 0, 0, 0]
    with pytest.raises(ValueError):
        oracle.na3d(np.zeros(24), np.zeros(24), np.zeros(24), (1, 2, 3, 4, 1, 1), (3, 3, 3))


def test_single_query_oracle_equals_full_pass():
    """rope_na3d_at (one query at a time, element-by-element rotation) gives
    the full pass's outputs, and its |v| sums are the full pass on |v|; so the
    sampled checks at full size rest on the same pins as the full pass."""
    B, T, H, W, heads, d = shape = (2, 3, 6, 7, 2, 16)
    split, kernel = (4, 6, 6), (3, 3, 5)
    g = _rng(11)
    n = int(np.prod(shape))
    to_bits = lambda a: (a.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)  # noqa: E731
    q, k, v = (to_bits(g.normal(size=n)) for _ in range(3))
    tabs = oracle.tables(T, H, W, split)
    full = oracle.rope_na3d(q, k, v, shape, split, tabs, kernel)
    qr = oracle.rope3d(q, shape, split, tabs)
    kr = oracle.rope3d(k, shape, split, tabs)
    to64 = lambda b: (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)  # noqa: E731
    full_abs = oracle.na3d(to64(qr), to64(kr), np.abs(to64(v)), shape, kernel)
    queries = list(itertools.product(range(B), range(T), range(H), range(W), range(heads)))
    out, absv = oracle.rope_na3d_at(q, k, v, shape, split, tabs, kernel, queries)
    ref = np.array([full[b, t, h, w, e] for b, t, h, w, e in queries])
    ref_abs = np.array([full_abs[b, t, h, w, e] for b, t, h, w, e in queries])
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-14)
    assert np.allclose(absv, ref_abs, rtol=1e-12, atol=1e-14)
    # without the rotation it is plain neighbourhood attention
    out0, _ = oracle.rope_na3d_at(q, k, v, shape, split, tabs, kernel, queries[:40], rope=False)
    plain = oracle.na3d(to64(q), to64(k), to64(v), shape, kernel)
    assert np.allclose(out0, [plain[x] for x in queries[:40]], rtol=1e-12, atol=1e-14)
