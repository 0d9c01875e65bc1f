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
