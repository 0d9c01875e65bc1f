"""Pins for the patchify / unpatchify oracle (sglang PR #34471 review,
"关键源码片段", _patchify): checked against an element-by-element loop written
from the stated channel order (channel, width offset, height offset), a hand
example, and the round trip."""
from __future__ import annotations

import itertools

import numpy as np
import pytest

import oracle


def loop_patchify(x, p):
    B, C, F, H, W = x.shape
    y = np.empty((B, C * p * p, F, H // p, W // p), x.dtype)
    for b, c, f, h, w in itertools.product(range(B), range(C), range(F), range(H), range(W)):
        i, ph = divmod(h, p)
        j, pw = divmod(w, p)
        y[b, c * p * p + pw * p + ph, f, i, j] = x[b, c, f, h, w]
    return y


@pytest.mark.parametrize("shape,p", [((1, 1, 1, 2, 2), 2), ((2, 3, 2, 4, 6), 2), ((1, 2, 3, 6, 9), 3),
                                     ((2, 1, 2, 8, 4), 4), ((1, 2, 1, 3, 5), 1)])
def test_patchify_matches_loop(shape, p):
    x = np.arange(int(np.prod(shape)), dtype=np.int32).reshape(shape)
    assert np.array_equal(oracle.patchify(x, p), loop_patchify(x, p))
    assert np.array_equal(oracle.unpatchify(oracle.patchify(x, p), p), x)


def test_patchify_hand_example():
    # one channel, one frame, a 2x2 image [[a, b], [c, d]] with p = 2: channel
    # index = w_off * 2 + h_off, so the four channels hold a, c, b, d
    x = np.array([10, 11, 12, 13], np.int32).reshape(1, 1, 1, 2, 2)   # a=10 b=11 c=12 d=13
    y = oracle.patchify(x, 2)
    assert y.shape == (1, 4, 1, 1, 1)
    assert y.reshape(-1).tolist() == [10, 12, 11, 13]


def test_unpatchify_is_inverse_on_random_bits():
    g = np.random.Generator(np.random.PCG64(70))
    y = g.integers(0, 1 << 16, (2, 3 * 16, 2, 3, 5), dtype=np.uint16)
    assert np.array_equal(oracle.patchify(oracle.unpatchify(y, 4), 4), y)


def test_patchify_rejects_ragged():
    with pytest.raises(ValueError):
        oracle.patchify(np.zeros((1, 1, 1, 3, 4)), 2)
