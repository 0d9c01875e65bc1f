"""Pins for the patchify / unpatchify oracle (sglang PR #34471 review,
"关键源码片段", _patchify): checked against an element-by-element loop written
from the stated channel order (channel, width offset, height offset), a hand
example, and the round trip. The last test plants mistakes in a copy of the
oracle and checks that some pin catches each one."""
from __future__ import annotations

import importlib.util
import itertools
import os

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


# planted mistakes: each mutation of the layout steps must fail a pin
def _pins(o):
    for shape, p in [((2, 3, 2, 4, 6), 2), ((1, 2, 3, 6, 9), 3), ((2, 1, 2, 8, 4), 4)]:
        x = np.arange(int(np.prod(shape)), dtype=np.int32).reshape(shape)
        assert np.array_equal(o.patchify(x, p), loop_patchify(x, p))
        assert np.array_equal(o.unpatchify(loop_patchify(x, p), p), x)
    x = np.array([10, 11, 12, 13], np.int32).reshape(1, 1, 1, 2, 2)
    assert o.patchify(x, 2).reshape(-1).tolist() == [10, 12, 11, 13]


MUTATIONS = {
    "height_offset_before_width": ("t = t.transpose(0, 1, 6, 4, 2, 3, 5)",
                                   "t = t.transpose(0, 1, 4, 6, 2, 3, 5)"),
    "patch_split_swapped": ("t = x.reshape(B, C, F, H // p, p, W // p, p)",
                            "t = x.reshape(B, C, F, p, H // p, p, W // p)"),
    "inverse_offsets_swapped": ("t = t.transpose(0, 1, 4, 5, 3, 6, 2)",
                                "t = t.transpose(0, 1, 4, 5, 2, 6, 3)"),
}


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


def test_patchify_pins_pass_on_an_unmutated_copy(tmp_path):
    _pins(_copy_of_oracle(tmp_path, "unmutated"))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_patchify_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    mutant = _copy_of_oracle(tmp_path, name, old, new)
    with pytest.raises((AssertionError, ValueError)):
        _pins(mutant)
