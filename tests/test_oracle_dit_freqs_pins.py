"""Pins for the LTX DiT RoPE frequency-vector oracle (sglang PR #24660 review,
"关键源码片段", ltx_2.py: theta ** linspace(0, 1, dim // num_rope_elems) * pi / 2,
each step in float64 or float32, cast to float32).

Checked against values that do not come from the oracle's own arithmetic:
- the float64 path against the exact frequency theta^(i/(n-1)) * pi / 2 from
  40-digit mpmath, rounded once to float32 (a float64 pipeline with a few
  roundings lands on the same float32 unless the exact value lies within
  2^-45 of a float32 rounding boundary, where either neighbour is accepted);
- the float32 path against an exact-rational model of each binary32 step
  (nearest linspace value, correctly rounded power from mpmath, product with
  the nearest float32 to pi rounded once, exact halving);
- closed forms: the first frequency is pi/2 and the last theta * pi / 2; one
  step gives [pi/2]; theta = 1 gives pi/2 everywhere; the sequence rises for
  theta > 1.
The last test plants mistakes in a copy of the oracle and checks that some
pin catches each one.
"""
from __future__ import annotations

import importlib.util
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests.exact import rn_f32

mpmath = pytest.importorskip("mpmath")

CASES = [(4096, 6, 10000.0), (2048, 2, 10000.0), (128, 6, 10000.0), (3072, 6, 10000.0),
         (96, 6, 1.0e6), (60, 6, 2.5), (12, 6, 10000.0), (6, 6, 10000.0)]


def _fraction(v) -> Fraction:
    """Exact rational value of a 40-digit mpmath number (as a decimal string)."""
    return Fraction(mpmath.nstr(v, 45, strip_zeros=False, min_fixed=-1e9, max_fixed=1e9))


def _allowed_f32(exact: Fraction) -> set[int]:
    """Bit patterns a float32 result of a value this close to `exact` may
    take: the nearest float32, or both neighbours of a boundary that lies
    within 2^-45 relative of it."""
    eps = Fraction(1, 2 ** 45)
    outs = {rn_f32(exact * (1 - eps)), rn_f32(exact), rn_f32(exact * (1 + eps))}
    return {int(np.float32(v).view(np.uint32)) for v in outs}


def _exact_f64_path(dim, elems, theta):
    mpmath.mp.dps = 45
    n = dim // elems
    out = []
    for i in range(n):
        e = mpmath.mpf(0) if n == 1 else mpmath.mpf(i) / (n - 1)
        out.append(_fraction(mpmath.power(mpmath.mpf(theta), e) * mpmath.pi / 2))
    return out


def _model_f32_path(dim, elems, theta):
    """Allowed bit sets per element of the float32 path, each binary32 step
    modelled exactly."""
    mpmath.mp.dps = 45
    n = dim // elems
    theta32 = Fraction(float(rn_f32(Fraction(theta))))
    pi32 = rn_f32(_fraction(mpmath.pi))
    allowed = []
    for i in range(n):
        lin32 = Fraction(0) if n == 1 else Fraction(float(rn_f32(Fraction(i, n - 1))))
        exact_pow = _fraction(mpmath.power(mpmath.mpf(theta32.numerator) / theta32.denominator,
                                           mpmath.mpf(lin32.numerator) / lin32.denominator))
        sets = set()
        for p_bits in _allowed_f32(exact_pow):
            p = Fraction(float(np.uint32(p_bits).view(np.float32)))
            prod = Fraction(float(rn_f32(p * Fraction(float(pi32)))))
            half = rn_f32(prod / 2)
            sets.add(int(np.float32(half).view(np.uint32)))
        allowed.append(sets)
    return allowed


def _pins(o):
    for dim, elems, theta in CASES:
        got = o.dit_rope_freqs(dim, elems, theta, double_precision=True)
        assert got.dtype == np.float32 and got.shape == (dim // elems,)
        bits = got.view(np.uint32)
        for i, exact in enumerate(_exact_f64_path(dim, elems, theta)):
            assert int(bits[i]) in _allowed_f32(exact), (dim, elems, theta, i)
        got32 = o.dit_rope_freqs(dim, elems, theta, double_precision=False)
        bits32 = got32.view(np.uint32)
        for i, allowed in enumerate(_model_f32_path(dim, elems, theta)):
            assert int(bits32[i]) in allowed, ("f32", dim, elems, theta, i)


def test_dit_freqs_pins():
    _pins(oracle)


@pytest.mark.parametrize("double_precision", [True, False])
def test_dit_freqs_closed_forms(double_precision):
    half_pi = np.float32(np.pi / 2)
    for dim, elems, theta in CASES:
        f = oracle.dit_rope_freqs(dim, elems, theta, double_precision)
        assert f[0] == half_pi
        if f.size > 1:
            assert np.all(np.diff(f) > 0)
            if double_precision:
                assert f[-1] == np.float32(np.float64(theta) * np.pi / 2)
    assert oracle.dit_rope_freqs(5, 6 - 1, 10000.0, double_precision).tolist() == [half_pi]
    assert np.all(oracle.dit_rope_freqs(60, 6, 1.0, double_precision) == half_pi)


def test_dit_freqs_rejects():
    for args in [(5, 6, 1e4), (0, 6, 1e4), (12, 0, 1e4), (12, 6, 0.0), (12, 6, -2.0),
                 (12, 6, float("inf")), (12, 6, float("nan"))]:
        with pytest.raises(ValueError):
            oracle.dit_rope_freqs(*args)


# planted mistakes: each must fail a pin
MUTATIONS = {
    "linspace_end_exclusive": ("lin = np.arange(n, dtype=np.float64) / np.float64(n - 1)",
                               "lin = np.arange(n, dtype=np.float64) / np.float64(n)"),
    "no_halving": ("freqs = pow_indices * np.float64(np.pi) / np.float64(2.0)",
                   "freqs = pow_indices * np.float64(np.pi) / np.float64(1.0)"),
    "pow_operands_swapped": ("pow_indices = np.power(np.float64(theta), lin)",
                             "pow_indices = np.power(lin, np.float64(theta))"),
    "f32_path_pi_in_float64": ("freqs = pow_indices * np.float32(np.pi) / np.float32(2.0)",
                               "freqs = pow_indices * np.float64(np.pi) / np.float32(2.0)"),
    "f32_path_exponent_unrounded": (
        "pow_indices = np.power(np.float64(theta32), lin32.astype(np.float64)).astype(np.float32)",
        "pow_indices = np.power(np.float64(theta32), lin).astype(np.float32)"),
    "inverse_frequencies": ("pow_indices = np.power(np.float64(theta), lin)",
                            "pow_indices = np.power(np.float64(theta), -lin)"),
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


def test_dit_freqs_pins_pass_on_an_unmutated_copy(tmp_path):
    _pins(_copy_of_oracle(tmp_path, "unmutated"))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_dit_freqs_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    mutant = _copy_of_oracle(tmp_path, name, old, new)
    with pytest.raises((AssertionError, ValueError)):
        _pins(mutant)
