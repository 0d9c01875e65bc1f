"""Pins for the NeoX-style RoPE oracle of the Gemma3 text encoder (sglang
PR #24660 review, "关键源码片段", gemma_3.py): rows of a [cos | sin] cache are
gathered by position and cast to the input dtype, then
q * cos + rotate_half(q) * sin is evaluated in that dtype, rotate_half(x) =
(-x2, x1) for the halves of head_dim. Checked against an exact-rational model
of each tensor operation's rounding, a float64 complex brute force, the
cache's high-precision values, the identity at position 0, marker caches and
planted mistakes."""
from __future__ import annotations

import math
import os
import subprocess

import numpy as np
import pytest

import oracle
import synthetic
from tests import exact


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _to16(v: np.ndarray, dtype: str) -> np.ndarray:
    v = np.asarray(v, np.float32)
    return synthetic.f32_to_bf16_bits(v) if dtype == "bf16" else v.astype(np.float16).view(np.uint16)


def _from16(b: np.ndarray, dtype: str) -> np.ndarray:
    b = np.asarray(b, np.uint16)
    if dtype == "bf16":
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return b.view(np.float16).astype(np.float32)


def _model16(x1, x2, c, s, dtype):
    """Exact-rational model: every product and sum of the eager expression
    rounded as PyTorch rounds a 16-bit tensor operation."""
    rn16 = exact.rn_bf16_bits if dtype == "bf16" else exact.rn_f16_bits
    val = (lambda b: float(_from16(np.array([b]), dtype)[0]))
    X1, X2, C, S = (exact.exact(val(v)) for v in (x1, x2, c, s))

    def prod(a, b, neg_zero):
        r = a * b
        f = exact.rn_f32(r, negative_zero=neg_zero)        # exact: 16-bit x 16-bit fits float
        assert exact.exact(f) == r
        return rn16(f)

    def neg(a):
        return -a

    def is_neg(v):
        return math.copysign(1.0, val(v)) < 0

    x1c = prod(X1, C, is_neg(x1) != is_neg(c))
    x2c = prod(X2, C, is_neg(x2) != is_neg(c))
    nx2s = prod(neg(X2), S, (not is_neg(x2)) != is_neg(s))
    x1s = prod(X1, S, is_neg(x1) != is_neg(s))

    def add(a, b):
        fa, fb = val(a), val(b)
        f = exact.add_model(np.float32(fa), np.float32(fb))
        return rn16(f)

    return add(x1c, nx2s), add(x2c, x1s)


def pin_neox_pair_rounding(lib):
    g = _rng(90)
    for dtype in ("bf16", "f16"):
        x = _to16(g.standard_normal(4000) * 3, dtype)
        ang = g.uniform(-50, 50, 2000)
        c = _to16(np.cos(ang), dtype)
        s = _to16(np.sin(ang), dtype)
        for i in range(2000):
            got = oracle.neox_pair16(x[2 * i], x[2 * i + 1], c[i], s[i], dtype, lib)
            want = _model16(int(x[2 * i]), int(x[2 * i + 1]), int(c[i]), int(s[i]), dtype)
            assert got == want, (dtype, i, got, want)


def _neox_bruteforce(x64, positions, head_dim, base):
    tokens, heads, _ = x64.shape
    half = head_dim // 2
    inv = base ** (-(2.0 * np.arange(half)) / head_dim)
    ang = positions.astype(np.float64)[:, None] * inv[None, :]          # [tokens, half]
    z = (x64[..., :half] + 1j * x64[..., half:]) * np.exp(1j * ang)[:, None, :]
    return np.concatenate([z.real, z.imag], axis=-1)


def pin_neox_bruteforce(lib):
    tokens, heads, hd = 9, 3, 16
    g = _rng(91)
    positions = g.integers(0, 60, tokens)
    cache = oracle.neox_cache(60, hd, 10000.0, lib)
    for dtype, tol in (("f32", 2e-6), ("bf16", 2.0 ** -6), ("f16", 2.0 ** -9)):
        xf = (g.standard_normal((tokens, heads, hd))).astype(np.float32)
        x = xf if dtype == "f32" else _to16(xf, dtype).reshape(xf.shape)
        y = oracle.rope_neox(x, tokens, heads, hd, positions, cache, dtype, lib)
        x64 = (x if dtype == "f32" else _from16(x, dtype)).astype(np.float64).reshape(tokens, heads, hd)
        y64 = (y if dtype == "f32" else _from16(y, dtype)).astype(np.float64).reshape(tokens, heads, hd)
        ref = _neox_bruteforce(x64, positions, hd, 10000.0)
        norm = np.sqrt(x64[..., : hd // 2] ** 2 + x64[..., hd // 2:] ** 2)
        err = np.maximum(np.abs(y64 - ref)[..., : hd // 2], np.abs(y64 - ref)[..., hd // 2:])
        assert np.all(err <= tol * norm + 1e-30), (dtype, err.max())


def pin_neox_cache_values(lib):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    cache = oracle.neox_cache(40, 8, 10000.0, lib)
    for p in range(40):
        for j in range(4):
            ang = p * mpmath.power(10000, mpmath.mpf(-2 * j) / 8)
            for got, true in ((cache[p, j], mpmath.cos(ang)), (cache[p, 4 + j], mpmath.sin(ang))):
                t = float(true)
                ulp = float(np.spacing(np.float32(abs(t)))) if t != 0 else 2.0 ** -149
                assert abs(float(got) - t) <= 0.5 * ulp + 1e-12


def pin_neox_position_zero_and_marker(lib):
    tokens, heads, hd = 6, 2, 8
    g = _rng(92)
    x = _to16(g.standard_normal((tokens, heads, hd)) + 0.25, "bf16")
    cache = oracle.neox_cache(5, hd, 10000.0, lib)
    y = oracle.rope_neox(x, tokens, heads, hd, np.zeros(tokens, np.int64), cache, "bf16", lib)
    assert np.array_equal(y, x)
    # identity rows except row 3, column 1, which turns by a quarter: channel 1
    # becomes -x[5], channel 5 becomes x[1], only for tokens at position 3
    marker = np.zeros((5, hd), np.float32)
    marker[:, : hd // 2] = 1.0
    marker[3, 1], marker[3, hd // 2 + 1] = 0.0, 1.0
    positions = np.array([0, 3, 1, 3, 4, 2], np.int64)
    y = oracle.rope_neox(x, tokens, heads, hd, positions, marker, "bf16", lib).reshape(tokens, heads, hd)
    want = x.reshape(tokens, heads, hd).copy()
    for t in (1, 3):
        want[t, :, 1] = x.reshape(tokens, heads, hd)[t, :, 5] ^ 0x8000
        want[t, :, 5] = x.reshape(tokens, heads, hd)[t, :, 1]
    assert np.array_equal(y, want)
    with pytest.raises(ValueError):
        oracle.rope_neox(x, tokens, heads, hd, np.full(tokens, 5, np.int64), cache, "bf16", lib)


PINS = [pin_neox_pair_rounding, pin_neox_bruteforce, pin_neox_cache_values,
        pin_neox_position_zero_and_marker]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_neox_pin(pin, oracle_lib):
    pin(oracle_lib)


MUTATIONS = {
    "pairs_adjacent": ("oracle_neox_pair16(xh[row + j], xh[row + half + j]",
                       "oracle_neox_pair16(xh[row + j], xh[row + (j ^ 1)]"),
    "rotate_sign": ("const float neg_x2 = -fx2;", "const float neg_x2 = fx2;"),
    "cos_not_cast": ("const float fc = from16(c, kind), fs = from16(s, kind);",
                     "const float fc = from16(c, kind) * 1.0001f, fs = from16(s, kind);"),
    "sum_unrounded_products": ("const uint16_t x1c = to16(fx1 * fc, kind);",
                               "const uint16_t x1c = to16(fx1 * fc + 1e-3f * fx1, kind);"),
    "cache_sin_column": ("cache[p * rotary_dim + half + j] = (float)sin(angle);",
                         "cache[p * rotary_dim + half + j] = (float)sin(angle * 1.5);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_neox_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "rope3d_oracle.c")).read()
    assert src.count(old) == 1, name
    c = tmp_path / "o.c"
    c.write_text(src.replace(old, new))
    so = tmp_path / "o.so"
    subprocess.run(["gcc", *oracle.CFLAGS, str(c), "-o", str(so), "-lm"], check=True)
    lib = oracle.load(str(so))
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught {name}"
