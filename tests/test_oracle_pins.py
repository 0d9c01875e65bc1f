"""Pins for the CPU oracle: checks against facts that do not come from the
oracle itself.

What fixes the result (sglang PR #35698 review, "fused LTX-2.5 decoder 3D
RoPE"):
  * "实现拆解" step 2 and "关键源码片段" (rotate_pair): each (even, odd) pair is
    rotated in float32 as even*cos - odd*sin and even*sin + odd*cos, four
    separately rounded products, one rounded subtract and one rounded add,
    then a cast back to the input dtype.
  * "关键源码片段" (the kernel's index decode): tokens are row-major over
    (frame, y, x); T, H, W take consecutive chunks of head_dim; the table row is
    the integer grid coordinate; table column j serves channels (2j, 2j+1).
  * "实现拆解" step 1: tables of shape [length, dim/2] built from
    (length, dim, base); the formula is our reading (standard RoPE,
    base^(-2j/d), evaluated in double, rounded once to float).

Each check is chosen so that a plausible mistake in the oracle fails it; the
last test plants such mistakes in a copy of the oracle and confirms that.
"""
from __future__ import annotations

import math
import os
import platform
import shutil
import struct
import subprocess

import numpy as np
import pytest

import oracle
import synthetic
from tests import exact


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def _bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) if a.dtype == np.float32 else a


def _bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def brute_force_complex(x64: np.ndarray, shape, split, base):
    """Float64 complex reference: each pair (e, o) of chunk X at position p is
    the complex number e + i*o multiplied by exp(i * p * base**(-2j/d_X))."""
    B, T, H, W, heads, hd = shape
    x = x64.reshape(B, T, H, W, heads, hd)
    out = np.empty_like(x)
    grids = np.meshgrid(np.arange(T), np.arange(H), np.arange(W), indexing="ij")
    start = 0
    for axis, d in enumerate(split):
        half = d // 2
        pos = grids[axis].astype(np.float64)                       # [T, H, W]
        inv = base ** (-(2.0 * np.arange(half)) / d)               # [half]
        angle = pos[..., None] * inv                                # [T, H, W, half]
        rot = np.exp(1j * angle)[None, :, :, :, None, :]            # [1,T,H,W,1,half]
        chunk = x[..., start:start + d].reshape(B, T, H, W, heads, half, 2)
        z = (chunk[..., 0] + 1j * chunk[..., 1]) * rot
        out[..., start:start + d:2] = z.real
        out[..., start + 1:start + d:2] = z.imag
        start += d
    return out.reshape(-1)


def pair_norms(x: np.ndarray) -> np.ndarray:
    p = x.reshape(-1, 2).astype(np.float64)
    return np.sqrt(p[:, 0] ** 2 + p[:, 1] ** 2)


def _random_f32(n, seed, scale=1.0):
    return (_rng(seed).standard_normal(n) * scale).astype(np.float32)


# The pins as functions of the loaded library, so the planted-mistake test can
# run them against a mutated copy of the oracle.

def pin_bf16_conversions(lib):
    # widening: bf16 bits are the top half of a binary32
    cases = {
        0x3F80: 1.0, 0xC000: -2.0, 0x0001: math.ldexp(1.0, -133),
        0x7F7F: (2 - 2 ** -7) * 2.0 ** 127, 0x0080: math.ldexp(1.0, -126),
        0x3E80: 0.25, 0x8000: -0.0,
    }
    for bits, val in cases.items():
        got = oracle.bf16_to_f32(bits, lib)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(bits)
    assert math.isinf(oracle.bf16_to_f32(0x7F80, lib))
    # narrowing: nearest, ties to even, against the exact-rational model
    specials = [1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -(1 + 3 * 2 ** -8),
                2.0 ** -134, 3 * 2.0 ** -134, 2.0 ** -149, float(np.finfo(np.float32).max),
                (2 - 2 ** -8) * 2.0 ** 127, 0.0, -0.0, 1.0, 65504.0, 3.1415926]
    vals = [np.float32(v) for v in specials]
    g = _rng(1)
    vals += list(exact.bits_f32(int(b)) for b in g.integers(0, 0x7F800000, 4000))
    vals += list(-np.float32(v) for v in _random_f32(1000, 2))
    for v in vals:
        v = np.float32(v)
        assert oracle.f32_to_bf16(v, lib) == exact.rn_bf16_bits(v), repr(v)
    assert oracle.f32_to_bf16(np.float32(np.inf), lib) == 0x7F80
    assert oracle.f32_to_bf16(np.float32(-np.inf), lib) == 0xFF80
    nan = oracle.f32_to_bf16(np.float32(np.nan), lib)
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x7F) != 0


def pin_f16_conversions(lib):
    # widening: every finite bit pattern against its exact value
    for bits in range(1 << 16):
        if (bits & 0x7C00) == 0x7C00 and (bits & 0x3FF):
            assert math.isnan(oracle.f16_to_f32(bits, lib))
            continue
        got = oracle.f16_to_f32(bits, lib)
        want = exact.f16_value(bits)
        assert got == float(want), hex(bits)
        assert math.copysign(1, got) == (-1 if bits & 0x8000 else 1), hex(bits)
    # narrowing: nearest binary16, ties to even, against the exact-rational model
    specials = [1.0, 65504.0, 65519.99, 65520.0, 70000.0, 2.0 ** -24, 2.0 ** -25,
                3 * 2.0 ** -25, 2.0 ** -25 * 1.0000001, 5 * 2.0 ** -26, 2.0 ** -14,
                2.0 ** -14 - 2.0 ** -25, 1 + 2 ** -11, 1 + 3 * 2 ** -11, 0.0, -0.0, 1e-30,
                -1e-8, 3.1415926, 2049.0, 2051.0, float(np.finfo(np.float32).max)]
    vals = [np.float32(v) for v in specials]
    g = _rng(5)
    vals += list(exact.bits_f32(int(b)) for b in g.integers(0x30000000, 0x48000000, 6000))
    vals += list(np.float32(v) for v in _random_f32(2000, 6, 100.0))
    for v in vals:
        v = np.float32(v)
        assert oracle.f32_to_f16(v, lib) == exact.rn_f16_bits(v), repr(v)
    assert oracle.f32_to_f16(np.float32(np.inf), lib) == 0x7C00
    nan = oracle.f32_to_f16(np.float32(np.nan), lib)
    assert (nan & 0x7C00) == 0x7C00 and (nan & 0x3FF) != 0


def pin_f16_bruteforce(lib):
    shape, split = (2, 3, 5, 7, 3, 18), (4, 6, 8)
    tabs = oracle.tables(3, 5, 7, split, 10000.0, lib)
    x = _random_f32(int(np.prod(shape)), 18, 1.0).astype(np.float16)
    y = oracle.rope3d(x.view(np.uint16), shape, split, tabs, lib, f16=True).view(np.float16)
    ref = brute_force_complex(x.astype(np.float64), shape, split, 10000.0)
    err = np.abs(y.astype(np.float64) - ref).reshape(-1, 2).max(axis=1)
    assert np.all(err <= (2.0 ** -11 + 2e-6) * pair_norms(x.astype(np.float32)) + 2.0 ** -25), err.max()


def pin_rotate_pair_rounding(lib):
    # A product that rounds away only without fusion: e*c = 1 - 2**-46 rounds
    # to 1, so y0 = 1 - 1 = 0 exactly; a fused multiply-subtract gives -2**-46.
    e, o, c, s = np.float32(1 + 2 ** -23), np.float32(1), np.float32(1 - 2 ** -23), np.float32(1)
    y0, y1 = oracle.rotate_pair(e, o, c, s, lib)
    assert exact.f32_bits(y0) == 0 and y1 == np.float32(2.0)
    # random pairs and table values against the exact-rational model, bitwise
    g = _rng(3)
    ang = g.uniform(-100, 100, 3000)
    quads = np.stack([
        _random_f32(3000, 4, 3.0), _random_f32(3000, 5, 3.0),
        np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)], axis=1)
    # add tiny operands so that subnormal products occur
    quads[:200, 0] *= np.float32(2.0 ** -120)
    quads[200:400, 1] *= np.float32(2.0 ** -125)
    for e, o, c, s in quads:
        y0, y1 = oracle.rotate_pair(e, o, c, s, lib)
        m0, m1 = exact.rotate_pair_model(e, o, c, s)
        assert exact.f32_bits(y0) == exact.f32_bits(m0), (e, o, c, s)
        assert exact.f32_bits(y1) == exact.f32_bits(m1), (e, o, c, s)


def pin_tables_high_precision(lib):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    for length, dim, base in [(24, 32, 10000.0), (96, 48, 10000.0), (5, 6, 500.0), (3, 2, 10000.0)]:
        c, s = oracle.axis_table(length, dim, base, lib)
        assert c.shape == (length, dim // 2)
        for pos in range(length):
            for j in range(dim // 2):
                ang = pos * mpmath.power(base, mpmath.mpf(-2 * j) / dim)
                for got, true in ((c[pos, j], mpmath.cos(ang)), (s[pos, j], mpmath.sin(ang))):
                    t = float(true)
                    ulp = float(np.spacing(np.float32(abs(t)))) if t != 0 else 2.0 ** -149
                    assert abs(float(got) - float(true)) <= 0.5 * ulp + 1e-12, (length, dim, pos, j)
        # position 0 is exactly the identity rotation; column 0 has frequency 1
        assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)
        assert c[min(1, length - 1), 0] == np.float32(math.cos(min(1, length - 1)))


def pin_complex_bruteforce(lib):
    for shape, split in [((1, 2, 4, 4, 2, 48), (16, 16, 16)), ((2, 3, 5, 7, 3, 18), (4, 6, 8))]:
        tabs = oracle.tables(*shape[1:4], split, 10000.0, lib)
        n = int(np.prod(shape))
        # float32 inputs: within 2e-6 of the pair's norm
        x = _random_f32(n, 10, 1.0)
        y = oracle.rope3d(x, shape, split, tabs, lib)
        ref = brute_force_complex(x.astype(np.float64), shape, split, 10000.0)
        err = np.abs(y.astype(np.float64) - ref).reshape(-1, 2).max(axis=1)
        assert np.all(err <= 2e-6 * pair_norms(x)), err.max()
        # bf16 inputs: the same plus the final bf16 rounding (half an ulp of 2**-7)
        xb = synthetic.f32_to_bf16_bits(_random_f32(n, 11, 1.0))
        yb = oracle.rope3d(xb, shape, split, tabs, lib)
        refb = brute_force_complex(_bf16_bits_to_f32(xb).astype(np.float64), shape, split, 10000.0)
        errb = np.abs(_bf16_bits_to_f32(yb).astype(np.float64) - refb).reshape(-1, 2).max(axis=1)
        assert np.all(errb <= (2.0 ** -8 + 2e-6) * pair_norms(_bf16_bits_to_f32(xb))), errb.max()


def pin_position_zero_identity(lib):
    # a 1x1x1 grid puts every token at position 0 on every axis: out == in
    shape, split = (3, 1, 1, 1, 4, 40), (8, 16, 16)
    tabs = oracle.tables(1, 1, 1, split, 10000.0, lib)
    x = _random_f32(int(np.prod(shape)), 12)
    assert np.array_equal(_bits(oracle.rope3d(x, shape, split, tabs, lib)), _bits(x))
    xb = synthetic.f32_to_bf16_bits(x)
    assert np.array_equal(oracle.rope3d(xb, shape, split, tabs, lib), xb)
    # on a real grid, the T chunk of every frame-0 token is unchanged, and the
    # whole head of token (0, 0, 0) is unchanged
    shape, split = (2, 3, 4, 5, 2, 24), (8, 8, 8)
    tabs = oracle.tables(3, 4, 5, split, 10000.0, lib)
    x = _random_f32(int(np.prod(shape)), 13)
    y = oracle.rope3d(x, shape, split, tabs, lib).reshape(shape)
    x6 = x.reshape(shape)
    assert np.array_equal(_bits(y[:, 0, :, :, :, :8]), _bits(x6[:, 0, :, :, :, :8]))
    assert np.array_equal(_bits(y[:, :, 0, :, :, 8:16]), _bits(x6[:, :, 0, :, :, 8:16]))
    assert np.array_equal(_bits(y[:, :, :, 0, :, 16:]), _bits(x6[:, :, :, 0, :, 16:]))
    assert np.array_equal(_bits(y[:, 0, 0, 0]), _bits(x6[:, 0, 0, 0]))


def pin_norm_preserved(lib):
    shape, split = (1, 4, 16, 16, 4, 64), (16, 24, 24)
    tabs = oracle.tables(4, 16, 16, split, 10000.0, lib)
    x = _random_f32(int(np.prod(shape)), 14, 2.0)
    y = oracle.rope3d(x, shape, split, tabs, lib)
    n0, n1 = pair_norms(x), pair_norms(y)
    assert np.all(np.abs(n1 - n0) <= 1e-6 * n0)


def pin_rotate_back(lib):
    shape, split = (1, 3, 5, 7, 3, 18), (4, 6, 8)
    tabs = oracle.tables(3, 5, 7, split, 10000.0, lib)
    inverse = tuple((c, -s) for c, s in tabs)
    x = _random_f32(int(np.prod(shape)), 15)
    back = oracle.rope3d(oracle.rope3d(x, shape, split, tabs, lib), shape, split, inverse, lib)
    err = np.abs(back.astype(np.float64) - x).reshape(-1, 2).max(axis=1)
    assert np.all(err <= 1e-6 * pair_norms(x))


def pin_marker_tables(lib):
    """Tables that are the identity except one (row, column) of one axis,
    where they rotate by a quarter turn (cos 0, sin 1), so the pair becomes
    (-odd, even) exactly. Only the channels of that axis's chunk, column and
    grid row may change: this pins the axis order, the chunk offsets, the
    interleaving of pairs and the token decode exactly."""
    shape, split = (2, 3, 4, 5, 2, 24), (6, 8, 10)
    B, T, H, W, heads, hd = shape
    x = synthetic.f32_to_bf16_bits(_random_f32(int(np.prod(shape)), 16))
    xf = _bf16_bits_to_f32(x).reshape(shape)
    lengths = (T, H, W)
    for axis in range(3):
        for row in range(lengths[axis]):
            col = (row + axis) % (split[axis] // 2)
            tabs = []
            for a in range(3):
                c = np.ones((lengths[a], split[a] // 2), np.float32)
                s = np.zeros_like(c)
                if a == axis:
                    c[row, col], s[row, col] = 0.0, 1.0
                tabs.append((c, s))
            y = _bf16_bits_to_f32(oracle.rope3d(x, shape, split, tabs, lib)).reshape(shape)
            expect = xf.copy()
            ch = sum(split[:axis]) + 2 * col
            sl = [slice(None)] * 6
            sl[1 + axis] = row
            sl5e = tuple(sl[:5] + [ch])
            sl5o = tuple(sl[:5] + [ch + 1])
            expect[sl5e] = -xf[sl5o]
            expect[sl5o] = xf[sl5e]
            assert np.array_equal(y.view(np.uint32), expect.view(np.uint32)), (axis, row)


def pin_sampled_matches_full(lib):
    shape, split = (2, 3, 5, 7, 3, 18), (4, 6, 8)
    tabs = oracle.tables(3, 5, 7, split, 10000.0, lib)
    for dt in ("bf16", "f32"):
        x = synthetic.normal(int(np.prod(shape)), 1.0, 17, 0, dt)
        y = oracle.rope3d(x, shape, split, tabs, lib)
        idx = synthetic.sample_indices(x.size, 500, 3, shape[-1])
        assert np.array_equal(_bits(oracle.rope3d_at(x, idx, shape, split, tabs, lib)), _bits(y[idx]))


PINS = [
    pin_bf16_conversions, pin_f16_conversions, pin_f16_bruteforce,
    pin_rotate_pair_rounding, pin_tables_high_precision,
    pin_complex_bruteforce, pin_position_zero_identity, pin_norm_preserved,
    pin_rotate_back, pin_marker_tables, pin_sampled_matches_full,
]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_oracle_rejects_bad_shapes(oracle_lib):
    tabs = oracle.tables(2, 2, 2, (2, 2, 2), 10000.0, oracle_lib)
    x = np.zeros(2 * 2 * 2 * 6, np.uint16)
    for shape, split in [((1, 2, 2, 2, 1, 6), (2, 2, 3)), ((1, 2, 2, 2, 1, 6), (2, 2, 4)),
                         ((1, 2, 2, 2, 1, 6), (0, 2, 4))]:
        with pytest.raises(ValueError):
            oracle.rope3d(x, shape, split, tabs, oracle_lib)
    with pytest.raises(ValueError):
        oracle.axis_table(4, 3, 10000.0, oracle_lib)


# ---------------------------------------------------------------------------
# planted mistakes: each mutation of the oracle source must fail some pin
# ---------------------------------------------------------------------------

MUTATIONS = {
    "y0_sign": ("float y0 = even_cos - odd_sin;", "float y0 = even_cos + odd_sin;"),
    "y1_sign": ("float y1 = even_sin + odd_cos;", "float y1 = even_sin - odd_cos;"),
    "cos_sin_swapped": ("float even_cos = even * c;", "float even_cos = even * s;"),
    "axis_positions": ("const int64_t pos[3] = {t, h, w};", "const int64_t pos[3] = {h, t, w};"),
    "pair_stride": ("const int64_t ch = chunk_start + 2 * j;",
                    "const int64_t ch = chunk_start + j;"),
    "table_exponent": ("double exponent = -(2.0 * (double)j) / (double)dim;",
                       "double exponent = -(1.0 * (double)j) / (double)dim;"),
    "table_row": ("const float *crow = cos_tab[axis] + pos[axis] * half;",
                  "const float *crow = cos_tab[axis] + pos[axis] * half + (pos[axis] > 0);"),
    "bf16_truncate": ("uint32_t rounded = bits + 0x7fffu + kept_lsb;",
                      "uint32_t rounded = bits;"),
    "bf16_ties_away": ("uint32_t rounded = bits + 0x7fffu + kept_lsb;",
                       "uint32_t rounded = bits + 0x8000u;"),
    "sample_decode": ("const int64_t w = token % W;", "const int64_t w = token % H;"),
    "f16_ties_away": ("if (rest > 0x1000u || (rest == 0x1000u && (h & 1u)))",
                      "if (rest >= 0x1000u)"),
    "f16_subnormal_shift": ("const int shift = -e - 1;", "const int shift = -e;"),
    "f16_overflow_edge": ("if (mag >= 0x477ff000u)", "if (mag >= 0x477fe000u)"),
    "f16_widen_bias": ("(int)exponent - 25", "(int)exponent - 24"),
}


def _build_mutant(tmp_path, name, old, new, extra=()):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "rope3d_oracle.c")).read()
    assert src.count(old) >= 1, name
    mutated = src.replace(old, new)
    d = tmp_path / name
    d.mkdir()
    c = d / "rope3d_oracle.c"
    c.write_text(mutated)
    so = d / "lib.so"
    subprocess.run(["gcc", *oracle.CFLAGS, *extra, str(c), "-o", str(so), "-lm"], check=True)
    return oracle.load(str(so))


def _caught(lib) -> list[str]:
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    return failed


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    assert _caught(lib), f"no pin caught mutation {name}"


@pytest.mark.skipif(platform.machine() not in ("x86_64", "aarch64"), reason="needs an FMA target")
def test_planted_fma_contraction_is_caught(tmp_path):
    """The same source compiled with contraction into fused multiply-add must
    fail the exact-rounding pin."""
    extra = ["-ffp-contract=fast", "-mfma"] if platform.machine() == "x86_64" else ["-ffp-contract=fast"]
    lib = _build_mutant(tmp_path, "fma", "float y0", "float y0", extra=extra)
    with pytest.raises(AssertionError):
        pin_rotate_pair_rounding(lib)


def test_tables_match_the_committed_digest():
    """The oracle's tables (from the host C library's pow, cos and sin) equal
    the digest tests/golden/make_golden.py wrote; it was checked on both
    x86-64 and aarch64 hosts."""
    from tests.golden import make_golden

    want = open(os.path.join(os.path.dirname(__file__), "golden", "oracle_tables_sha256.txt")).read().strip()
    assert make_golden.tables_digest() == want
