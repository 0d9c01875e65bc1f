"""CPU oracle for the paired 3D RoPE of the LTX-2.5 diffusion decoder.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference leg of ``bench.py`` import this package. The product
library (``rope_rope3d_apply_gb300``) never imports it and shares no code with
it; the two meet only through the seeded inputs of the ``synthetic`` package.

The arithmetic lives in ``rope3d_oracle.c`` (plain C, built with
``-ffp-contract=off``); this module compiles it with gcc and wraps it with
ctypes over numpy arrays. What each function follows is cited in the C file:
sglang PR #35698 review ("fused LTX-2.5 decoder 3D RoPE"), sections
"实现拆解" (steps 1 and 2) and "关键源码片段" (the rotate_pair arithmetic, the
kernel's index decode and the wrapper's preflight).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, exact-rational rounding, a float64 complex brute force,
high-precision table values, invariants and planted-mistake checks).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rope3d_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "librope3d_oracle.so")

# Flags: no contraction into fused multiply-add, no fast-math, IEEE defaults.
CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(out_path: str = _LIB_PATH, extra_flags: list[str] | None = None) -> str:
    """Compile the oracle with gcc; returns the path of the shared library."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, *(extra_flags or []), _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def _declare(lib):
    i64, f32p = ctypes.c_int64, ctypes.c_void_p
    vp = ctypes.c_void_p
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_f16.restype = ctypes.c_uint16
    lib.oracle_axis_table.argtypes = [i64, i64, ctypes.c_double, f32p, f32p]
    lib.oracle_axis_table.restype = ctypes.c_int
    lib.oracle_rotate_pair_f32.argtypes = [ctypes.c_float] * 4 + [vp, vp]
    lib.oracle_rotate_pair_f32.restype = None
    full = [vp, vp] + [i64] * 6 + [vp] + [vp] * 6
    lib.oracle_rope3d_bf16.argtypes = full
    lib.oracle_rope3d_bf16.restype = ctypes.c_int
    lib.oracle_rope3d_f32.argtypes = full
    lib.oracle_rope3d_f32.restype = ctypes.c_int
    lib.oracle_rope3d_f16.argtypes = full
    lib.oracle_rope3d_f16.restype = ctypes.c_int
    at = [vp, vp, i64, vp] + [i64] * 6 + [vp] + [vp] * 6
    lib.oracle_rope3d_bf16_at.argtypes = at
    lib.oracle_rope3d_bf16_at.restype = ctypes.c_int
    lib.oracle_rope3d_f32_at.argtypes = at
    lib.oracle_rope3d_f32_at.restype = ctypes.c_int
    lib.oracle_neox_cache.argtypes = [i64, i64, ctypes.c_double, vp]
    lib.oracle_neox_cache.restype = ctypes.c_int
    lib.oracle_neox_pair16.argtypes = [ctypes.c_uint16] * 4 + [ctypes.c_int, vp, vp]
    lib.oracle_neox_pair16.restype = None
    lib.oracle_neox_pair_f32.argtypes = [ctypes.c_float] * 4 + [vp, vp]
    lib.oracle_neox_pair_f32.restype = None
    lib.oracle_rope_neox.argtypes = [vp, vp, i64, i64, i64, vp, vp, i64, ctypes.c_int]
    lib.oracle_rope_neox.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library. ``path`` loads a
    separately built copy, e.g. one compiled with a planted mistake."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH) or (
                os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
            ):
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _split_arr(split) -> np.ndarray:
    s = np.asarray(split, dtype=np.int32)
    if s.shape != (3,):
        raise ValueError("split must have three entries (d_T, d_H, d_W)")
    return np.ascontiguousarray(s)


# ---------------------------------------------------------------------------
# scalar conversions
# ---------------------------------------------------------------------------

def bf16_to_f32(bits: int, lib=None) -> float:
    return (lib or load()).oracle_bf16_to_f32(int(bits))


def f32_to_bf16(value: float, lib=None) -> int:
    return int((lib or load()).oracle_f32_to_bf16(float(np.float32(value))))


def f16_to_f32(bits: int, lib=None) -> float:
    return (lib or load()).oracle_f16_to_f32(int(bits))


def f32_to_f16(value: float, lib=None) -> int:
    return int((lib or load()).oracle_f32_to_f16(float(np.float32(value))))


def rotate_pair(even: float, odd: float, c: float, s: float, lib=None):
    """One pair in the eager order; returns float32 (y_even, y_odd)."""
    y = np.zeros(2, dtype=np.float32)
    (lib or load()).oracle_rotate_pair_f32(
        float(np.float32(even)), float(np.float32(odd)),
        float(np.float32(c)), float(np.float32(s)),
        _ptr(y), _ptr(y) + 4)
    return y[0], y[1]


# ---------------------------------------------------------------------------
# tables
# ---------------------------------------------------------------------------

def axis_table(length: int, dim: int, base: float = 10000.0, lib=None):
    """(cos, sin) float32 arrays of shape [length, dim // 2]."""
    c = np.empty((length, dim // 2), dtype=np.float32)
    s = np.empty((length, dim // 2), dtype=np.float32)
    rc = (lib or load()).oracle_axis_table(length, dim, float(base), _ptr(c), _ptr(s))
    if rc != 0:
        raise ValueError(f"oracle_axis_table rejected length={length} dim={dim} base={base}")
    return c, s


def tables(T: int, H: int, W: int, split, base: float = 10000.0, lib=None):
    """((cos_t, sin_t), (cos_h, sin_h), (cos_w, sin_w))."""
    return tuple(axis_table(n, d, base, lib) for n, d in zip((T, H, W), split))


def _table_args(tabs):
    flat = []
    for c, s in tabs:
        flat += [np.ascontiguousarray(c, dtype=np.float32),
                 np.ascontiguousarray(s, dtype=np.float32)]
    return flat


# ---------------------------------------------------------------------------
# the rotation
# ---------------------------------------------------------------------------

def rope3d(x: np.ndarray, shape, split, tabs, lib=None, f16: bool = False) -> np.ndarray:
    """Full oracle pass.

    x: uint16 (bf16 bit patterns, or binary16 bit patterns with f16=True) or
    float32 array with B*T*H*W*heads*head_dim elements in
    [B, T, H, W, heads, head_dim] order. shape = (B, T, H, W, heads,
    head_dim). Returns an array of the same dtype and shape as x.
    """
    lib = lib or load()
    B, T, H, W, heads, head_dim = (int(v) for v in shape)
    x = np.ascontiguousarray(x)
    if x.size != B * T * H * W * heads * head_dim:
        raise ValueError("x does not match shape")
    y = np.empty_like(x)
    sp = _split_arr(split)
    tb = _table_args(tabs)
    if x.dtype == np.uint16:
        fn = lib.oracle_rope3d_f16 if f16 else lib.oracle_rope3d_bf16
    elif x.dtype == np.float32:
        fn = lib.oracle_rope3d_f32
    else:
        raise TypeError("x must be uint16 (bf16 / f16 bits) or float32")
    rc = fn(_ptr(x), _ptr(y), B, T, H, W, heads, head_dim, _ptr(sp), *[_ptr(t) for t in tb])
    if rc != 0:
        raise ValueError(f"oracle rejected shape={shape} split={tuple(split)}")
    return y


def rope3d_at(x: np.ndarray, indices: np.ndarray, shape, split, tabs, lib=None) -> np.ndarray:
    """Output elements at the given flat indices, computed one at a time."""
    lib = lib or load()
    B, T, H, W, heads, head_dim = (int(v) for v in shape)
    x = np.ascontiguousarray(x).reshape(-1)
    idx = np.ascontiguousarray(indices, dtype=np.int64)
    out = np.empty(idx.size, dtype=x.dtype)
    sp = _split_arr(split)
    tb = _table_args(tabs)
    if x.dtype == np.uint16:
        fn = lib.oracle_rope3d_bf16_at
    elif x.dtype == np.float32:
        fn = lib.oracle_rope3d_f32_at
    else:
        raise TypeError("x must be uint16 (bf16 bits) or float32")
    rc = fn(_ptr(x), _ptr(idx), idx.size, _ptr(out), B, T, H, W, heads, head_dim,
            _ptr(sp), *[_ptr(t) for t in tb])
    if rc != 0:
        raise ValueError("oracle rejected the sample request")
    return out


# ---------------------------------------------------------------------------
# patchify / unpatchify (sglang PR #34471 review, "关键源码片段", _patchify in
# ltx_2_5_diffusion_decoder.py): space-to-depth over H and W,
# (B, C, F, H, W) -> (B, C*p*p, F, H/p, W/p), channels packed in the order
# (channel, width offset, height offset). Written out as the page's three
# steps: split H and W into (blocks, offset), move the offsets next to the
# channel in the order (width offset, height offset), merge. Exact (a
# permutation), so numpy reshape/transpose is the whole definition.
# _unpatchify is named on the page without code; our reading is the exact
# inverse of _patchify.
# ---------------------------------------------------------------------------

def patchify(x: np.ndarray, p: int) -> np.ndarray:
    B, C, F, H, W = x.shape
    if H % p or W % p:
        raise ValueError("H and W must be multiples of the patch size")
    t = x.reshape(B, C, F, H // p, p, W // p, p)            # (b, c, f, i, ph, j, pw)
    t = t.transpose(0, 1, 6, 4, 2, 3, 5)                    # (b, c, pw, ph, f, i, j)
    return np.ascontiguousarray(t).reshape(B, C * p * p, F, H // p, W // p)


def unpatchify(y: np.ndarray, p: int) -> np.ndarray:
    B, Cpp, F, Hp, Wp = y.shape
    if Cpp % (p * p):
        raise ValueError("channels must be a multiple of p*p")
    C = Cpp // (p * p)
    t = y.reshape(B, C, p, p, F, Hp, Wp)                    # (b, c, pw, ph, f, i, j)
    t = t.transpose(0, 1, 4, 5, 3, 6, 2)                    # (b, c, f, i, ph, j, pw)
    return np.ascontiguousarray(t).reshape(B, C, F, Hp * p, Wp * p)


# ---------------------------------------------------------------------------
# NeoX-style RoPE of the Gemma3 text encoder (sglang PR #24660 review,
# "关键源码片段", gemma_3.py): see rope3d_oracle.c.
# ---------------------------------------------------------------------------

KIND = {"bf16": 0, "f32": 1, "f16": 2}


def neox_cache(max_position: int, rotary_dim: int, base: float = 10000.0, lib=None) -> np.ndarray:
    """[max_position, rotary_dim] float32 rows [cos | sin]."""
    c = np.empty((max_position, rotary_dim), np.float32)
    if (lib or load()).oracle_neox_cache(max_position, rotary_dim, float(base), _ptr(c)) != 0:
        raise ValueError("bad cache arguments")
    return c


def neox_pair16(x1: int, x2: int, c: int, s: int, dtype: str = "bf16", lib=None):
    y = np.zeros(2, np.uint16)
    (lib or load()).oracle_neox_pair16(int(x1), int(x2), int(c), int(s), KIND[dtype],
                                       _ptr(y), _ptr(y) + 2)
    return int(y[0]), int(y[1])


def rope_neox(x: np.ndarray, tokens: int, heads: int, head_dim: int, positions: np.ndarray,
              cache: np.ndarray, dtype: str, lib=None) -> np.ndarray:
    """x: [tokens, heads, head_dim] (uint16 bits for bf16/f16, float32 for f32)."""
    x = np.ascontiguousarray(x)
    y = np.empty_like(x)
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    cache = np.ascontiguousarray(cache, dtype=np.float32)
    rc = (lib or load()).oracle_rope_neox(_ptr(x), _ptr(y), tokens, heads, head_dim, _ptr(pos),
                                          _ptr(cache), cache.shape[0], KIND[dtype])
    if rc != 0:
        raise ValueError("oracle_rope_neox rejected its arguments")
    return y


# ---------------------------------------------------------------------------
# 3D neighbourhood attention with the decoder's RoPE on Q and K (sglang
# PR #34471 review, "关键源码片段": the decoder attends with NATTEN's na3d; the
# PR #35698 review, "功能与动机": 3D RoPE precedes each of its attention
# blocks). Neighbourhood attention as published (Hassani et al.,
# "Neighborhood Attention Transformer", CVPR 2023): a query attends to the
# k_t x k_h x k_w grid window centred on it, shifted to stay inside the grid
# at the borders (window start min(max(i - k//2, 0), L - k) per axis).
# Scores q.k / sqrt(head_dim), softmax over the window, weights times V.
# Evaluated in float64 on the bf16 inputs (after the exact RoPE of rope3d).
# ---------------------------------------------------------------------------

def na_window_starts(length: int, k: int) -> np.ndarray:
    i = np.arange(length)
    return np.minimum(np.maximum(i - k // 2, 0), length - k)


def na3d(q: np.ndarray, k: np.ndarray, v: np.ndarray, shape, kernel) -> np.ndarray:
    """q, k, v: float64 [B, T, H, W, heads, d]; kernel (kt, kh, kw) odd and no
    larger than the grid. Returns float64 [B, T, H, W, heads, d]."""
    B, T, H, W, heads, d = shape
    kt, kh, kw = kernel
    if min(kt, kh, kw) < 1 or kt > T or kh > H or kw > W or not (kt % 2 and kh % 2 and kw % 2):
        raise ValueError("kernel sizes must be odd and fit the grid")
    q = q.reshape(shape)
    k = k.reshape(shape)
    v = v.reshape(shape)
    st, sh, sw = na_window_starts(T, kt), na_window_starts(H, kh), na_window_starts(W, kw)
    # key coordinates of every (query, window slot): [T, H, W, kt*kh*kw] each
    dt, dh, dw = np.meshgrid(np.arange(kt), np.arange(kh), np.arange(kw), indexing="ij")
    kt_idx = st[:, None, None, None] + dt.reshape(1, 1, 1, -1)
    kh_idx = sh[None, :, None, None] + dh.reshape(1, 1, 1, -1)
    kw_idx = sw[None, None, :, None] + dw.reshape(1, 1, 1, -1)
    kt_idx, kh_idx, kw_idx = np.broadcast_arrays(kt_idx, kh_idx, kw_idx)
    out = np.empty(shape, np.float64)
    scale = 1.0 / np.sqrt(d)
    for b in range(B):
        kk = k[b][kt_idx, kh_idx, kw_idx]          # [T, H, W, n, heads, d]
        vv = v[b][kt_idx, kh_idx, kw_idx]
        s = np.einsum("thwed,thwned->thwen", q[b], kk) * scale   # [T, H, W, heads, n]
        s = s - s.max(axis=-1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=-1, keepdims=True)
        out[b] = np.einsum("thwen,thwned->thwed", p, vv)
    return out


def rope_na3d(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, shape, split, tabs,
              kernel, rope: bool = True, lib=None) -> np.ndarray:
    """bf16 inputs (uint16 bits): RoPE on Q and K exactly as rope3d (bf16
    outputs), then na3d in float64. Returns float64."""
    if rope:
        q_bits = rope3d(q_bits, shape, split, tabs, lib)
        k_bits = rope3d(k_bits, shape, split, tabs, lib)
    to64 = lambda b: (np.ascontiguousarray(b).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)  # noqa: E731
    return na3d(to64(q_bits), to64(k_bits), to64(v_bits), shape, kernel)


def rope_na3d_at(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, shape, split, tabs,
                 kernel, queries, rope: bool = True, lib=None):
    """rope_na3d for single queries, one at a time: queries is a list of
    (b, t, h, w, head). Each query vector and each key of its window is rotated
    element by element (rope3d_at), then the window's softmax attention is
    taken in float64. Returns (out, absv), each [len(queries), head_dim]:
    the attention output and the same weights applied to |v|."""
    B, T, H, W, heads, d = (int(x) for x in shape)
    kt, kh, kw = kernel
    st, sh, sw = na_window_starts(T, kt), na_window_starts(H, kh), na_window_starts(W, kw)
    q_flat = np.ascontiguousarray(q_bits).reshape(-1)
    k_flat = np.ascontiguousarray(k_bits).reshape(-1)
    v_flat = np.ascontiguousarray(v_bits).reshape(-1)
    to64 = lambda b: (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)  # noqa: E731
    chan = np.arange(d, dtype=np.int64)

    def row(b, t, h, w, e):   # flat index of channel 0 of (b, t, h, w, head e)
        return ((((b * T + t) * H + h) * W + w) * heads + e) * d

    out = np.empty((len(queries), d))
    absv = np.empty((len(queries), d))
    for n, (b, t, h, w, e) in enumerate(queries):
        qi = row(b, t, h, w, e) + chan
        qv = rope3d_at(q_flat, qi, shape, split, tabs, lib) if rope else q_flat[qi]
        keys = [row(b, tt, hh, ww, e) for tt in range(st[t], st[t] + kt)
                for hh in range(sh[h], sh[h] + kh) for ww in range(sw[w], sw[w] + kw)]
        ki = (np.array(keys, dtype=np.int64)[:, None] + chan[None, :]).reshape(-1)
        kv = rope3d_at(k_flat, ki, shape, split, tabs, lib) if rope else k_flat[ki]
        vv = to64(v_flat[ki]).reshape(len(keys), d)
        s = to64(kv).reshape(len(keys), d) @ to64(qv) / np.sqrt(d)
        p = np.exp(s - s.max())
        p /= p.sum()
        out[n] = p @ vv
        absv[n] = p @ np.abs(vv)
    return out, absv


# ---------------------------------------------------------------------------
# The LTX DiT's RoPE frequency vector (sglang PR #24660 review, "关键源码片段",
# ltx_2.py, the frequency generation that replaced _ltx2_rope_freq_grid_np):
# n = dim // num_rope_elems evenly spaced exponents from 0 to 1, theta raised
# to each, times pi, halved, the result cast to float32. Every step runs in
# the page's freqs_dtype: float64 when double_precision is set, else float32.
# The page then combines the vector with the positions grid and elides how;
# that part is not defined here.
#
# Readings (the page fixes the precision of each step, not the rounding of
# the framework routines it calls):
# - linspace value i is the nearest value of the precision to i / (n - 1)
#   (n = 1 gives the start, 0);
# - pow is correctly rounded in the precision (float32: the float64 power,
#   then one rounding to float32);
# - pi is the nearest value of the precision to pi, the product is rounded
#   once, and the halving is exact.
# ---------------------------------------------------------------------------

def dit_rope_freqs(dim: int, num_rope_elems: int, theta: float = 10000.0,
                   double_precision: bool = True) -> np.ndarray:
    """float32 [dim // num_rope_elems] frequencies, in the page's order of
    steps: linspace, pow, times pi, divided by 2, cast."""
    if dim <= 0 or num_rope_elems <= 0 or dim // num_rope_elems == 0:
        raise ValueError("dim // num_rope_elems must be at least 1")
    if not (np.isfinite(theta) and theta > 0):
        raise ValueError("theta must be finite and > 0")
    n = dim // num_rope_elems
    # step 1: linspace(0, 1, n) in freqs_dtype
    if n == 1:
        lin = np.zeros(1, np.float64)
    else:
        lin = np.arange(n, dtype=np.float64) / np.float64(n - 1)
    if double_precision:
        # steps 2-4 in float64
        pow_indices = np.power(np.float64(theta), lin)
        freqs = pow_indices * np.float64(np.pi) / np.float64(2.0)
    else:
        # steps 2-4 in float32
        lin32 = lin.astype(np.float32)
        theta32 = np.float32(theta)
        pow_indices = np.power(np.float64(theta32), lin32.astype(np.float64)).astype(np.float32)
        freqs = pow_indices * np.float32(np.pi) / np.float32(2.0)
    # step 5: cast to float32
    return freqs.astype(np.float32)
