"""Python binding of the fused paired 3D RoPE library (``include/rope3d.h``).

Argument marshalling only: every step of the rotation runs in the CUDA
kernels of ``_build/librope3d.so``; this module turns tensors into pointers,
sizes and a stream and turns status codes into exceptions. PyTorch is used for
nothing but device memory and streams. When the library has not been built,
loading raises: there is no other code path.

The operation (sglang PR #35698 review, "fused LTX-2.5 decoder 3D RoPE",
sections "实现拆解" and "关键源码片段"): Q and K of shape
[B, T*H*W, heads, head_dim] are rotated pair by pair, T, H and W each using
their own chunk of head_dim and their own fp32 cos/sin table, in the eager
float32 order, in one kernel launch.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "Rope3dError", "Tables", "load_library", "rope3d_build_tables", "rope3d_apply_pair",
    "rope3d_apply_pair_host", "rope3d_preflight", "rope3d_axis_table_host",
    "rope3d_tables_read", "rope3d_cache_stats", "rope3d_cache_clear", "rope3d_gate_set_mode",
    "rope3d_gate_get_mode", "rope3d_gate_reset", "rope3d_gate_verdict",
    "rope3d_testing_corrupt_gate", "rope3d_last_launch", "rope3d_status_string",
    "rope3d_release_scratch", "rope3d_testing_fastdiv", "rope3d_testing_host_tables",
    "rope3d_testing_max_units_per_launch", "rope3d_apply_pair_noalloc",
    "STATUS", "BF16", "F32", "F16", "GATE_OFF", "GATE_FIRST", "LIB_PATH",
    "rope3d_apply_pair_strided", "rope3d_preflight_strided", "view_strides",
    "rope3d_patchify", "rope3d_unpatchify", "rope3d_patchify_check", "rope3d_patchify_last_kernel",
    "rope3d_apply_neox", "rope3d_neox_check", "rope3d_neox_cache_host", "rope3d_neox_last_kernel",
    "rope3d_na3d", "rope3d_na3d_rotate_once", "rope3d_na3d_preflight", "rope3d_debug_bounds",
    "rope3d_testing_debug_shrink_tables", "rope3d_dit_freqs_host", "rope3d_cache_retired",
    "rope3d_testing_na3d_kernel", "rope3d_testing_na3d_last_kernel", "rope3d_testing_na3d_per_cta",
    "rope3d_testing_na3d_wait_timeouts",
]

HERE = os.path.dirname(os.path.abspath(__file__))
# The library this module loads; ROPE3D_LIB names another build of it (for
# example the bounds-checking debug build) to load instead.
LIB_PATH = os.environ.get("ROPE3D_LIB") or os.path.join(HERE, "_build", "librope3d.so")

BF16, F32, F16 = 0, 1, 2
GATE_OFF, GATE_FIRST = 0, 1
STATUS = {
    0: "OK", -1: "ERR_NULL", -2: "ERR_SHAPE", -3: "ERR_DTYPE", -4: "ERR_ALIGN",
    -5: "ERR_ALIAS", -6: "ERR_DEVICE", -7: "ERR_PARITY", -8: "ERR_CUDA", -9: "ERR_TABLES",
    -10: "ERR_NOMEM", -11: "ERR_ARG", -12: "ERR_SCRATCH",
}

_lock = threading.Lock()
_lib = None


class Rope3dError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        self.name = STATUS.get(status, str(status))
        msg = rope3d_status_string(status) if _lib is not None else self.name
        super().__init__(f"{what}: {msg}" if what else msg)


def _declare(lib):
    c = ctypes
    i64, i32, vp, dbl = c.c_int64, c.c_int32, c.c_void_p, c.c_double
    sig = {
        "rope3d_build_tables": ([i64, i64, i64, vp, dbl, vp, vp], c.c_int),
        "rope3d_release_tables": ([vp], c.c_int),
        "rope3d_retain_tables": ([vp], c.c_int),
        "rope3d_apply_pair": ([vp, vp, vp, vp, vp] + [i64] * 6 + [vp, i32, vp], c.c_int),
        "rope3d_apply_pair_host": ([vp, vp, vp, vp, vp] + [i64] * 6 + [vp, i32, vp], c.c_int),
        "rope3d_release_scratch": ([], c.c_int),
        "rope3d_preflight": ([vp, vp, vp, vp, vp] + [i64] * 6 + [vp, i32, i32], c.c_int),
        "rope3d_axis_table_host": ([i64, i64, dbl, vp, vp], c.c_int),
        "rope3d_dit_freqs_host": ([i64, i64, dbl, i32, vp], c.c_int),
        "rope3d_tables_info": ([vp, vp, vp, vp], c.c_int),
        "rope3d_tables_read": ([vp, i32, i32, vp, vp], c.c_int),
        "rope3d_cache_stats": ([vp, vp, vp, vp], c.c_int),
        "rope3d_cache_clear": ([], c.c_int),
        "rope3d_cache_retired": ([vp], c.c_int),
        "rope3d_testing_na3d_kernel": ([i32], c.c_int),
        "rope3d_testing_na3d_last_kernel": ([], c.c_int),
        "rope3d_testing_na3d_per_cta": ([c.c_int32], c.c_int),
        "rope3d_testing_na3d_wait_timeouts": ([vp, i32], c.c_int),
        "rope3d_gate_set_mode": ([i32], c.c_int),
        "rope3d_gate_get_mode": ([], c.c_int),
        "rope3d_gate_reset": ([], c.c_int),
        "rope3d_gate_verdict": ([i64] * 6 + [vp, dbl, i32], c.c_int),
        "rope3d_testing_corrupt_gate": ([i32], c.c_int),
        "rope3d_last_launch": ([vp, vp], c.c_int),
        "rope3d_status_string": ([c.c_int], c.c_char_p),
        "rope3d_abi_version": ([], c.c_int),
        "rope3d_testing_fastdiv": ([i64, i64], i64),
        "rope3d_testing_host_tables": ([i32], c.c_int),
        "rope3d_testing_max_units_per_launch": ([i64], c.c_int),
        "rope3d_debug_bounds": ([vp, i32], c.c_int),
        "rope3d_testing_debug_shrink_tables": ([i32], c.c_int),
        "rope3d_apply_pair_noalloc": ([vp, vp, vp, vp] + [i64] * 6 + [vp, dbl, i32, vp], c.c_int),
        "rope3d_apply_pair_strided": ([vp, vp, vp, vp, vp] + [i64] * 6 + [vp, i32] + [vp] * 4 + [vp],
                                      c.c_int),
        "rope3d_patchify": ([vp, vp] + [i64] * 6 + [i32, vp], c.c_int),
        "rope3d_unpatchify": ([vp, vp] + [i64] * 6 + [i32, vp], c.c_int),
        "rope3d_patchify_check": ([vp, vp] + [i64] * 6 + [i32], c.c_int),
        "rope3d_patchify_last_kernel": ([], c.c_int),
        "rope3d_apply_neox": ([vp] * 6 + [i64] * 5 + [i32, vp, vp], c.c_int),
        "rope3d_neox_check": ([vp] * 6 + [i64] * 5 + [i32, vp], c.c_int),
        "rope3d_neox_cache_host": ([i64, i64, dbl, vp], c.c_int),
        "rope3d_neox_last_kernel": ([], c.c_int),
        "rope3d_na3d": ([vp] * 5 + [i64] * 6 + [vp, vp, i32, vp], c.c_int),
        "rope3d_na3d_rotate_once": ([vp] * 6 + [i64] * 6 + [vp, vp, vp], c.c_int),
        "rope3d_na3d_preflight": ([vp] * 6 + [i64] * 6 + [vp, vp, i32, i32], c.c_int),
        "rope3d_preflight_strided": ([vp, vp, vp, vp, vp] + [i64] * 6 + [vp, i32] + [vp] * 4 + [i32],
                                     c.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def load_library(path: str | None = None):
    """Load the built library (fails loudly when it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise ImportError(
                    f"{p} is missing: build the CUDA library first "
                    "(python -m rope_rope3d_apply_gb300.build)")
            _lib = _declare(ctypes.CDLL(p))
    return _lib


def _check(rc: int, what: str):
    if rc != 0:
        raise Rope3dError(rc, what)


def _split(split):
    if len(split) != 3:
        raise ValueError("split must have three entries (d_T, d_H, d_W)")
    return (ctypes.c_int32 * 3)(*[int(v) for v in split])


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if hasattr(x, "ctypes"):
        return int(x.ctypes.data)
    raise TypeError(f"cannot take a pointer of {type(x)!r}")


def _stream(stream, like=None) -> int:
    if stream is None:
        if like is not None and getattr(like, "is_cuda", False):
            import torch

            return int(torch.cuda.current_stream(like.device).cuda_stream)
        return 0
    if hasattr(stream, "cuda_stream"):
        return int(stream.cuda_stream)
    return int(stream)


def _dtype_code(x) -> int:
    dt = str(getattr(x, "dtype", ""))
    if dt in ("torch.bfloat16", "uint16"):
        return BF16
    if dt in ("torch.float32", "float32"):
        return F32
    if dt in ("torch.float16", "float16"):
        return F16
    raise TypeError(f"unsupported dtype {dt} (bfloat16, float16 or float32)")


def _contiguous(x) -> bool:
    if hasattr(x, "is_contiguous"):
        return bool(x.is_contiguous())
    if hasattr(x, "flags"):
        return bool(x.flags["C_CONTIGUOUS"])
    return True


class Tables:
    """One reference to a cached table set; released by close() or on
    garbage collection."""

    def __init__(self, handle: int):
        self.handle = handle
        dims = (ctypes.c_int64 * 3)()
        split = (ctypes.c_int32 * 3)()
        base = ctypes.c_double()
        _check(load_library().rope3d_tables_info(handle, dims, split, ctypes.byref(base)),
               "rope3d_tables_info")
        self.T, self.H, self.W = (int(v) for v in dims)
        self.split = tuple(int(v) for v in split)
        self.base = float(base.value)

    def close(self):
        if self.handle:
            load_library().rope3d_release_tables(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def rope3d_build_tables(T: int, H: int, W: int, split, base: float = 10000.0,
                        stream=None) -> Tables:
    out = ctypes.c_void_p()
    _check(load_library().rope3d_build_tables(int(T), int(H), int(W), _split(split),
                                              float(base), _stream(stream),
                                              ctypes.byref(out)), "rope3d_build_tables")
    return Tables(out.value)


def _grid_geometry(q, T: int, H: int, W: int):
    """(B, heads, head_dim) of q laid out as [B, T*H*W, heads, head_dim] or
    [B, T, H, W, heads, head_dim] over the grid (T, H, W)."""
    shape = tuple(int(v) for v in q.shape)
    grid = (int(T), int(H), int(W))
    if len(shape) == 6:
        if shape[1:4] != grid:
            raise ValueError(f"q grid {shape[1:4]} != the call's grid {grid}")
        return shape[0], shape[4], shape[5]
    if len(shape) == 4:
        N = grid[0] * grid[1] * grid[2]
        if shape[1] != N:
            raise ValueError(f"q has {shape[1]} tokens, the grid {grid} has {N}")
        return shape[0], shape[2], shape[3]
    raise ValueError("q must be [B, T*H*W, heads, head_dim] or [B, T, H, W, heads, head_dim]")


def _geometry(q, tables: Tables):
    return _grid_geometry(q, tables.T, tables.H, tables.W)


def _marshal_grid(q, k, q_out, k_out, T: int, H: int, W: int):
    """Checks that the four buffers are contiguous, of q's shape and of q's
    dtype, and that q covers the grid; returns (B, heads, head_dim, dtype).
    The C ABI takes bare pointers and cannot see a buffer's extent, so these
    checks are what keeps a call inside the caller's memory."""
    for name, t in (("q", q), ("k", k), ("q_out", q_out), ("k_out", k_out)):
        if not _contiguous(t):
            raise ValueError(f"{name} must be contiguous")
        if tuple(t.shape) != tuple(q.shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, q has {tuple(q.shape)}")
    B, heads, head_dim = _grid_geometry(q, T, H, W)
    dt = _dtype_code(q)
    for t in (k, q_out, k_out):
        if _dtype_code(t) != dt:
            raise TypeError("q, k, q_out and k_out must have one dtype")
    return B, heads, head_dim, dt


def _marshal(q, k, q_out, k_out, tables: Tables):
    return _marshal_grid(q, k, q_out, k_out, tables.T, tables.H, tables.W)


def rope3d_apply_pair(q, k, tables: Tables, q_out=None, k_out=None, stream=None):
    """Rotate device tensors q and k; returns (q_out, k_out). Outputs are
    allocated with torch.empty_like when not given."""
    if q_out is None or k_out is None:
        import torch

        q_out = torch.empty_like(q) if q_out is None else q_out
        k_out = torch.empty_like(k) if k_out is None else k_out
    B, heads, head_dim, dt = _marshal(q, k, q_out, k_out, tables)
    rc = load_library().rope3d_apply_pair(
        _ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), tables.handle, B, tables.T, tables.H,
        tables.W, heads, head_dim, _split(tables.split), dt, _stream(stream, q))
    _check(rc, "rope3d_apply_pair")
    return q_out, k_out


def rope3d_apply_pair_host(q, k, q_out, k_out, tables: Tables, stream=None):
    """Rotate host buffers (torch CPU tensors, ideally pinned, or numpy arrays;
    bf16 may be given as uint16 bit patterns). Returns when the outputs are in
    host memory."""
    B, heads, head_dim, dt = _marshal(q, k, q_out, k_out, tables)
    rc = load_library().rope3d_apply_pair_host(
        _ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), tables.handle, B, tables.T, tables.H,
        tables.W, heads, head_dim, _split(tables.split), dt, _stream(stream))
    _check(rc, "rope3d_apply_pair_host")
    return q_out, k_out


def rope3d_apply_pair_noalloc(q, k, q_out, k_out, T: int, H: int, W: int, split,
                              base: float = 10000.0, stream=None):
    """rope3d_apply_pair without a table handle, for callers that cannot
    allocate device memory: the tables go into the library's fixed 64 KiB
    static table area (see include/rope3d.h). q_out and k_out are required;
    this function allocates nothing. The buffers are checked as for
    rope3d_apply_pair: contiguous, one shape and one dtype, covering the grid."""
    B, heads, head_dim, dt = _marshal_grid(q, k, q_out, k_out, T, H, W)
    rc = load_library().rope3d_apply_pair_noalloc(
        _ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), B, int(T), int(H), int(W), heads, head_dim,
        _split(split), float(base), dt, _stream(stream, q))
    _check(rc, "rope3d_apply_pair_noalloc")
    return q_out, k_out


def view_strides(x, T: int, H: int, W: int):
    """(B, heads, head_dim) and the element strides of (batch, t, h, w, head)
    of a [B, T, H, W, heads, head_dim] or [B, T*H*W, heads, head_dim] view
    whose channels are contiguous."""
    shape = tuple(int(v) for v in x.shape)
    if hasattr(x, "stride") and callable(x.stride):
        st = tuple(int(v) for v in x.stride())
    else:  # numpy: byte strides
        st = tuple(int(v) // x.itemsize for v in x.strides)
    if st[-1] != 1 and shape[-1] > 1:
        raise ValueError("channels (the last dimension) must be contiguous")
    if len(shape) == 6:
        if shape[1:4] != (T, H, W):
            raise ValueError(f"view grid {shape[1:4]} != tables grid {(T, H, W)}")
        return (shape[0], shape[4], shape[5]), st[:5]
    if len(shape) == 4:
        if shape[1] != T * H * W:
            raise ValueError(f"view has {shape[1]} tokens, the tables' grid has {T * H * W}")
        sn = st[1]
        return (shape[0], shape[2], shape[3]), (st[0], H * W * sn, W * sn, sn, st[2])
    raise ValueError("expected [B, T*H*W, heads, head_dim] or [B, T, H, W, heads, head_dim]")


def _strides_arg(st):
    return (ctypes.c_int64 * 5)(*[int(v) for v in st])


def rope3d_apply_pair_strided(q, k, tables: Tables, q_out=None, k_out=None, stream=None):
    """Rotate strided device views (e.g. Q and K slices of a fused QKV
    buffer); q_out=q and k_out=k rotate in place. Missing outputs are
    allocated contiguous with torch.empty."""
    if q_out is None or k_out is None:
        import torch

        q_out = torch.empty(q.shape, dtype=q.dtype, device=q.device) if q_out is None else q_out
        k_out = torch.empty(k.shape, dtype=k.dtype, device=k.device) if k_out is None else k_out
    geo, sts = None, []
    for name, t in (("q", q), ("k", k), ("q_out", q_out), ("k_out", k_out)):
        g, st = view_strides(t, tables.T, tables.H, tables.W)
        if geo is not None and g != geo:
            raise ValueError(f"{name} has (B, heads, head_dim) {g}, q has {geo}")
        geo = g
        sts.append(_strides_arg(st))
    dt = _dtype_code(q)
    for t in (k, q_out, k_out):
        if _dtype_code(t) != dt:
            raise TypeError("q, k, q_out and k_out must have one dtype")
    B, heads, head_dim = geo
    rc = load_library().rope3d_apply_pair_strided(
        _ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), tables.handle, B, tables.T, tables.H,
        tables.W, heads, head_dim, _split(tables.split), dt, *sts, _stream(stream, q))
    _check(rc, "rope3d_apply_pair_strided")
    return q_out, k_out


def rope3d_preflight_strided(ptrs, strides, tables, B, T, H, W, heads, head_dim, split, dtype,
                             check_device=True) -> int:
    """Status that rope3d_apply_pair_strided would return before launching.
    ptrs: (q, k, q_out, k_out) addresses; strides: four 5-tuples (or None)."""
    handle = tables.handle if isinstance(tables, Tables) else (tables or 0)
    sts = [None if st is None else _strides_arg(st) for st in strides]
    return load_library().rope3d_preflight_strided(
        *[_ptr(p) for p in ptrs], handle, int(B), int(T), int(H), int(W), int(heads),
        int(head_dim), _split(split), int(dtype), *sts, 1 if check_device else 0)


def _elem_bytes(t) -> int:
    if hasattr(t, "element_size"):
        return int(t.element_size())
    return int(t.itemsize)


def rope3d_patchify(x, p: int, y=None, stream=None):
    """Space-to-depth (B, C, F, H, W) -> (B, C*p*p, F, H/p, W/p), channels in
    the order (channel, width offset, height offset). x and y are contiguous
    device tensors; y is allocated with torch.empty when not given."""
    B, C, F, H, W = (int(v) for v in x.shape)
    if y is None:
        import torch

        y = torch.empty((B, C * p * p, F, H // p, W // p), dtype=x.dtype, device=x.device)
    for name, t in (("x", x), ("y", y)):
        if not _contiguous(t):
            raise ValueError(f"{name} must be contiguous")
    if tuple(int(v) for v in y.shape) != (B, C * p * p, F, H // p, W // p) or y.dtype != x.dtype:
        raise ValueError("y must have shape (B, C*p*p, F, H/p, W/p) and the dtype of x")
    _check(load_library().rope3d_patchify(_ptr(x), _ptr(y), B, C, F, H, W, int(p),
                                          _elem_bytes(x), _stream(stream, x)), "rope3d_patchify")
    return y


def rope3d_unpatchify(y, p: int, x=None, stream=None):
    """Inverse of rope3d_patchify: (B, C*p*p, F, H/p, W/p) -> (B, C, F, H, W)."""
    B, Cpp, F, Hp, Wp = (int(v) for v in y.shape)
    if Cpp % (p * p):
        raise ValueError("channels must be a multiple of p*p")
    C, H, W = Cpp // (p * p), Hp * p, Wp * p
    if x is None:
        import torch

        x = torch.empty((B, C, F, H, W), dtype=y.dtype, device=y.device)
    for name, t in (("x", x), ("y", y)):
        if not _contiguous(t):
            raise ValueError(f"{name} must be contiguous")
    if tuple(int(v) for v in x.shape) != (B, C, F, H, W) or x.dtype != y.dtype:
        raise ValueError("x must have shape (B, C, F, H, W) and the dtype of y")
    _check(load_library().rope3d_unpatchify(_ptr(y), _ptr(x), B, C, F, H, W, int(p),
                                            _elem_bytes(y), _stream(stream, y)), "rope3d_unpatchify")
    return x


def rope3d_patchify_check(src, dst, B, C, F, H, W, p, elem_bytes) -> str:
    """Name of the status the host-side checks give (no GPU needed)."""
    return STATUS[load_library().rope3d_patchify_check(_ptr(src), _ptr(dst), int(B), int(C), int(F),
                                                       int(H), int(W), int(p), int(elem_bytes))]


def rope3d_patchify_last_kernel() -> int:
    return int(load_library().rope3d_patchify_last_kernel())


def rope3d_neox_cache_host(max_position: int, rotary_dim: int, base: float = 10000.0):
    """Host cos_sin_cache [max_position, rotary_dim] = [cos | sin] (float32 numpy)."""
    import numpy as np

    c = np.empty((max_position, rotary_dim), np.float32)
    _check(load_library().rope3d_neox_cache_host(int(max_position), int(rotary_dim), float(base),
                                                 _ptr(c)), "rope3d_neox_cache_host")
    return c


def rope3d_apply_neox(q, k, positions, cos_sin_cache, q_out=None, k_out=None,
                      invalid_count=None, stream=None):
    """NeoX-style RoPE (Gemma3): q [tokens, q_heads, head_dim], k [tokens,
    k_heads, head_dim], positions int64 [tokens], cos_sin_cache float32
    [max_position, head_dim], all on the device. q_out=q / k_out=k rotate in
    place; missing outputs are allocated with torch.empty_like."""
    if q_out is None or k_out is None:
        import torch

        q_out = torch.empty_like(q) if q_out is None else q_out
        k_out = torch.empty_like(k) if k_out is None else k_out
    for name, t in (("q", q), ("k", k), ("q_out", q_out), ("k_out", k_out),
                    ("positions", positions), ("cos_sin_cache", cos_sin_cache)):
        if not _contiguous(t):
            raise ValueError(f"{name} must be contiguous")
    if q.dim() != 3 or k.dim() != 3 or q.shape[0] != k.shape[0] or q.shape[2] != k.shape[2]:
        raise ValueError("q and k must be [tokens, heads, head_dim] with one tokens and head_dim")
    if tuple(q_out.shape) != tuple(q.shape) or tuple(k_out.shape) != tuple(k.shape):
        raise ValueError("outputs must have the shapes of q and k")
    tokens, q_heads, head_dim = (int(v) for v in q.shape)
    k_heads = int(k.shape[1])
    if str(positions.dtype) != "torch.int64" or positions.numel() != tokens:
        raise ValueError("positions must be int64 with one entry per token")
    if str(cos_sin_cache.dtype) != "torch.float32" or cos_sin_cache.dim() != 2 or \
            int(cos_sin_cache.shape[1]) != head_dim:
        raise ValueError("cos_sin_cache must be float32 [max_position, head_dim]")
    dt = _dtype_code(q)
    for t in (k, q_out, k_out):
        if _dtype_code(t) != dt:
            raise TypeError("q, k, q_out and k_out must have one dtype")
    rc = load_library().rope3d_apply_neox(
        _ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), _ptr(positions), _ptr(cos_sin_cache),
        int(cos_sin_cache.shape[0]), tokens, q_heads, k_heads, head_dim, dt,
        _ptr(invalid_count), _stream(stream, q))
    _check(rc, "rope3d_apply_neox")
    return q_out, k_out


def rope3d_neox_check(ptrs, max_position, tokens, q_heads, k_heads, head_dim, dtype) -> str:
    """Status name of the host-side checks of rope3d_apply_neox. ptrs: (q, k,
    q_out, k_out, positions, cache, invalid_count) addresses."""
    return STATUS[load_library().rope3d_neox_check(*[_ptr(p) for p in ptrs[:6]], int(max_position),
                                                   int(tokens), int(q_heads), int(k_heads),
                                                   int(head_dim), int(dtype), _ptr(ptrs[6]))]


def rope3d_neox_last_kernel() -> int:
    return int(load_library().rope3d_neox_last_kernel())


def rope3d_na3d(q, k, v, tables: Tables, kernel_size, out=None, apply_rope: bool = True,
                stream=None):
    """3D neighbourhood attention over [B, T*H*W, heads, 128] (or 6-D) bf16
    device tensors, with Q and K rotated first when apply_rope (K once, into
    scratch the library takes from its pool; Q inside the attention)."""
    if out is None:
        import torch

        out = torch.empty_like(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if not _contiguous(t):
            raise ValueError(f"{name} must be contiguous")
        if tuple(t.shape) != tuple(q.shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, q has {tuple(q.shape)}")
        if _dtype_code(t) != BF16:
            raise TypeError("rope3d_na3d takes bf16 tensors")
    B, heads, head_dim = _geometry(q, tables)
    ks = (ctypes.c_int32 * 3)(*[int(x) for x in kernel_size])
    rc = load_library().rope3d_na3d(_ptr(q), _ptr(k), _ptr(v), _ptr(out), tables.handle, B,
                                    tables.T, tables.H, tables.W, heads, head_dim,
                                    _split(tables.split), ks, 1 if apply_rope else 0,
                                    _stream(stream, q))
    _check(rc, "rope3d_na3d")
    return out


def rope3d_na3d_rotate_once(q, k, v, tables: Tables, kernel_size, out=None, k_rot=None,
                            stream=None):
    """rope3d_na3d with Q and K rotated, each element once: K is rotated into
    k_rot (allocated when None; k_rot=k rotates in place), then the attention
    rotates its Q tiles. Returns (out, k_rot)."""
    import torch

    if out is None:
        out = torch.empty_like(q)
    if k_rot is None:
        k_rot = torch.empty_like(k)
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("k_rot", k_rot)):
        if not _contiguous(t):
            raise ValueError(f"{name} must be contiguous")
        if tuple(t.shape) != tuple(q.shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, q has {tuple(q.shape)}")
        if _dtype_code(t) != BF16:
            raise TypeError("rope3d_na3d_rotate_once takes bf16 tensors")
    B, heads, head_dim = _geometry(q, tables)
    ks = (ctypes.c_int32 * 3)(*[int(x) for x in kernel_size])
    rc = load_library().rope3d_na3d_rotate_once(
        _ptr(q), _ptr(k), _ptr(v), _ptr(k_rot), _ptr(out), tables.handle, B, tables.T, tables.H,
        tables.W, heads, head_dim, _split(tables.split), ks, _stream(stream, q))
    _check(rc, "rope3d_na3d_rotate_once")
    return out, k_rot


def rope3d_na3d_preflight(q, k, v, k_rot, out, tables, B, T, H, W, heads, kernel_size,
                          apply_rope=True, head_dim=128, split=None, check_device=True) -> str:
    """Status name that rope3d_na3d (k_rot None) or rope3d_na3d_rotate_once
    would return before launching; pointers may be plain integers."""
    handle = tables.handle if isinstance(tables, Tables) else (tables or 0)
    if split is None and isinstance(tables, Tables):
        split = tables.split
    ks = (ctypes.c_int32 * 3)(*[int(x) for x in kernel_size])
    rc = load_library().rope3d_na3d_preflight(
        _ptr(q), _ptr(k), _ptr(v), _ptr(k_rot), _ptr(out), handle, int(B), int(T), int(H),
        int(W), int(heads), int(head_dim), _split(split) if split is not None else None, ks,
        1 if apply_rope else 0, 1 if check_device else 0)
    return STATUS.get(rc, str(rc))


def rope3d_preflight(q, k, q_out, k_out, tables, B, T, H, W, heads, head_dim, split, dtype,
                     check_device=True) -> int:
    """Status that rope3d_apply_pair would return before launching (no launch)."""
    handle = tables.handle if isinstance(tables, Tables) else (tables or 0)
    return load_library().rope3d_preflight(
        _ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), handle, int(B), int(T), int(H), int(W),
        int(heads), int(head_dim), _split(split) if split is not None else None, int(dtype),
        1 if check_device else 0)


def rope3d_axis_table_host(length: int, dim: int, base: float = 10000.0):
    import numpy as np

    c = np.empty((length, dim // 2), np.float32)
    s = np.empty((length, dim // 2), np.float32)
    _check(load_library().rope3d_axis_table_host(int(length), int(dim), float(base),
                                                 _ptr(c), _ptr(s)), "rope3d_axis_table_host")
    return c, s


def rope3d_dit_freqs_host(dim: int, num_rope_elems: int, theta: float = 10000.0,
                          double_precision: bool = True):
    """The LTX DiT's RoPE frequency vector, float32 [dim // num_rope_elems]
    (see rope3d_dit_freqs_host in include/rope3d.h)."""
    import numpy as np

    if dim <= 0 or num_rope_elems <= 0:
        raise ValueError("dim and num_rope_elems must be > 0")
    out = np.empty(max(dim // num_rope_elems, 1), dtype=np.float32)
    _check(load_library().rope3d_dit_freqs_host(int(dim), int(num_rope_elems), float(theta),
                                                int(bool(double_precision)), _ptr(out)),
           "rope3d_dit_freqs_host")
    return out


def rope3d_tables_read(tables: Tables, axis: int, from_device: bool = False):
    import numpy as np

    L = (tables.T, tables.H, tables.W)[axis]
    d = tables.split[axis]
    c = np.empty((L, d // 2), np.float32)
    s = np.empty((L, d // 2), np.float32)
    _check(load_library().rope3d_tables_read(tables.handle, int(axis), 1 if from_device else 0,
                                             _ptr(c), _ptr(s)), "rope3d_tables_read")
    return c, s


def rope3d_cache_stats() -> dict:
    v = [ctypes.c_int64() for _ in range(4)]
    _check(load_library().rope3d_cache_stats(*[ctypes.byref(x) for x in v]), "rope3d_cache_stats")
    return dict(zip(("entries", "hits", "misses", "evictions"), (x.value for x in v)))


def rope3d_testing_na3d_kernel(which: int):
    """0: the tensor-core attention where the geometry allows it (default);
    1: the same; 2: always the warp-MMA kernel."""
    _check(load_library().rope3d_testing_na3d_kernel(int(which)), "rope3d_testing_na3d_kernel")


def rope3d_testing_na3d_last_kernel() -> int:
    """1 tensor-core, 2 warp-MMA: the kernel of this thread's last attention launch."""
    return int(load_library().rope3d_testing_na3d_last_kernel())


def rope3d_testing_na3d_per_cta(on: bool):
    """True: rope3d_na3d with the RoPE runs the kernel form that rotates Q and
    every K tile inside each CTA (no scratch); False: the default."""
    _check(load_library().rope3d_testing_na3d_per_cta(1 if on else 0), "rope3d_testing_na3d_per_cta")


def rope3d_testing_na3d_wait_timeouts(reset: bool = True) -> int:
    """Bounded waits of the tensor-core attention that ran out (0 normally)."""
    n = ctypes.c_int64()
    _check(load_library().rope3d_testing_na3d_wait_timeouts(ctypes.byref(n), int(bool(reset))),
           "rope3d_testing_na3d_wait_timeouts")
    return int(n.value)


def rope3d_cache_retired() -> int:
    """Free released table buffers whose launches have completed; returns how
    many released buffers still wait for launches in flight."""
    n = ctypes.c_int64()
    _check(load_library().rope3d_cache_retired(ctypes.byref(n)), "rope3d_cache_retired")
    return int(n.value)


def rope3d_cache_clear():
    _check(load_library().rope3d_cache_clear(), "rope3d_cache_clear")


def rope3d_gate_set_mode(mode: int):
    _check(load_library().rope3d_gate_set_mode(int(mode)), "rope3d_gate_set_mode")


def rope3d_gate_get_mode() -> int:
    return int(load_library().rope3d_gate_get_mode())


def rope3d_gate_reset():
    _check(load_library().rope3d_gate_reset(), "rope3d_gate_reset")


def rope3d_gate_verdict(B, T, H, W, heads, head_dim, split, base, dtype) -> int:
    r = load_library().rope3d_gate_verdict(int(B), int(T), int(H), int(W), int(heads),
                                           int(head_dim), _split(split), float(base), int(dtype))
    if r < 0:
        raise Rope3dError(r, "rope3d_gate_verdict")
    return r


def rope3d_testing_corrupt_gate(count: int):
    _check(load_library().rope3d_testing_corrupt_gate(int(count)), "rope3d_testing_corrupt_gate")


def rope3d_testing_host_tables(on: bool):
    _check(load_library().rope3d_testing_host_tables(1 if on else 0), "rope3d_testing_host_tables")


def rope3d_testing_fastdiv(n: int, d: int) -> int:
    return int(load_library().rope3d_testing_fastdiv(int(n), int(d)))


def rope3d_testing_max_units_per_launch(n: int):
    _check(load_library().rope3d_testing_max_units_per_launch(int(n)),
           "rope3d_testing_max_units_per_launch")


def rope3d_debug_bounds(reset: bool = True):
    """(built_with_checks, failed_checks): the bounds checks of a debug build
    (see build(debug_bounds=True)); the count is cleared when reset."""
    n = ctypes.c_int64()
    rc = load_library().rope3d_debug_bounds(ctypes.byref(n), 1 if reset else 0)
    if rc < 0:
        _check(rc, "rope3d_debug_bounds")
    return bool(rc), int(n.value)


def rope3d_testing_debug_shrink_tables(n: int):
    _check(load_library().rope3d_testing_debug_shrink_tables(int(n)),
           "rope3d_testing_debug_shrink_tables")


def rope3d_last_launch():
    g, b = ctypes.c_int32(), ctypes.c_int32()
    kernel = load_library().rope3d_last_launch(ctypes.byref(g), ctypes.byref(b))
    return {"kernel": int(kernel), "grid": g.value, "block": b.value}


def rope3d_release_scratch():
    _check(load_library().rope3d_release_scratch(), "rope3d_release_scratch")


def rope3d_status_string(status: int) -> str:
    return load_library().rope3d_status_string(int(status)).decode()
