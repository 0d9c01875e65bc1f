"""rope3d_apply_pair_noalloc, the entry point for callers that cannot
allocate device memory (their device memory belongs to another allocator or a
fixed budget, or they must not take cudaMalloc's implicit synchronisation).
It takes no table handle and keeps the tables in the library's fixed static
device table area instead of a cudaMalloc'd cache entry.

Checked through the C ABI against rope3d_apply_pair and against the CPU
oracle, bit for bit (the same bar as every other GPU test; the library's
first-call gate does not run on this path), on two calls in a row: the second
call uses a smaller grid, so it reads an area whose tail still holds the first
call's tables. Both kernels are covered: the 16-byte vector kernel and the
per-pair kernel that unaligned buffers or narrow chunks take. This file is
collected last on purpose.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU hosts
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import rope_rope3d_apply_gb300 as r  # noqa: E402

DEV = torch.device("cuda:0")


def _to_device(a: np.ndarray, shp, dtype: str):
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if dtype == "bf16" \
        else torch.from_numpy(a)
    return t.reshape(shp).to(DEV)


def _host_bits(t) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return t.numpy().reshape(-1).view(np.uint32)


def _oracle_bits(a: np.ndarray) -> np.ndarray:
    return a if a.dtype == np.uint16 else a.view(np.uint32)


def _offset_empty(like, offset_elems: int):
    """An uninitialised buffer of like's shape that starts offset_elems
    elements into a larger allocation (4-byte aligned, not 16-byte aligned)."""
    big = torch.empty(like.numel() + offset_elems, dtype=like.dtype, device=DEV)
    return big[offset_elems:].view(like.shape)


def _check_case(q_np, k_np, shape6, split, dtype, base=10000.0, offset_elems=0):
    """One rope3d_apply_pair_noalloc call, compared with rope3d_apply_pair on
    the same inputs and with the oracle. Returns the kernel the reference call
    took (1 = vector, 2 = pair)."""
    B, T, H, W, heads, hd = shape6
    shp = (B, T * H * W, heads, hd)
    q, k = _to_device(q_np, shp, dtype), _to_device(k_np, shp, dtype)
    if offset_elems:
        qo, ko = _offset_empty(q, offset_elems), _offset_empty(k, offset_elems)
    else:
        qo, ko = torch.empty_like(q), torch.empty_like(k)
    r.rope3d_apply_pair_noalloc(q, k, qo, ko, T, H, W, split, base)
    torch.cuda.synchronize()
    tabs = r.rope3d_build_tables(T, H, W, split, base)
    want_q, want_k = r.rope3d_apply_pair(q, k, tabs, _offset_empty(q, offset_elems),
                                         _offset_empty(k, offset_elems))
    torch.cuda.synchronize()
    kernel = r.rope3d_last_launch()["kernel"]
    tabs.close()
    got_q, got_k = _host_bits(qo), _host_bits(ko)
    assert np.array_equal(got_q, _host_bits(want_q))
    assert np.array_equal(got_k, _host_bits(want_k))
    otabs = oracle.tables(T, H, W, split, base)
    assert np.array_equal(got_q, _oracle_bits(oracle.rope3d(q_np, shape6, split, otabs)))
    assert np.array_equal(got_k, _oracle_bits(oracle.rope3d(k_np, shape6, split, otabs)))
    return kernel


def test_noalloc_matches_apply_pair_and_oracle_on_two_calls_in_a_row():
    for name in ("stage5_w63", "stage0_f32"):
        w = synthetic.WORKLOADS[name]
        q_np, k_np = synthetic.qk(w)
        assert _check_case(q_np, k_np, w.shape6, w.split, w.dtype, w.base) == 1, name


def test_noalloc_per_pair_kernel_on_two_calls_in_a_row():
    # outputs 2 elements into their allocations: 4-byte aligned only
    w = synthetic.WORKLOADS["stage0"]
    q_np, k_np = synthetic.qk(w)
    assert _check_case(q_np, k_np, w.shape6, w.split, w.dtype, w.base, offset_elems=2) == 2
    # chunks of 2 channels (not a multiple of the 8-element vector), fp32 and bf16
    rng = np.random.default_rng(7)
    shape6 = (2, 3, 5, 7, 3, 6)
    n = int(np.prod(shape6))
    q32 = rng.standard_normal(n, dtype=np.float32)
    k32 = rng.standard_normal(n, dtype=np.float32)
    assert _check_case(q32, k32, shape6, (2, 2, 2), "f32") == 2
    qb = (q32.view(np.uint32) >> 16).astype(np.uint16)  # truncated to bf16 patterns
    kb = (k32.view(np.uint32) >> 16).astype(np.uint16)
    assert _check_case(qb, kb, shape6, (2, 2, 2), "bf16") == 2


def test_noalloc_rejects_tables_beyond_the_area():
    # W = 8200 positions of a 2-channel chunk: 8200 entries > 8192
    shp = (1, 8200, 1, 6)
    q = torch.randn(shp, device=DEV).to(torch.bfloat16)
    k = torch.randn(shp, device=DEV).to(torch.bfloat16)
    qo = torch.full(shp, 5.0, dtype=torch.bfloat16, device=DEV)
    ko = torch.full(shp, 5.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_apply_pair_noalloc(q, k, qo, ko, 1, 1, 8200, (2, 2, 2))
    assert e.value.name == "ERR_SCRATCH"
    torch.cuda.synchronize()
    assert torch.all(qo == 5.0) and torch.all(ko == 5.0)


def test_noalloc_binding_rejects_a_grid_or_dtype_mismatch():
    shp6 = (1, 2, 4, 4, 2, 48)
    q = torch.randn(shp6, device=DEV).to(torch.bfloat16)
    k = torch.randn(shp6, device=DEV).to(torch.bfloat16)
    qo = torch.full(shp6, 5.0, dtype=torch.bfloat16, device=DEV)
    ko = torch.full(shp6, 5.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):      # a 6-D view of another grid
        r.rope3d_apply_pair_noalloc(q, k, qo, ko, 2, 4, 8, (16, 16, 16))
    with pytest.raises(ValueError):      # 4-D, token count of another grid
        r.rope3d_apply_pair_noalloc(q.view(1, 32, 2, 48), k.view(1, 32, 2, 48),
                                    qo.view(1, 32, 2, 48), ko.view(1, 32, 2, 48),
                                    2, 4, 2, (16, 16, 16))
    q32 = q.float()
    with pytest.raises(TypeError):       # fp32 q with bf16 outputs
        r.rope3d_apply_pair_noalloc(q32, q32, qo, ko, 2, 4, 4, (16, 16, 16))
    torch.cuda.synchronize()
    assert torch.all(qo == 5.0) and torch.all(ko == 5.0)


def test_noalloc_refuses_a_capturing_stream():
    w = synthetic.WORKLOADS["tiny"]
    shp = (w.B, w.N, w.heads, w.head_dim)
    q = torch.randn(shp, device=DEV).to(torch.bfloat16)
    k = torch.randn(shp, device=DEV).to(torch.bfloat16)
    qo = torch.full(shp, 5.0, dtype=torch.bfloat16, device=DEV)
    ko = torch.full(shp, 5.0, dtype=torch.bfloat16, device=DEV)
    r.rope3d_apply_pair_noalloc(q, k, qo, ko, w.T, w.H, w.W, w.split)  # set-up outside capture
    torch.cuda.synchronize()
    qo.fill_(5.0)
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    refused = None
    with torch.cuda.graph(g, stream=side, capture_error_mode="relaxed"):
        qo.add_(0.0)  # something for the graph to hold
        try:
            r.rope3d_apply_pair_noalloc(q, k, qo, ko, w.T, w.H, w.W, w.split, stream=side)
        except r.Rope3dError as e:
            refused = e.name
    assert refused == "ERR_ARG"
    torch.cuda.synchronize()
    assert torch.all(qo == 5.0)
