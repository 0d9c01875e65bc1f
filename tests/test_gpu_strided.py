"""GPU parity of the wider variants against the CPU oracle: IEEE fp16, strided
views (Q and K read straight out of fused QKV buffers, crops of a larger
grid) and rotation in place. The oracle rotates contiguous copies of the
same views; the bar is bit-exactness, as for the contiguous path."""
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
TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
CODE = {"bf16": r.BF16, "f16": r.F16, "f32": r.F32}


@pytest.fixture(autouse=True)
def _fresh_gate():
    r.rope3d_gate_reset()
    r.rope3d_gate_set_mode(r.GATE_FIRST)
    yield
    r.rope3d_gate_reset()


def draw(n, seed, which, dtype):
    """Seeded values as the numpy array the oracle takes (uint16 bits for the
    16-bit types)."""
    if dtype == "f16":
        return synthetic.normal(n, 1.0, seed, which, "f32").astype(np.float16).view(np.uint16)
    return synthetic.normal(n, 1.0, seed, which, dtype)


def to_torch(a: np.ndarray, dtype: str):
    if dtype == "f32":
        return torch.from_numpy(a.copy())
    return torch.from_numpy(a.view(np.int16).copy()).view(TORCH_DT[dtype])


def to_numpy(t) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return t.numpy().reshape(-1)


def bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) if a.dtype == np.float32 else a


def assert_bit_exact(got, want, what=""):
    g, w = bits(got), bits(want)
    if g.dtype == np.uint32:
        nan = lambda b: (b & 0x7FFFFFFF) > 0x7F800000  # noqa: E731
    else:
        nan = lambda b: (b & 0x7FFF) > (0x7C00 if what.endswith("f16") else 0x7F80)  # noqa: E731
    bad = (g != w) & ~(nan(g) & nan(w))
    assert not bad.any(), f"{what}: {int(bad.sum())} mismatches, first at {np.flatnonzero(bad)[:5]}"


def oracle_rotate(x_np, shape6, split, dtype):
    tabs = oracle.tables(*shape6[1:4], split)
    return oracle.rope3d(x_np, shape6, split, tabs, f16=(dtype == "f16"))


# ---------------------------------------------------------------------------
# fp16, contiguous
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shape6,split,kernel", [
    ((1, 4, 16, 16, 16, 64), (16, 24, 24), 1),
    ((2, 3, 5, 7, 3, 24), (6, 8, 10), 2),
    ((1, 16, 64, 63, 16, 128), (32, 48, 48), 1),
])
def test_fp16_bit_exact(shape6, split, kernel):
    n = int(np.prod(shape6))
    q_np, k_np = draw(n, 60, 0, "f16"), draw(n, 60, 1, "f16")
    B, T, H, W, heads, hd = shape6
    shp = (B, T * H * W, heads, hd)
    q = to_torch(q_np, "f16").reshape(shp).to(DEV)
    k = to_torch(k_np, "f16").reshape(shp).to(DEV)
    tabs = r.rope3d_build_tables(T, H, W, split)
    qo, ko = r.rope3d_apply_pair(q, k, tabs)
    torch.cuda.synchronize()
    assert r.rope3d_last_launch()["kernel"] == kernel
    assert r.rope3d_gate_verdict(B, T, H, W, heads, hd, split, 10000.0, r.F16) == 1
    assert_bit_exact(to_numpy(qo), oracle_rotate(q_np, shape6, split, "f16"), "Q f16")
    assert_bit_exact(to_numpy(ko), oracle_rotate(k_np, shape6, split, "f16"), "K f16")
    tabs.close()


def test_fp16_special_values():
    shape6, split = (2, 3, 4, 5, 2, 32), (8, 8, 16)
    n = int(np.prod(shape6))
    g = np.random.Generator(np.random.PCG64(61))
    x = synthetic.normal(n, 1.0, 61, 0, "f32")
    pool = np.array([0.0, -0.0, 2.0 ** -24, -(2.0 ** -20), 6e-5, 65504.0, -65504.0, 60000.0,
                     np.inf, -np.inf, np.nan, 1.0], np.float32)
    pick = g.integers(0, n, n // 4)
    x[pick] = pool[g.integers(0, pool.size, pick.size)]
    x[g.integers(0, n, n // 8)] *= np.float32(2.0 ** -12)   # products into the subnormal range
    q_np = x.astype(np.float16).view(np.uint16)
    k_np = q_np[::-1].copy()
    B, T, H, W, heads, hd = shape6
    shp = (B, T * H * W, heads, hd)
    q = to_torch(q_np, "f16").reshape(shp).to(DEV)
    k = to_torch(k_np, "f16").reshape(shp).to(DEV)
    tabs = r.rope3d_build_tables(T, H, W, split)
    qo, ko = r.rope3d_apply_pair(q, k, tabs)
    torch.cuda.synchronize()
    assert_bit_exact(to_numpy(qo), oracle_rotate(q_np, shape6, split, "f16"), "Q f16")
    assert_bit_exact(to_numpy(ko), oracle_rotate(k_np, shape6, split, "f16"), "K f16")
    tabs.close()


# ---------------------------------------------------------------------------
# strided views and in place
# ---------------------------------------------------------------------------

def _qkv(B, N, heads, hd, dtype, seed, interleaved: bool):
    """A fused QKV buffer ([B, N, 3, heads, hd] or [B, N, heads, 3, hd]) and
    its q, k, v views ([B, N, heads, hd])."""
    n = B * N * 3 * heads * hd
    buf_np = draw(n, seed, 0, dtype)
    if interleaved:
        buf = to_torch(buf_np, dtype).reshape(B, N, heads, 3, hd).to(DEV)
        return buf, buf[:, :, :, 0], buf[:, :, :, 1], buf[:, :, :, 2]
    buf = to_torch(buf_np, dtype).reshape(B, N, 3, heads, hd).to(DEV)
    return buf, buf[:, :, 0], buf[:, :, 1], buf[:, :, 2]


def _host(view, dtype):
    return to_numpy(view)


def bitview(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("inplace", [False, True])
def test_fused_qkv_views(dtype, interleaved, inplace):
    w = synthetic.WORKLOADS["stage0"]
    B, T, H, W, heads, hd, split = w.B, w.T, w.H, w.W, w.heads, w.head_dim, w.split
    buf, q, k, v = _qkv(B, w.N, heads, hd, dtype, 62, interleaved)
    q_np, k_np, v_before = _host(q, dtype), _host(k, dtype), v.clone()
    tabs = r.rope3d_build_tables(T, H, W, split)
    if inplace:
        qo, ko = r.rope3d_apply_pair_strided(q, k, tabs, q, k)
    else:
        qo, ko = r.rope3d_apply_pair_strided(q, k, tabs)
    torch.cuda.synchronize()
    assert r.rope3d_last_launch()["kernel"] == 1
    shape6 = (B, T, H, W, heads, hd)
    assert_bit_exact(_host(qo, dtype), oracle_rotate(q_np, shape6, split, dtype), f"Q {dtype}")
    assert_bit_exact(_host(ko, dtype), oracle_rotate(k_np, shape6, split, dtype), f"K {dtype}")
    assert torch.equal(bitview(v), bitview(v_before))  # V is untouched
    if not inplace:  # the inputs are untouched
        assert np.array_equal(bits(_host(q, dtype)), bits(q_np))
    tabs.close()


def test_strided_pair_kernel_and_crop():
    """head_dim 20 with a (4, 8, 8) split cannot take 16-byte vectors; the
    views are a crop of a larger grid, written into a crop of another buffer."""
    B, T, H, W, heads, hd, split = 2, 3, 5, 4, 3, 20, (4, 8, 8)
    big_shape = (B, T + 1, H + 3, W + 2, heads, hd)
    n = int(np.prod(big_shape))
    big_q = to_torch(draw(n, 63, 0, "bf16"), "bf16").reshape(big_shape).to(DEV)
    big_k = to_torch(draw(n, 63, 1, "bf16"), "bf16").reshape(big_shape).to(DEV)
    q = big_q[:, 1:, 2:2 + H, 1:1 + W]
    k = big_k[:, :T, 3:3 + H, 2:]
    out_buf = torch.full((B, T, H + 1, 2 * W, heads, hd), 9.0, dtype=torch.bfloat16, device=DEV)
    qo = out_buf[:, :, :H, :W]
    ko = out_buf[:, :, 1:, W:]   # overlapping rows but disjoint columns: no shared element
    tabs = r.rope3d_build_tables(T, H, W, split)
    r.rope3d_apply_pair_strided(q, k, tabs, qo, ko)
    torch.cuda.synchronize()
    assert r.rope3d_last_launch()["kernel"] == 2
    shape6 = (B, T, H, W, heads, hd)
    assert_bit_exact(_host(qo, "bf16"), oracle_rotate(_host(q, "bf16"), shape6, split, "bf16"), "Q")
    assert_bit_exact(_host(ko, "bf16"), oracle_rotate(_host(k, "bf16"), shape6, split, "bf16"), "K")
    # the rest of the output buffer is untouched
    mask = torch.ones(out_buf.shape[:4], dtype=torch.bool, device=DEV)
    mask[:, :, :H, :W] = False
    mask[:, :, 1:, W:] = False
    assert torch.all(out_buf[mask] == 9.0)
    tabs.close()


def test_strided_gate_refuses_on_planted_mismatch():
    w = synthetic.WORKLOADS["tiny"]
    buf, q, k, v = _qkv(w.B, w.N, w.heads, w.head_dim, "bf16", 64, False)
    tabs = r.rope3d_build_tables(w.T, w.H, w.W, w.split)
    r.rope3d_testing_corrupt_gate(1)
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_apply_pair_strided(q, k, tabs)
    assert e.value.name == "ERR_PARITY"
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_apply_pair_strided(q, k, tabs)
    assert e.value.name == "ERR_PARITY"
    # another layout of the same shapes is a different configuration
    qc, kc = q.contiguous(), k.contiguous()
    r.rope3d_apply_pair_strided(qc, kc, tabs)
    tabs.close()


def test_strided_rejects_overlap_on_device():
    w = synthetic.WORKLOADS["tiny"]
    buf, q, k, v = _qkv(w.B, w.N, w.heads, w.head_dim, "bf16", 65, False)
    tabs = r.rope3d_build_tables(w.T, w.H, w.W, w.split)
    before = buf.clone()
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_apply_pair_strided(q, k, tabs, k, q)  # swapped in place
    assert e.value.name == "ERR_ALIAS"
    torch.cuda.synchronize()
    assert torch.equal(buf.view(torch.int16), before.view(torch.int16))
    tabs.close()
