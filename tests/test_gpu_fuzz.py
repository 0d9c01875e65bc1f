"""Seeded random shapes through every GPU entry point, each compared with the
oracle bit for bit: grids, head counts, splits, dtypes, bases, pointer
offsets, padded (strided) views, in-place calls, patch sizes, NeoX head
layouts and neighbourhood-attention windows drawn from a fixed generator, so
that every run checks the same cases (the attention against the float64
oracle within its derived bound, everything else bit for bit)."""
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
TDT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
ES = {"bf16": 2, "f16": 2, "f32": 4}


def draw(n, seed, which, dtype):
    return synthetic.normal(n, 1.0, seed, which, dtype)


def np_to_torch(a, dtype):
    if dtype == "f32":
        return torch.from_numpy(a.copy())
    return torch.from_numpy(a.view(np.int16).copy()).view(TDT[dtype])


def to_np(t):
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return t.numpy().reshape(-1)


def bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


def random_case(g):
    B = int(g.integers(1, 4))
    T, H, W = (int(v) for v in g.integers(1, 8, 3))
    heads = int(g.integers(1, 5))
    split = tuple(int(v) * 2 for v in g.integers(1, 13, 3))
    dtype = str(g.choice(["bf16", "f16", "f32"]))
    base = float(g.choice([10000.0, 500.0, 1e6]))
    return B, T, H, W, heads, sum(split), split, dtype, base


@pytest.mark.parametrize("seed", range(40))
def test_fuzz_apply_pair(seed):
    g = np.random.Generator(np.random.PCG64(1000 + seed))
    B, T, H, W, heads, hd, split, dtype, base = random_case(g)
    shape6 = (B, T, H, W, heads, hd)
    n = int(np.prod(shape6))
    q_np, k_np = draw(n, 2000 + seed, 0, dtype), draw(n, 2000 + seed, 1, dtype)
    off = int(g.choice([0, 4 // ES[dtype] if dtype != "f32" else 1, 8 // ES[dtype]]))

    def placed(a):
        big = torch.empty(n + off + 8, dtype=TDT[dtype], device=DEV)
        v = big[off:off + n].view(shape6)
        v.copy_(np_to_torch(a, dtype).view(shape6).to(DEV))
        return v

    q, k = placed(q_np), placed(k_np)
    qo = torch.empty(n + off, dtype=TDT[dtype], device=DEV)[off:].view(shape6)
    ko = torch.empty(n + off, dtype=TDT[dtype], device=DEV)[off:].view(shape6)
    tabs = r.rope3d_build_tables(T, H, W, split, base)
    r.rope3d_apply_pair(q, k, tabs, qo, ko)
    torch.cuda.synchronize()
    otabs = oracle.tables(T, H, W, split, base)
    f16 = dtype == "f16"
    assert np.array_equal(bits(to_np(qo)), bits(oracle.rope3d(q_np, shape6, split, otabs, f16=f16)))
    assert np.array_equal(bits(to_np(ko)), bits(oracle.rope3d(k_np, shape6, split, otabs, f16=f16)))
    tabs.close()


@pytest.mark.parametrize("seed", range(24))
def test_fuzz_strided_views(seed):
    g = np.random.Generator(np.random.PCG64(3000 + seed))
    B, T, H, W, heads, hd, split, dtype, base = random_case(g)
    shape6 = (B, T, H, W, heads, hd)
    # views into buffers padded along every dimension, channels contiguous
    pad = tuple(int(v) for v in g.integers(0, 3, 5)) + (int(g.integers(0, 3)) * 2,)
    big_shape = tuple(s + p for s, p in zip(shape6, pad))

    def view_of(seed_which):
        nb = int(np.prod(big_shape))
        buf = np_to_torch(draw(nb, 4000 + seed, seed_which, dtype), dtype).view(big_shape).to(DEV)
        lo = [int(g.integers(0, p + 1)) for p in pad]
        lo[-1] -= lo[-1] % 2                      # pairs stay 4-byte aligned
        sl = tuple(slice(a, a + s) for a, s in zip(lo, shape6))
        return buf, buf[sl]

    qbuf, q = view_of(0)
    kbuf, k = view_of(1)
    q_np, k_np = to_np(q), to_np(k)
    inplace = bool(g.integers(0, 2))
    tabs = r.rope3d_build_tables(T, H, W, split, base)
    if inplace:
        qo, ko = r.rope3d_apply_pair_strided(q, k, tabs, q, k)
    else:
        qo, ko = r.rope3d_apply_pair_strided(q, k, tabs)
    torch.cuda.synchronize()
    otabs = oracle.tables(T, H, W, split, base)
    f16 = dtype == "f16"
    assert np.array_equal(bits(to_np(qo)), bits(oracle.rope3d(q_np, shape6, split, otabs, f16=f16)))
    assert np.array_equal(bits(to_np(ko)), bits(oracle.rope3d(k_np, shape6, split, otabs, f16=f16)))
    tabs.close()


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_patchify(seed):
    g = np.random.Generator(np.random.PCG64(5000 + seed))
    p = int(g.choice([1, 2, 3, 4, 8]))
    es = int(g.choice([1, 2, 4, 8]))
    B, C, F = (int(v) for v in g.integers(1, 4, 3))
    H = p * int(g.integers(1, 9))
    W = p * int(g.choice([1, 3, 8, 16, 32]))
    dt = {1: np.uint8, 2: np.int16, 4: np.int32, 8: np.int64}[es]
    x_np = g.integers(np.iinfo(dt).min, np.iinfo(dt).max, (B, C, F, H, W), dtype=dt, endpoint=True)
    x = torch.from_numpy(x_np).to(DEV)
    y = r.rope3d_patchify(x, p)
    back = r.rope3d_unpatchify(y, p)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), oracle.patchify(x_np, p))
    assert np.array_equal(back.cpu().numpy(), x_np)


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_neox(seed):
    g = np.random.Generator(np.random.PCG64(6000 + seed))
    tokens = int(g.integers(1, 200))
    qh, kh = (int(v) for v in g.integers(1, 6, 2))
    hd = int(g.choice([4, 8, 12, 16, 32, 64, 96, 128, 256]))
    dtype = str(g.choice(["bf16", "f16", "f32"]))
    max_pos = int(g.integers(1, 3000))
    base = float(g.choice([10000.0, 1e6]))
    positions = g.integers(0, max_pos, tokens, dtype=np.int64)
    cache = oracle.neox_cache(max_pos, hd, base)
    q_np = draw(tokens * qh * hd, 7000 + seed, 0, dtype)
    k_np = draw(tokens * kh * hd, 7000 + seed, 1, dtype)
    q = np_to_torch(q_np, dtype).view(tokens, qh, hd).to(DEV)
    k = np_to_torch(k_np, dtype).view(tokens, kh, hd).to(DEV)
    inplace = bool(g.integers(0, 2))
    args = (q, k) if inplace else (None, None)
    qo, ko = r.rope3d_apply_neox(q, k, torch.from_numpy(positions).to(DEV),
                                 torch.from_numpy(cache).to(DEV), *args)
    torch.cuda.synchronize()
    assert np.array_equal(bits(to_np(qo)), bits(oracle.rope_neox(q_np, tokens, qh, hd, positions, cache, dtype).reshape(-1)))
    assert np.array_equal(bits(to_np(ko)), bits(oracle.rope_neox(k_np, tokens, kh, hd, positions, cache, dtype).reshape(-1)))


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_na3d(seed):
    """Neighbourhood attention on random grids, heads, batches, splits and
    odd windows, with and without the rotation: within the derived bound of
    the float64 oracle, and both fused forms equal to the unfused pair."""
    g = np.random.Generator(np.random.PCG64(8000 + seed))
    B = int(g.integers(1, 3))
    T, H, W = int(g.integers(1, 6)), int(g.integers(1, 21)), int(g.integers(1, 21))
    heads = int(g.integers(1, 4))
    dT = 8 * int(g.integers(1, 7))
    dH = 8 * int(g.integers(1, 15 - dT // 8))
    split = (dT, dH, 128 - dT - dH)
    kernel = tuple(int(2 * g.integers(0, (L + 1) // 2) + 1) for L in (T, H, W))
    rope = bool(g.integers(0, 2))
    shape6 = (B, T, H, W, heads, 128)
    n = int(np.prod(shape6))
    q_np, k_np, v_np = (draw(n, 9000 + seed, i, "bf16") for i in range(3))
    shp = (B, T * H * W, heads, 128)
    q, k, v = (np_to_torch(a, "bf16").reshape(shp).to(DEV) for a in (q_np, k_np, v_np))
    tabs = r.rope3d_build_tables(T, H, W, split)
    out = r.rope3d_na3d(q, k, v, tabs, kernel, apply_rope=rope)
    if rope:
        qr, kr = r.rope3d_apply_pair(q, k, tabs)
        unfused = r.rope3d_na3d(qr, kr, v, tabs, kernel, apply_rope=False)
        once, k_rot = r.rope3d_na3d_rotate_once(q, k, v, tabs, kernel)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), unfused.view(torch.int16))
        assert torch.equal(once.view(torch.int16), unfused.view(torch.int16))
        assert torch.equal(k_rot.view(torch.int16), kr.view(torch.int16))
    torch.cuda.synchronize()
    to64 = lambda b: (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)  # noqa: E731
    got = to64(to_np(out)).reshape(shape6)
    otabs = oracle.tables(T, H, W, split)
    ref = oracle.rope_na3d(q_np, k_np, v_np, shape6, split, otabs, kernel, rope=rope)
    qr_np = oracle.rope3d(q_np, shape6, split, otabs) if rope else q_np
    kr_np = oracle.rope3d(k_np, shape6, split, otabs) if rope else k_np
    absv = oracle.na3d(to64(qr_np), to64(kr_np), np.abs(to64(v_np)), shape6, kernel)
    bound = 2.0 ** -7 * absv + 2.0 ** -8 * np.abs(ref) + 1e-6
    assert np.all(np.abs(got - ref) <= bound), (seed, shape6, split, kernel, rope)
    tabs.close()
