"""GPU parity of rope3d_apply_neox (the Gemma3 text encoder's NeoX-style
RoPE, sglang PR #24660 review, "关键源码片段", gemma_3.py) against the oracle:
bit-exact in every dtype, with grouped-query head counts, repeated and
out-of-range positions, and rotation in place."""
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


def draw(n, seed, which, dtype):
    return synthetic.normal(n, 1.0, seed, which, dtype)


def to_dev(a, shape, dtype):
    t = torch.from_numpy(a.copy()) if dtype == "f32" else torch.from_numpy(a.view(np.int16).copy()).view(TDT[dtype])
    return t.reshape(shape).to(DEV)


def to_np(t):
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return t.numpy().reshape(-1)


def bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


CASES = [
    # tokens, q_heads, k_heads, head_dim, max_position, dtype, kernel
    (257, 8, 4, 256, 8192, "bf16", 1),
    (300, 4, 1, 128, 4096, "f16", 1),
    (129, 2, 2, 64, 1000, "f32", 1),
    (77, 3, 5, 12, 500, "bf16", 2),       # half of 6 is not a whole 8-element vector
    (64, 2, 1, 20, 100, "f32", 2),
    (32768, 8, 4, 256, 131072, "bf16", 1),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}x{c[1]}/{c[2]}x{c[3]}-{c[5]}" for c in CASES])
def test_neox_bit_exact(case):
    tokens, qh, kh, hd, max_pos, dtype, kernel = case
    g = np.random.Generator(np.random.PCG64(100 + tokens))
    positions = g.integers(0, max_pos, tokens, dtype=np.int64)
    positions[: min(8, tokens)] = positions[0]          # repeated positions
    cache = oracle.neox_cache(max_pos, hd)
    q_np = draw(tokens * qh * hd, 101, 0, dtype)
    k_np = draw(tokens * kh * hd, 101, 1, dtype)
    q = to_dev(q_np, (tokens, qh, hd), dtype)
    k = to_dev(k_np, (tokens, kh, hd), dtype)
    pos = torch.from_numpy(positions).to(DEV)
    cache_d = torch.from_numpy(r.rope3d_neox_cache_host(max_pos, hd)).to(DEV)
    qo, ko = r.rope3d_apply_neox(q, k, pos, cache_d)
    torch.cuda.synchronize()
    assert r.rope3d_neox_last_kernel() == kernel
    want_q = oracle.rope_neox(q_np, tokens, qh, hd, positions, cache, dtype)
    want_k = oracle.rope_neox(k_np, tokens, kh, hd, positions, cache, dtype)
    assert np.array_equal(bits(to_np(qo)), bits(want_q.reshape(-1)))
    assert np.array_equal(bits(to_np(ko)), bits(want_k.reshape(-1)))


def test_neox_in_place_and_invalid_positions():
    tokens, qh, kh, hd, max_pos = 40, 4, 2, 64, 128
    g = np.random.Generator(np.random.PCG64(102))
    positions = g.integers(0, max_pos, tokens, dtype=np.int64)
    bad = np.array([3, 17, 39])
    positions[bad] = [-1, max_pos, 1 << 40]
    q_np = draw(tokens * qh * hd, 103, 0, "bf16")
    k_np = draw(tokens * kh * hd, 103, 1, "bf16")
    q = to_dev(q_np, (tokens, qh, hd), "bf16")
    k = to_dev(k_np, (tokens, kh, hd), "bf16")
    cache = oracle.neox_cache(max_pos, hd)
    cache_d = torch.from_numpy(cache).to(DEV)
    counter = torch.zeros(1, dtype=torch.int32, device=DEV)
    r.rope3d_apply_neox(q, k, torch.from_numpy(positions).to(DEV), cache_d, q, k, counter)
    torch.cuda.synchronize()
    per_head = (hd // 2) // 8
    assert int(counter.item()) == len(bad) * (qh + kh) * per_head
    good = np.ones(tokens, bool)
    good[bad] = False
    safe = positions.copy()
    safe[bad] = 0
    want_q = oracle.rope_neox(q_np, tokens, qh, hd, safe, cache, "bf16").reshape(tokens, qh, hd)
    want_k = oracle.rope_neox(k_np, tokens, kh, hd, safe, cache, "bf16").reshape(tokens, kh, hd)
    got_q = to_np(q).reshape(tokens, qh, hd)
    got_k = to_np(k).reshape(tokens, kh, hd)
    assert np.array_equal(got_q[good], want_q[good])
    assert np.array_equal(got_k[good], want_k[good])
    # tokens with an invalid position were left as they were (in place: the input)
    assert np.array_equal(got_q[~good], q_np.reshape(tokens, qh, hd)[~good])
    assert np.array_equal(got_k[~good], k_np.reshape(tokens, kh, hd)[~good])


def test_neox_rejects_on_device():
    buf = torch.zeros(200, dtype=torch.bfloat16, device=DEV)
    q = buf[0:64].view(4, 2, 8)
    k = buf[64:96].view(4, 1, 8)
    q_out = buf[60:124].view(4, 2, 8)            # overlaps both inputs
    pos = torch.zeros(4, dtype=torch.int64, device=DEV)
    cache = torch.zeros((16, 8), dtype=torch.float32, device=DEV)
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_apply_neox(q, k, pos, cache, q_out, torch.empty_like(k))
    assert e.value.name == "ERR_ALIAS"
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_apply_neox(q, k, pos.cpu(), cache)
    assert e.value.name == "ERR_DEVICE"


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("hd,kernel", [(64, 1), (12, 2)])
def test_neox_special_values(dtype, hd, kernel):
    """Signed zeros, subnormal products and sums, infinities and NaNs: the
    packed 16-bit arithmetic of the vector kernel and the float arithmetic of
    the pair kernel must both match the oracle (NaN against any NaN)."""
    tokens, qh, kh, max_pos = 64, 2, 1, 300
    g = np.random.Generator(np.random.PCG64(104))
    n = tokens * qh * hd
    x = g.standard_normal(n).astype(np.float32)
    pool = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1.0, -2.5, 6e-5, 1e-7, 3e4, 60000.0],
                    np.float32)
    pick = g.integers(0, n, n // 3)
    x[pick] = pool[g.integers(0, pool.size, pick.size)]
    x[g.integers(0, n, n // 6)] *= np.float32(2.0 ** -14 if dtype == "f16" else 2.0 ** -125)
    q_np = synthetic.f32_to_bf16_bits(x) if dtype == "bf16" else x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        q_np = np.where(np.isnan(x), np.uint16(0x7FC0), q_np).astype(np.uint16)
    k_np = q_np[: tokens * kh * hd][::-1].copy()
    positions = g.integers(0, max_pos, tokens, dtype=np.int64)
    cache = oracle.neox_cache(max_pos, hd)
    qo, ko = r.rope3d_apply_neox(to_dev(q_np, (tokens, qh, hd), dtype), to_dev(k_np, (tokens, kh, hd), dtype),
                                 torch.from_numpy(positions).to(DEV), torch.from_numpy(cache).to(DEV))
    torch.cuda.synchronize()
    assert r.rope3d_neox_last_kernel() == kernel
    nanmax = 0x7F80 if dtype == "bf16" else 0x7C00
    for got, src, heads in ((to_np(qo), q_np, qh), (to_np(ko), k_np, kh)):
        want = oracle.rope_neox(src, tokens, heads, hd, positions, cache, dtype).reshape(-1)
        both_nan = ((got & 0x7FFF) > nanmax) & ((want & 0x7FFF) > nanmax)
        bad = (got != want) & ~both_nan
        assert not bad.any(), (int(bad.sum()), np.flatnonzero(bad)[:5])
