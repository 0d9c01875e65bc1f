"""GPU parity of rope3d_patchify / rope3d_unpatchify against the oracle's
definition (sglang PR #34471 review, "关键源码片段", _patchify): a
permutation, so the bar is bit-exactness (compared as raw bytes)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU hosts
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import rope_rope3d_apply_gb300 as r  # noqa: E402

DEV = torch.device("cuda:0")
BITS = {1: (np.uint8, torch.uint8), 2: (np.int16, torch.int16), 4: (np.int32, torch.int32),
        8: (np.int64, torch.int64)}


def _random(shape, es, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    npt, _ = BITS[es]
    return g.integers(np.iinfo(npt).min, np.iinfo(npt).max, size=shape, dtype=npt, endpoint=True)


CASES = [
    # (B, C, F, H, W), p, elem_bytes, expected kernel (1 vector, 2 element)
    ((1, 3, 2, 32, 64), 4, 2, 1),
    ((2, 4, 3, 16, 128), 2, 2, 1),
    ((1, 2, 2, 64, 512), 8, 2, 1),
    ((1, 3, 4, 8, 8), 1, 4, 1),
    ((1, 5, 2, 12, 24), 4, 2, 2),      # W/p = 6 is not a whole number of 8-element vectors
    ((1, 2, 3, 9, 27), 3, 2, 2),       # p = 3
    ((2, 3, 2, 16, 64), 4, 1, 1),      # bytes
    ((1, 2, 2, 16, 32), 2, 8, 1),      # 8-byte elements
    ((1, 1, 1, 4, 4), 4, 4, 2),        # one output pixel per channel
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-p{c[1]}-e{c[2]}" for c in CASES])
def test_patchify_round_trip_bit_exact(case):
    shape, p, es, kernel = case
    x_np = _random(shape, es, 80)
    _, tdt = BITS[es]
    x = torch.from_numpy(x_np).to(DEV)
    y = r.rope3d_patchify(x, p)
    torch.cuda.synchronize()
    assert r.rope3d_patchify_last_kernel() == kernel
    want = oracle.patchify(x_np, p)
    assert np.array_equal(y.cpu().numpy(), want)
    back = r.rope3d_unpatchify(y, p)
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy(), x_np)
    # unpatchify of an independent tensor against the oracle's inverse
    y2_np = _random(want.shape, es, 81)
    x2 = r.rope3d_unpatchify(torch.from_numpy(y2_np).to(DEV), p)
    assert np.array_equal(x2.cpu().numpy(), oracle.unpatchify(y2_np, p))


def test_patchify_unaligned_and_guard_bytes():
    shape, p = (1, 3, 2, 16, 64), 4
    n = int(np.prod(shape))
    x_np = _random(shape, 2, 82)
    base = torch.zeros(n + 1, dtype=torch.int16, device=DEV)
    x = base[1:].view(shape)                  # 2-byte aligned, not 16-byte aligned
    x.copy_(torch.from_numpy(x_np).to(DEV))
    guard = 1024
    out = torch.full((n + 2 * guard,), 77, dtype=torch.int16, device=DEV)
    y = out[guard:guard + n].view(1, 3 * 16, 2, 4, 16)
    r.rope3d_patchify(x, p, y)
    torch.cuda.synchronize()
    assert r.rope3d_patchify_last_kernel() == 2
    assert np.array_equal(y.cpu().numpy(), oracle.patchify(x_np, p))
    assert torch.all(out[:guard] == 77) and torch.all(out[-guard:] == 77)


def test_patchify_rejections():
    x = torch.zeros((1, 2, 2, 6, 8), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_patchify(x, 4)                                # H = 6 is not a multiple of 4
    assert e.value.name == "ERR_SHAPE"
    big = torch.zeros(2 * 2 * 2 * 8 * 8 * 2, dtype=torch.bfloat16, device=DEV)
    x2 = big[: 2 * 2 * 8 * 8].view(1, 2, 2, 8, 8)
    y2 = big[64: 64 + 2 * 2 * 8 * 8].view(1, 8, 2, 4, 4)       # overlaps x2
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_patchify(x2, 2, y2)
    assert e.value.name == "ERR_ALIAS"
    host = torch.zeros((1, 2, 2, 8, 8), dtype=torch.bfloat16)
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_patchify(host, 2, torch.empty((1, 8, 2, 4, 4), dtype=torch.bfloat16, device=DEV))
    assert e.value.name == "ERR_DEVICE"
