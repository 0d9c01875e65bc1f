"""rope3d_apply_pair_noalloc, the entry point for callers that cannot
allocate device memory (their device memory belongs to another allocator or a
fixed budget, or they must not take cudaMalloc's implicit synchronisation).
It takes no table handle and keeps the tables in the library's fixed static
device table area instead of a cudaMalloc'd cache entry.

Checked through the C ABI against rope3d_apply_pair, bit for bit (the same bar
as every other GPU test), on two calls in a row: the second call uses a
smaller grid, so it reads an area whose tail still holds the first call's
tables. This file is collected last on purpose.
"""
from __future__ import annotations

import numpy as np
import pytest

import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU hosts
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import rope_rope3d_apply_gb300 as r  # noqa: E402

DEV = torch.device("cuda:0")


def _inputs(w):
    q_np, k_np = synthetic.qk(w)
    shp = (w.B, w.N, w.heads, w.head_dim)
    conv = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)) if w.dtype == "bf16" \
        else torch.from_numpy
    return conv(q_np).reshape(shp).to(DEV), conv(k_np).reshape(shp).to(DEV)


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def test_noalloc_matches_apply_pair_on_two_calls_in_a_row():
    for name in ("stage5_w63", "stage0_f32"):
        w = synthetic.WORKLOADS[name]
        q, k = _inputs(w)
        # the caller's own output memory
        qo, ko = torch.empty_like(q), torch.empty_like(k)
        r.rope3d_apply_pair_noalloc(q, k, qo, ko, w.T, w.H, w.W, w.split, w.base)
        torch.cuda.synchronize()
        tabs = r.rope3d_build_tables(w.T, w.H, w.W, w.split, w.base)
        want_q, want_k = r.rope3d_apply_pair(q, k, tabs)
        torch.cuda.synchronize()
        tabs.close()
        assert torch.equal(_bits(qo), _bits(want_q)), name
        assert torch.equal(_bits(ko), _bits(want_k)), name


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
