"""Under the bounds-checking debug build only (ROPE3D_LIB, see
test_gpu_debug_bounds.py): the checks do fire. A test hook makes the rotation
kernels see the tables four entries shorter than they are; the memory stays
valid, so nothing can fault, and every lookup past the shortened end must be
counted and skipped."""
from __future__ import annotations

import numpy as np
import pytest

import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU hosts
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import rope_rope3d_apply_gb300 as r  # noqa: E402


def test_table_checks_fire_and_count():
    built, _ = r.rope3d_debug_bounds(reset=True)
    if not built:
        pytest.skip("runs under the bounds-checking build only")
    w = synthetic.WORKLOADS["stage0"]
    shp = (w.B, w.N, w.heads, w.head_dim)
    q, k = (torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).reshape(shp).cuda()
            for a in synthetic.qk(w))
    tabs = r.rope3d_build_tables(w.T, w.H, w.W, w.split, w.base)
    mode = r.rope3d_gate_get_mode()
    r.rope3d_gate_set_mode(r.GATE_OFF)
    try:
        r.rope3d_testing_debug_shrink_tables(4)
        r.rope3d_apply_pair(q, k, tabs)
        torch.cuda.synchronize()
        _, errors = r.rope3d_debug_bounds(reset=True)
        assert errors > 0
        r.rope3d_testing_debug_shrink_tables(0)
        r.rope3d_apply_pair(q, k, tabs)
        torch.cuda.synchronize()
        assert r.rope3d_debug_bounds(reset=True) == (True, 0)
    finally:
        r.rope3d_testing_debug_shrink_tables(0)
        r.rope3d_gate_set_mode(mode)
        tabs.close()
