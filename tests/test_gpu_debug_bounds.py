"""The bounds-checking debug build: every kernel checks each index it computes
(table entries, strided and permuted offsets, token and key positions, shared-
memory slots) before the access it guards and counts failures instead of
faulting. This test builds that variant and runs the GPU suites of every entry
point against it in a child process; conftest.py then asserts after each test
that no check failed, and the suites' own comparisons hold the debug build to
the same results as the normal one."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU hosts
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["test_gpu_debug_checks_fire.py", "test_gpu_parity.py", "test_gpu_strided.py",
          "test_gpu_patchify.py", "test_gpu_neox.py", "test_gpu_na3d.py", "test_gpu_fuzz.py"]


def test_suites_pass_under_the_bounds_checking_build():
    from rope_rope3d_apply_gb300 import build

    lib = build.build(debug_bounds=True)
    env = dict(os.environ, ROPE3D_LIB=lib)
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "gpu",
           *[os.path.join(ROOT, "tests", s) for s in SUITES]]
    out = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert out.returncode == 0, out.stdout[-4000:] + out.stderr[-2000:]
    summary = out.stdout.strip().splitlines()[-1]
    # every test ran, the one that makes the checks fire included
    assert " passed" in summary and "skipped" not in summary, summary


def test_debug_build_reports_itself():
    from rope_rope3d_apply_gb300 import build

    lib = build.build(debug_bounds=True)
    code = ("import rope_rope3d_apply_gb300 as r; import torch; torch.cuda.init(); "
            "print(r.rope3d_debug_bounds())")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=dict(os.environ, ROPE3D_LIB=lib),
                         capture_output=True, text=True, timeout=300, check=True)
    assert out.stdout.strip().splitlines()[-1] == "(True, 0)"
