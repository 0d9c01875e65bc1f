"""The C ABI used from plain C: tests/abi_consumer.c is compiled against
include/rope3d.h and the built library, run on seeded inputs, and its outputs
are compared bit for bit with the CPU oracle."""
from __future__ import annotations

import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import synthetic

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU hosts
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import rope_rope3d_apply_gb300 as r  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    nvcc = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc))) if nvcc else "/usr/local/cuda"


@pytest.fixture(scope="module")
def consumer(tmp_path_factory):
    r.load_library()
    out = tmp_path_factory.mktemp("c_abi") / "abi_consumer"
    lib_dir = os.path.dirname(r.LIB_PATH)
    cuda = _cuda_home()
    cmd = ["gcc", "-std=c99", "-O2", os.path.join(ROOT, "tests", "abi_consumer.c"),
           f"-I{os.path.join(ROOT, 'include')}", f"-I{cuda}/include", "-o", str(out),
           f"-L{lib_dir}", "-lrope3d", f"-Wl,-rpath,{lib_dir}",
           f"-L{cuda}/lib64", f"-L{cuda}/lib", "-lcudart", f"-Wl,-rpath,{cuda}/lib64"]
    subprocess.run(cmd, check=True)
    return str(out)


@pytest.mark.parametrize("name", ["tiny", "stage0", "stage0_f32"])
def test_c_consumer_matches_oracle(consumer, tmp_path, name):
    w = synthetic.WORKLOADS[name]
    q, k = synthetic.qk(w)
    paths = [str(tmp_path / f) for f in ("q.bin", "k.bin", "qo.bin", "ko.bin")]
    q.tofile(paths[0])
    k.tofile(paths[1])
    dtype = r.F32 if w.dtype == "f32" else r.BF16
    args = [consumer, *paths, *(str(v) for v in w.shape6), *(str(v) for v in w.split), str(dtype)]
    res = subprocess.run(args, capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == "ok"
    tabs = oracle.tables(w.T, w.H, w.W, w.split, w.base)
    npdt = np.float32 if w.dtype == "f32" else np.uint16
    got_q = np.fromfile(paths[2], dtype=npdt)
    got_k = np.fromfile(paths[3], dtype=npdt)
    want_q = oracle.rope3d(q, w.shape6, w.split, tabs)
    want_k = oracle.rope3d(k, w.shape6, w.split, tabs)
    view = (lambda a: a.view(np.uint32)) if w.dtype == "f32" else (lambda a: a)
    assert np.array_equal(view(got_q), view(want_q))
    assert np.array_equal(view(got_k), view(want_k))
