"""The JSON line of bench.py's GPU arm carries every field of its contract:
the base keys, the roofline object, the CPU baseline, the end-to-end figure
through host buffers, the clock record and the launch count (run on the
small stage-0 workload so that it takes seconds)."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU hosts
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gpu_arm_line_has_every_contract_field():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5",
                          "--warmup", "3", "--workload", "stage0", "--cpu-seconds", "1"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600, check=True)
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert key in d, key
    assert d["unit"] == "GB/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] >= 3
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert "workload" in d["config"]
    rf = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in rf, key
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    sv, link = e2e["step_values"], e2e["host_link_gbs"]
    assert 0 < sv["min"] <= sv["median"] <= sv["max"]
    assert 0 < link["min"] <= link["median"] <= link["max"] and link["rounds"] >= 3
    # the whole-run value lies within its steps' spread
    assert sv["min"] * (1 - 1e-9) <= e2e["value"] <= sv["max"] * (1 + 1e-9)
    assert e2e["frac_of_host_link"] > 0
    for key in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert key in d["clocks"], key
    assert d["gpu_launches"] >= d["steps"]
    assert d["gate_verdict"] == "verified"
