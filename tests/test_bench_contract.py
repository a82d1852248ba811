"""The bench's JSON line carries what the measurement contract asks for: the reference arm
(the fp64 oracle on the host cores, no GPU) here, the CUDA arm on a GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

COMMON = {"metric": str, "value": (int, float), "unit": str, "n_gpus": int, "steps": int,
          "warmup": int, "ms_per_step": (int, float), "higher_is_better": bool, "scaling": str,
          "dtype": str, "data": str, "config": dict}


def run_bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-3000:]
    return json.loads(lines[0])


def check_common(d, steps):
    for key, typ in COMMON.items():
        assert isinstance(d[key], typ), key
    assert "vs_baseline" in d and d["steps"] == steps and d["warmup"] >= 3
    assert d["config"]["workload"] and d["data"] == "synthetic" and d["value"] > 0


def test_reference_arm_line():
    d = run_bench("--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-step-s", "0.2")
    check_common(d, 1)
    assert d["impl"] == "reference" and d["dtype"] == "f64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
@pytest.mark.parametrize("workload,launches", [("layer_16h_4k", 2), ("tiny_f32", 2)])
def test_cuda_arm_line(workload, launches):
    d = run_bench("--workload", workload, "--steps", "5", "--warmup", "3",
                  "--cpu-baseline-s", "0.3", "--no-decode")
    check_common(d, 5)
    assert d["n_gpus"] == 1 and d["config"]["workload"] == workload
    r = d["roofline"]
    assert r["bound"] in ("hbm", "tensor", "alu") and r["unit"] in ("GB/s", "TFLOP/s")
    assert r["peak"] > 0 and r["achieved"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert 0 < r["frac_of_nominal"] <= r["frac"]  # the nominal 7.9 TB/s is above the measured peak
    assert r["traffic"] is None or r["traffic"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == launches * 5
    c = d["clocks"]
    assert "sm_mhz" in c and "sm_max_mhz" in c and isinstance(c["reasons"], list)
