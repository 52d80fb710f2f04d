"""bench.py's output line, checked as a consumer reads it: one JSON object on stdout per run,
with the keys, units and internal consistency the measurement contract asks for.  The oracle
arm (--impl reference) runs on the host cores, so its check needs no GPU; the library arm's
needs one."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
M, K, N = 8192, 5120, 20480


def _run_bench(*args, timeout=600):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def _common(d):
    sys.path.insert(0, ROOT)
    import bench
    assert d["metric"] == bench.METRIC
    assert d["config"]["workload"] == bench.WORKLOAD
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] > 0


def test_reference_arm_line():
    d = _run_bench("--impl", "reference", "--steps", "3", "--warmup", "3", timeout=300)
    _common(d)
    assert d["impl"] == "reference"
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["sample"]
    assert cpu["value"] == d["value"] and cpu["unit"] == d["unit"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


@pytest.mark.gpu
def test_library_arm_line():
    d = _run_bench("--steps", "3", "--warmup", "3", "--no-cpu-baseline")
    _common(d)
    assert "impl" not in d or d["impl"] == "ours"
    assert d["device_status"] == 0
    # value is three 2MNK GEMMs per step over the device-timed step
    assert d["value"] == pytest.approx(3 * 2.0 * M * N * K / (d["ms_per_step"] * 1e-3) / 1e12, rel=2e-3)
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] > 0
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-3)
    assert 0 < r["frac"] < 1.2
    e = d["e2e"]
    assert e["unit"] == "TFLOP/s" and 0 < e["value"] <= d["value"]
    assert e["h2d_bytes_per_step"] == 2 * (M * K + N * K + M * N)        # X, W, dY in bf16
    assert e["d2h_bytes_per_step"] == 2 * (M * N + M * K + N * K)        # Y, dX, dW in bf16
    assert d["gpu_launches"] > 0
    c = d["clocks"]
    assert c["sm_mhz"] > 0 and c["sm_max_mhz"] >= c["sm_mhz"] and isinstance(c["reasons"], list)
    q = d["quantize_roofline"]
    assert q["bound"] == "hbm" and q["frac"] == pytest.approx(q["achieved"] / q["peak"], rel=1e-3)
