"""The bench's CPU legs, run here without a GPU: the reference arm (the oracle on
a bounded sample per timed step) prints one JSON line whose ms_per_step is the
wall time a step actually took and whose sample fields keep the measured time,
the whole-step estimate and the scale factor apart; the CPU sample reports the
same three figures for the cpu_baseline legs."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    s = d["sample"]
    # ms_per_step is what a timed step took, not the whole-step extrapolation
    assert abs(d["ms_per_step"] - 1e3 * s["measured_seconds_per_step"]) < 1e-6
    assert s["full_step_seconds_est"] > s["measured_seconds_per_step"]
    assert abs(s["scale_to_full_step"] * s["measured_seconds_per_step"]
               - s["full_step_seconds_est"]) < 1e-6 * s["full_step_seconds_est"]
    assert abs(d["value"] - 65536 / s["full_step_seconds_est"]) < 1e-6 * d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_cpu_model_and_legs_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
