"""The JSON line bench.py prints: keys and types that the measurement
contract fixes, for the reference arm (the oracle on the host cores, no GPU)
and for this library's arm (GPU)."""
import json
import math
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, capture_output=True,
                         text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def _common(d, steps, warmup):
    assert d["metric"] and d["unit"] == "TFLOP/s"
    assert isinstance(d["value"], float) and d["value"] > 0 and math.isfinite(d["value"])
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["scaling"] in ("weak", "strong")
    assert d["vs_baseline"] is None
    assert isinstance(d["dtype"], str) and d["data"] == "synthetic"
    assert d["config"]["workload"] == "single_128x128x256"
    e = d["e2e"]
    assert e["unit"] == d["unit"] and e["value"] > 0
    assert isinstance(e["h2d_bytes_per_step"], int) and isinstance(e["d2h_bytes_per_step"], int)
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["sample"]


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--workload", "single_128x128x256", "--steps", "2", "--warmup", "1"], 600)
    _common(d, 2, 1)
    assert d["impl"] == "reference"
    assert d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["value"] == d["value"]


def test_more_than_one_gpu_is_declined():
    d = _run(["--gpus", "2"], 600)
    assert "unavailable" in d and d["n_gpus"] == 2


@pytest.mark.gpu
def test_our_arm_line():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = _run(["--workload", "single_128x128x256", "--configs", "none", "--steps", "5", "--warmup", "3",
              "--e2e-steps", "2", "--cpu-seconds", "1", "--no-quantize", "--no-repack-step",
              "--clock-window-s", "0.3"], 900)
    _common(d, 5, 3)
    assert "impl" not in d or d["impl"] != "reference"
    r = d["roofline"]
    assert r["bound"] in ("hbm", "tensor", "alu") and r["unit"] in ("GB/s", "TFLOP/s")
    assert r["peak"] > 0 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert r["traffic"] is None or r["traffic"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 5
    clocks = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(clocks) and isinstance(clocks["reasons"], list)
