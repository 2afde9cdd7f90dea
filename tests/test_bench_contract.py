"""bench.py's JSON line carries every key of its contract: the reference arm
(the CPU oracle; no GPU) and, on a GPU, our arm on a small prefill case."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
             "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e")


def _run(args, timeout):
    r = subprocess.run([sys.executable, "bench.py"] + args, cwd=ROOT, capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--steps", "2", "--warmup", "1"], 600)
    for k in BASE_KEYS:
        assert k in d, k
    assert d["impl"] == "reference" and d["higher_is_better"] is True and d["unit"] == "tokens/s"
    assert d["config"]["workload"] == "prefill"
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == d["value"] and cpu["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # steps x ms_per_step is the time the timed samples took (each sample is one step)
    assert 0 < d["ms_per_step"] < 60_000 and d["ms_per_full_step_extrapolated"] >= d["ms_per_step"]


@pytest.mark.gpu
def test_our_arm_line_small_case():
    d = _run(["--tokens", "256", "--steps", "3", "--warmup", "3", "--no-cpu"], 900)
    for k in BASE_KEYS + ("roofline", "gpu_launches", "clocks", "kernels", "ll_decode"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["scaling"] == "weak"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["dtype"] == "bf16" and d["data"] == "synthetic"
    rl = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in rl, k
    assert rl["bound"] == "hbm" and rl["unit"] == "GB/s" and abs(rl["frac"] - rl["achieved"] / rl["peak"]) < 1e-3
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "tokens/s"
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 6 * 3            # layout, notify (2), dispatch, permute, combine per step
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    assert d["ll_decode"]["us_per_layer"] > 0 and "layer" in d["ll_decode"]
