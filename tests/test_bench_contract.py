"""The benchmark's one-line JSON contract, checked on the lines bench.py
prints: the reference arm (the oracle, on the host) here on the CPU, our arm
on the GPU, both on the small 256x256 workload."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=600):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         capture_output=True, text=True, timeout=timeout, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def _common(d, steps, warmup):
    for k in ("metric", "unit", "dtype", "data"):
        assert isinstance(d[k], str) and d[k]
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # at least 3 warm-up steps whatever is asked; the line reports those run
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == max(3, warmup)
    assert d["higher_is_better"] is True
    assert d["scaling"] in ("weak", "strong")
    assert d["vs_baseline"] is None
    assert isinstance(d["config"], dict) and "workload" in d["config"]
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] >= 0 and e["d2h_bytes_per_step"] >= 0


def test_reference_arm_line():
    d = _bench("--impl", "reference", "--workload", "toy256", "--steps", "2", "--warmup", "1")
    _common(d, 2, 1)
    assert d["impl"] == "reference"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and cb["sample"]
    assert d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_our_arm_line():
    d = _bench("--workload", "toy256", "--steps", "3", "--warmup", "3", "--cpu-seconds", "1",
               "--no-extra-ops")
    _common(d, 3, 3)
    assert d.get("impl", "ours") != "reference"
    r = d["roofline"]
    assert r["bound"] in ("hbm", "tensor", "alu") and r["unit"] in ("GB/s", "TFLOP/s")
    assert r["achieved"] > 0 and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) <= 1e-3 * max(1.0, r["frac"])
    assert r["traffic"] is None or r["traffic"] > 0
    assert r["gather_gbs"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
    assert cb["all_cores"]["cores"] >= 1 and cb["all_cores"]["value"] > 0
    assert d["gpu_launches"] > 0
    c = d["clocks"]
    assert c["sm_mhz"] > 0 and c["sm_max_mhz"] > 0 and isinstance(c["reasons"], list)
    # the end-to-end number moves real bytes and is not the device-timed value
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["e2e"]["value"] != d["value"]
    lo, mid, hi = d["e2e"]["ms_per_step_min_median_max"]
    assert 0 < lo <= mid <= hi
    for o in d["ops"]:
        assert o["us"] > 0 and o["us_median"] > 0 and o["gather_gbs"] > 0
