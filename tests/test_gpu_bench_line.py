"""bench.py's JSON line on a GPU: a short run of the default workload must
print one line with every key of the benchmark contract, of the right type
and consistent with itself (roofline fraction, launch count, copy bytes)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def line():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    steps, warmup = 5, 3
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", str(steps),
                        "--warmup", str(warmup), "--e2e-steps", "3"],
                       capture_output=True, text=True, cwd=ROOT, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    d["_steps"], d["_warmup"] = steps, warmup
    return d


def test_headline_keys(line):
    assert "queries" in line["metric"] and line["unit"] == "queries/s"
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["n_gpus"] == 1 and line["steps"] == line["_steps"]
    assert line["warmup"] == line["_warmup"]
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["vs_baseline"] is None and line["data"] == "synthetic"
    assert line["dtype"] == "f32"                      # bf16 storage, fp32 workspace
    assert "workload" in line["config"] and "l2" in line["config"]
    # value = queries per step / time per step
    q = line["config"]["queries_per_step"]
    assert abs(line["value"] - q / (line["ms_per_step"] * 1e-3)) <= 1e-3 * line["value"]


def test_roofline(line):
    r = line["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] > 0 and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert r["traffic"] is None or r["traffic"] > 0
    for k in ("atomic_roofline", "gather_roofline"):
        s = line[k]
        assert 0 < s["frac"] < 1.5 and abs(s["frac"] - s["achieved"] / s["peak"]) < 1e-3


def test_cpu_baseline_e2e_launches_clocks(line):
    c = line["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["sample"]
    e = line["e2e"]
    assert e["value"] > 0 and e["unit"] == line["unit"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert line["gpu_launches"] == 4 * line["steps"]     # forward, zero, accumulate, finish
    clk = line["clocks"]
    assert clk is None or (clk["sm_mhz"] > 0 and isinstance(clk["reasons"], list))


def test_sub_lines(line):
    f = line["f32_encoder"]
    assert f["dtype"] == "f32" and f["value"] > 0 and f["gpu_launches"] == 3 * f["steps"]
    modes = line["accumulator_modes"]
    assert modes["native"]["accumulator_resolved"] == "native"
    assert modes["fp16_buffer"]["accumulator_resolved"] == "fp16_buffer"
    assert modes["fp16_buffer"]["dtype"] == "f16" and modes["native"]["dtype"] == "bf16"
    for m in ("native", "fp16_buffer"):
        assert modes[m]["value"] > 0
