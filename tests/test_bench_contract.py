"""bench.py's JSON line: the keys and units the benchmark contract asks for.

The reference arm (the fp64 oracle on the host cores) runs without a GPU;
our arm runs on a small shape under the gpu marker.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                         timeout=timeout, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_reference_arm_json_line():
    d = _run(["--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-heads", "1"], timeout=300)
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_our_arm_json_line():
    d = _run(["--shape", "2,8,1024,128,1", "--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--graph"],
             timeout=600)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks",
                "hbm", "kernels"):
        assert key in d, key
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and 0 < r["frac"] < 1.5
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert d["gpu_launches"] == 4 * d["steps"]  # forward, row terms, dK/dV pass, dQ pass
    e = d["e2e"]
    assert e["unit"] == "TFLOP/s" and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["value"] < d["value"]  # host copies are inside its timed region
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    assert d["config"]["causal"] is True and d["dtype"] == "bf16"
    # median and spread over the timed steps, peak allocated memory
    sp = d["spread"]
    assert sp["ms_p10"] <= sp["ms_median"] <= sp["ms_p90"]
    assert sp["value_p10"] <= sp["value_median"] <= sp["value_p90"]
    assert d["peak_mem_bytes"] > 0
    # the end-to-end line explains itself: copy bandwidths and the floor they set
    assert e["h2d_gbs_alone"] > 0 and e["d2h_gbs_alone"] > 0
    assert e["floor_ms"] >= e["copy_ms_both_directions_at_once"] and e["floor_ms"] > 0
    # the same step replayed from a CUDA graph
    g = d["graph"]
    assert g["ms_per_step"] > 0 and g["value"] > 0
