"""bench.py's JSON line on a reduced workload: one line carrying every key the
measurement contract asks for, with self-consistent values."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_has_the_contract_keys():
    args = [sys.executable, os.path.join(ROOT, "bench.py"), "--N", "8192", "--heads", "2", "--steps", "2",
            "--warmup", "3", "--cpu-rows", "8", "--no-striped", "--no-varlen", "--no-ffn"]
    r = subprocess.run(args, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(ln) for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] >= 3 and d["value"] > 0
    assert d["config"]["N"] == 8192 and "workload" in d["config"]
    roof = d["roofline"]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s" and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert roof["traffic"] is None   # DRAM bytes are only known for the captured workload
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 4 * 8192 * 2 * 128 * 2   # q, k, v, dO in bf16
    assert e["d2h_bytes_per_step"] > 0
    # per step: 1 forward, 1 backward and the small passes around them
    assert d["gpu_launches"] >= 2 * d["steps"]
    assert d["clocks"]["sm_max_mhz"] > 0
    # which of copies and kernels sets the end-to-end pace, from the library's own events
    br = e["breakdown"]
    assert br["bound_by"] in ("copies", "kernels")
    assert br["h2d_ms_per_step"] > 0 and br["d2h_ms_per_step"] > 0 and br["kernel_ms_per_step"] > 0
    assert br["h2d_gbs"] > 0 and br["d2h_gbs"] > 0
    assert d["other_workloads"] is None   # the other named workloads run only at the bench workload
