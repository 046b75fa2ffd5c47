"""bench.py accounting: the per-row flops used for the CPU baseline add up to
the whole-problem formula used for the GPU metric, and the formula matches the
stated causal-adjusted counts (fwd 4*B*H*N^2*d/2, bwd 2.5x fwd)."""
import os

import pytest

import bench


def test_causal_flops_formula():
    fwd, bwd = bench.algo_flops(1, 131072, 16, 128, causal=True)
    assert fwd == pytest.approx(70.37e12, rel=1e-3)
    assert bwd == pytest.approx(175.9e12, rel=1e-3)
    fwd_nc, _ = bench.algo_flops(1, 512, 2, 64, causal=False)
    assert fwd_nc == 4 * 2 * 512 * 512 * 64


@pytest.mark.parametrize("N,H,d", [(64, 3, 32), (1024, 2, 128)])
def test_row_flops_sum_to_whole_problem(N, H, d):
    fwd, bwd = bench.algo_flops(1, N, H, d, causal=True)
    rows = H * sum(bench.row_flops(i, d, True, N) for i in range(N))
    # rows see i+1 keys: N(N+1)/2 visible pairs against the formula's N^2/2
    assert rows == pytest.approx((fwd + bwd) * (N + 1) / N, rel=1e-12)
    rows_nc = H * sum(bench.row_flops(i, d, False, N) for i in range(N))
    f2, b2 = bench.algo_flops(1, N, H, d, causal=False)
    assert rows_nc == pytest.approx(f2 + b2, rel=1e-12)


def _run_bench(args, env_extra=None):
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ)
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py")] + args, cwd=root, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    return [json.loads(ln) for ln in lines]


def test_reference_arm_prints_one_contract_line():
    # the reference arm (the oracle on host cores) on a small override of the workload
    lines = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-rows", "8",
                        "--N", "2048", "--heads", "2"])
    assert len(lines) == 1
    d = lines[0]
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["warmup"] >= 3
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert "workload" in d["config"] and d["config"]["N"] == 2048
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    lines = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-rows", "8",
                        "--N", "2048", "--heads", "2"],
                       {"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2", "MASTER_ADDR": "127.0.0.1"})
    assert lines == []


def test_reference_arm_named_workload_preset():
    # workload 1 (fp32, non-causal) through the preset: its sizes and mask reach the line
    lines = _run_bench(["--impl", "reference", "--config", "1", "--steps", "1", "--warmup", "3",
                        "--ref-rows", "64"])
    assert len(lines) == 1
    c = lines[0]["config"]
    assert c["N"] == 512 and c["Hq"] == 2 and c["d"] == 64 and c["P"] == 4 and c["causal"] is False
    assert c["workload"].startswith("workload 1")


def test_reference_arm_config_has_the_gpu_arms_keys():
    lines = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-rows", "8",
                        "--N", "2048", "--heads", "2"])
    assert set(lines[0]["config"]) == set(bench.bench_config(1))
    assert lines[0]["config"]["parallelism"] == "single GPU"


def test_input_generators_do_not_map_the_library():
    # the reference arm and the oracle's callers import the seeded generators;
    # that import must leave the product library unloaded
    import subprocess
    import sys
    code = ("import blockwise_exact_attention_ra_gb300.inputs, oracle\n"
            "maps = open('/proc/self/maps').read()\n"
            "print('libra.so' in maps)\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == "False"
