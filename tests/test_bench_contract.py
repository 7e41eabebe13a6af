"""bench.py on the CPU: the reference arm (the float64 oracle on host cores) prints one
JSON line with the contract's keys, and the algorithmic accounting matches its formulas.
The GPU arm is exercised on the GPU (tests marked gpu, and the bench itself)."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_accounting():
    # 8 d flops per visible (query, key) pair; causal counts B H N^2 / 2 pairs.
    assert bench.alg_flops(2, 16, 4096, 64) == 8 * 64 * 2 * 16 * 4096 * 4096 / 2
    assert bench.alg_flops(1, 1, 6, 8, causal=False) == 8 * 8 * 36
    # 16 N d bytes per head in bf16: q1, k1, q2, k2 (4d) + v (2d) in, out (2d) out.
    assert bench.alg_bytes(2, 16, 4096, 64) == 2 * 16 * 4096 * 16 * 64
    # e4m3 queries/keys halve the 4d part.
    assert bench.alg_bytes(1, 1, 128, 64, qk_elem=1) == 128 * (4 * 64 + 4 * 64 * 2)


def test_traffic_record_parses():
    t = bench.read_traffic("needle_4k")
    # None when the committed record belongs to another kernel source; else bytes
    # per launch, at least the algorithmic bytes.
    assert t is None or t >= bench.alg_bytes(2, 16, 4096, 64)
    assert len(bench.kernel_source_hash()) == 16


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3
    assert d["config"]["workload"] == "needle_4k"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
