"""The benchmark's JSON contract, checked on the CPU: the reference arm (the oracle on the host cores)
runs without a GPU, and its one JSON line carries the keys and types the contract names."""
import json
import os
import subprocess
import sys

import numpy as np

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, stdout=subprocess.PIPE,
                       stderr=subprocess.PIPE, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout  # exactly one JSON line
    return json.loads(lines[0])


def test_reference_arm_json_line():
    d = run_bench("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert d["impl"] == "reference"
    for key, typ in (("metric", str), ("value", float), ("unit", str), ("steps", int), ("warmup", int),
                     ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str), ("dtype", str),
                     ("data", str), ("config", dict), ("cpu_baseline", dict), ("e2e", dict)):
        assert isinstance(d[key], typ), key
    assert d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    # the default workload, the same as the GPU arm's headline
    assert d["config"]["workload"] == "prefill_8192tok_48layer_stack"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert cb["cores"] == cb["threads"] == bench.host_cores()
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_whole_job_rate():
    # tokens per step x steps x ranks / total seconds
    assert bench.whole_job_rate(4, 10, 2, 100.0) == 4 * 10 * 2 / 0.1


def test_oracle_baseline_uses_every_core_and_one_thread():
    rec = bench.oracle_baseline(0, 0, budget_s=0.0, single_thread=True)
    assert rec["cores"] == rec["threads"] == rec["host_cores"] == bench.host_cores()
    assert rec["value"] > 0 and rec["single_thread"]["threads"] == 1 and rec["single_thread"]["value"] > 0


def test_expert_load_record():
    ids = np.array([[[0, 1], [0, 2], [0, 1]]], dtype=np.int32)  # one layer, 3 tokens, top-2
    rec = bench.expert_load(ids)
    assert rec["experts_touched"] == 3 and rec["max_tokens_per_expert"] == 3
    assert rec["mean_tokens_per_touched_expert"] == 2.0 and rec["max_over_mean"] == 1.5
    assert rec["tokens_per_expert_sorted"] == [3, 2, 1]


def test_step_tensor_fraction_counts_expert_and_router_flops():
    rec = bench.step_tensor_fraction({"T": 8192, "L": 48}, 100.0)
    assert rec["flops_per_step"] == 48 * 8192 * (10 * 9830400 + 2 * 512 * 2560)


def test_expert_roofline_takes_each_expert_by_its_bound():
    """One expert with 10,000 tokens is bound by its flops, 100 experts with one token each by their
    blobs' bytes; the ideal time is the sum of the two, and frac is ideal / measured."""
    hbm, tc, _, _ = bench.load_peaks()
    ids = np.concatenate([np.zeros(10000, dtype=np.int32), np.arange(1, 101, dtype=np.int32)])[None]
    roof = {"avg_launch_ms": 1.0, "other_expert_kernel": {"avg_launch_ms": 1.0}}
    rec = bench.expert_roofline({"T": 10100, "L": 1}, ids, roof)
    per_pair = bench.FLOPS_PER_PAIR["TC_GATEUP"] + bench.FLOPS_PER_PAIR["TC_DOWN"]
    want = (10000 * per_pair / (tc * 1e12) + 100 * bench.BLOB / (hbm * 1e9)) * 1e3
    assert abs(rec["ideal_ms_per_layer"] - want) < 1e-12
    assert rec["expert_kernels_ms_per_layer"] == 2.0 and abs(rec["frac"] - want / 2.0) < 1e-12
