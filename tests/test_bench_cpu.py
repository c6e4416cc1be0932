"""bench.py's reference arm (the fp64 oracle on the host cores) prints the
JSON line the benchmark contract asks for; runs on the CPU."""

import argparse
import json

import bench


def test_reference_arm_line_keeps_the_contract():
    args = argparse.Namespace(workload="ring_bf16", density=None, steps=1, warmup=3)
    line = json.loads(json.dumps(bench.run_reference(args)))
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["steps"] == 1
    # the same metric and config as the GPU arm, so that the two lines divide
    assert line["metric"] == bench.METRIC and line["unit"] == "GB/s" and line["higher_is_better"]
    wl = bench.kvc_synth.make_workload("ring_bf16")
    assert line["config"] == bench.workload_config(wl, bench.DEFAULT_LAYERS["ring_bf16"], 1, {})
    assert line["config"]["workload"] == "ring_bf16" and line["value"] > 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_takes_the_pool_density():
    args = argparse.Namespace(workload="long_context_pool_bf16", density=0.25, steps=1, warmup=3)
    line = bench.run_reference(args)
    assert line["config"]["workload"] == "long_context_pool_bf16" and line["config"]["density"] == 0.25
