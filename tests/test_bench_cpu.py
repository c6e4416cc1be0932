"""bench.py's reference arm (the fp64 oracle on the host cores) prints the
JSON line the benchmark contract asks for; runs on the CPU."""

import argparse
import json

import bench
import kvc_synth


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


def test_attended_count_matches_the_oracle_sets():
    """The bench's closed-form key counts (its FLOP and byte figures) equal the
    sizes of the oracle's attended sets ([ring] 2.2, [sink] cache-set
    equation, [pool] mapped and valid blocks)."""
    import oracle
    for name in ("ring_bf16", "sink_window_bf16", "paged_shared_prefix_bf16", "long_context_pool_bf16"):
        for small in (True, False):
            wl = bench.kvc_synth.make_workload(name, small=small)
            for b in range(min(wl.batch, 3)):
                tb = int(wl.positions[b])
                for t in (tb, tb - 5, 0, 3, tb - 200):
                    if t < 0:
                        continue
                    if wl.layout == "window":
                        ref = len(oracle.window_attended(t, wl.sinks, wl.window))
                    else:
                        ref = len(oracle.paged_attended(t, wl.block_table[b], wl.valid, wl.block_size))
                    assert bench.attended_count(wl, b, t) == ref, (name, b, t)


def test_launches_per_step_follow_the_library():
    """The launch count bench.py claims per kvc_decode_step, as the library's
    host code launches them: a paged batch's plan kernel, the decode kernel and
    its combine; window layouts and a one-sequence paged cache (planned in the
    decode kernel): decode and combine; fp32 window caches: append and decode."""
    class _St:
        pass
    want = {"paged_shared_prefix_bf16": 3, "paged_shared_prefix_int8": 3, "ring_bf16": 2, "sink_window_bf16": 2,
            "ring_int8": 2, "sink_window_int8": 2, "long_context_pool_bf16": 2, "tiny_ring_sink_f32": 2}
    for name, n in want.items():
        st = _St()
        st.wl = kvc_synth.make_workload(name)
        assert bench.DecodeState.launches_per_step(st) == n, name


def test_profile_commands_run_with_the_current_options_and_kernels():
    """Every bench.py command quoted under profiles/ parses with the bench's
    own options, and every ncu kernel filter there names a kernel defined in
    the sources, so each summary can be re-made as written."""
    import glob
    import os
    import re
    import shlex

    root = os.path.dirname(os.path.abspath(bench.__file__))
    src = ""
    for path in glob.glob(os.path.join(root, "sliding_window_attention_kvc_gb300", "csrc", "*")):
        with open(path) as f:
            src += f.read()
    kernels = set()
    for m in re.finditer(r"__global__", src):
        # the first name followed by "(" that is not the launch-bounds qualifier
        # or an expression inside it
        for name in re.findall(r"\b(\w+)\s*\(", src[m.end():m.end() + 300]):
            if name not in ("__launch_bounds__", "decode_ctas_per_sm"):
                kernels.add(name)
                break
    assert {"decode_mma_kernel", "combine_streamk_kernel", "plan_rows_kernel", "prefill_ws_kernel"} <= kernels
    ap = bench.build_parser()
    commands = filters = 0
    for path in sorted(glob.glob(os.path.join(root, "profiles", "*.md"))):
        with open(path) as f:
            text = f.read()
        for m in re.finditer(r"python bench\.py([^`\n]*)", text):
            argv = shlex.split(re.sub(r"\[[^\]]*\]", "", m.group(1)))   # drop optional parts in brackets
            ap.parse_args(argv)
            commands += 1
        for m in re.finditer(r"-k regex:(\"[^\"]+\"|\S+)", text):
            pat = re.compile(m.group(1).strip('"'))
            assert any(pat.search(k) for k in kernels), (os.path.basename(path), m.group(1))
            filters += 1
    assert commands >= 10 and filters >= 5
