"""The N > 1 path of bench.py on CPU: two gloo ranks.

The decode path shards into independent (sequence, kv head) units, so N GPUs
run N replicas with no collective on the data path; the ranks meet only for
the barriers around the timed region and the maximum of their times.  These
tests run bench.py's replica helpers and its reference arm's rank gating in
two spawned CPU processes with the gloo backend.
"""

import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    bench.replica_init(world, "gloo")
    bench.replica_barrier(world)
    local_ms = 10.0 * (rank + 1)                      # rank 1 is the slower replica
    job_ms = bench.replica_max(local_ms, world, device="cpu")
    value = bench.job_throughput(1_000_000, world, job_ms)
    bench.replica_barrier(world)

    # reference arm: rank 0 alone runs (the oracle replaced by a fixed sample here)
    bench.oracle_sample = lambda wl, budget, max_rows=None: (2_000_000, 0.001, 3)
    args = bench.argparse.Namespace(workload="tiny_ring_sink_f32", steps=2, warmup=0)
    ref = bench.run_reference(args)
    bench.replica_done(world)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"job_ms": job_ms, "value": value, "ref": ref}, f)


@pytest.mark.timeout(300)
def test_two_gloo_replicas(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    # every rank sees the slowest replica's time; throughput counts all ranks' bytes
    assert [r["job_ms"] for r in res] == [20.0, 20.0]
    assert res[0]["value"] == pytest.approx(2 * 1_000_000 / 20e-3 / 1e9)
    assert res[0]["value"] == res[1]["value"]
    # reference arm: a line from rank 0 only, naming the world size
    assert res[1]["ref"] is None
    ref = res[0]["ref"]
    assert ref["impl"] == "reference" and ref["n_gpus"] == world
    assert ref["value"] == pytest.approx(2_000_000 / 0.001 / 1e9)
    assert ref["e2e"]["h2d_bytes_per_step"] == 0 and ref["e2e"]["d2h_bytes_per_step"] == 0
