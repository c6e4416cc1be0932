"""The seeded input generator: determinism, keying, workload structure."""

import numpy as np
import pytest
import torch

from kvc_synth import POSITION_BLOCK, make_workload, randn
from kvc_synth.workloads import paged_shared_prefix_bf16, long_context_pool_bf16, ring_bf16


def test_randn_is_keyed_and_deterministic():
    a = randn((1, 2, 3), (4, 5), "bf16")
    b = randn((1, 2, 3), (4, 5), "bf16")
    c = randn((1, 2, 4), (4, 5), "bf16")
    assert a.dtype == torch.bfloat16 and torch.equal(a, b) and not torch.equal(a, c)


def test_position_values_do_not_depend_on_the_requested_range():
    wl = ring_bf16(small=True)
    k_all, v_all = wl.kv_history(0, 2, np.arange(POSITION_BLOCK - 5, POSITION_BLOCK + 40))
    k_one, v_one = wl.kv_history(0, 2, [POSITION_BLOCK + 3])
    assert torch.equal(k_all[8], k_one[0]) and torch.equal(v_all[8], v_one[0])


def test_shared_prefix_tokens_are_one_token_per_group():
    wl = paged_shared_prefix_bf16(small=True)
    g = wl.group
    b0, b1 = [b for b in range(wl.batch) if g[b] == g[2]][:2]
    n = int(min(wl.shared_tokens[b0], wl.shared_tokens[b1]))
    assert n > 0
    k0, _ = wl.kv_history(0, b0, np.arange(n))
    k1, _ = wl.kv_history(0, b1, np.arange(n))
    assert torch.equal(k0, k1)
    # own tokens differ
    p = int(max(wl.shared_tokens[b0], wl.shared_tokens[b1]))
    ka, _ = wl.kv_history(0, b0, [p])
    kb, _ = wl.kv_history(0, b1, [p])
    assert not torch.equal(ka, kb)


def test_paged_tables_map_each_private_block_once():
    for small in (True, False):
        wl = paged_shared_prefix_bf16(small=small)
        t = wl.table if hasattr(wl, "table") else wl.block_table
        used = {}
        for b in range(wl.batch):
            nblk = int(wl.positions[b]) // wl.block_size + 1
            assert (t[b, :nblk] >= 0).all() and (t[b, nblk:] == -1).all()
            for lb in range(nblk):
                used.setdefault(int(t[b, lb]), set()).add((int(wl.group[b]), lb))
        # a physical block is shared only by members of one group at one logical index
        for phys, owners in used.items():
            assert len(owners) == 1
        assert sorted(used) == list(range(wl.num_blocks))


def test_pool_workload_structure():
    wl = long_context_pool_bf16(small=False)
    tb = wl.block_table[0]
    assert wl.positions[0] == 262143 and tb.shape[0] == 4096
    mapped = tb[tb >= 0]
    assert sorted(mapped) == list(range(1024))
    assert (tb[-64:] >= 0).all() and wl.valid[tb[-64:]].all()
    assert 0.4 < wl.valid.mean() < 0.6


@pytest.mark.parametrize("density", [0.25, 1.0])
def test_pool_valid_density_sweep(density):
    # the same resident blocks and slot order; only the valid bits follow the
    # density, and the last 4096 tokens stay valid
    base = long_context_pool_bf16(small=False)
    wl = long_context_pool_bf16(small=False, density=density)
    assert np.array_equal(wl.block_table, base.block_table)
    tb = wl.block_table[0]
    assert wl.valid[tb[-64:]].all()
    # Bernoulli(density) over the 960 earlier slots, plus the 64 forced ones
    assert abs(wl.valid.mean() - (density + (1 - density) * 64 / 1024)) < 0.03
    if density == 1.0:
        assert wl.valid.all()


def test_bench_density_option_is_pool_only():
    import argparse

    import bench
    ns = argparse.Namespace(workload="long_context_pool_bf16", density=0.25)
    assert bench._workload_kw(ns) == {"density": 0.25}
    assert bench._workload_kw(argparse.Namespace(workload="ring_bf16", density=None)) == {}
    with pytest.raises(SystemExit):
        bench._workload_kw(argparse.Namespace(workload="ring_bf16", density=0.25))
    with pytest.raises(SystemExit):
        bench._workload_kw(argparse.Namespace(workload="long_context_pool_bf16", density=1.5))
    rows = [bench.step_bytes(make_workload("long_context_pool_bf16", density=x))["kv_unique"]
            for x in (0.25, 0.5, 1.0)]
    assert rows[0] < rows[1] < rows[2]


def test_full_size_shapes():
    wl = make_workload("ring_bf16")
    assert wl.cache_shape(8) == (8, 2, 8, 8, 4096, 128)
    assert (wl.positions >= 4096).all() and (wl.positions <= 65536).all()
    wl = make_workload("sink_window_bf16")
    assert wl.capacity == 4096 and wl.sinks == 4
    wl = make_workload("tiny_ring_sink_f32")
    assert wl.capacity == 64 and wl.steps == 256
