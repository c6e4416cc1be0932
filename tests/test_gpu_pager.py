"""Page-in of pool blocks from pinned host memory, then decode ([pool] "KV
cache paging": a fixed pool of slots, blocks moved on demand by the copy
engine while attention runs, LRU residency, window blocks pinned).

One sequence of 64 blocks pages through a 12-slot pool over several steps.
Each step needs the 4 blocks of its sliding window (pinned) and 6 earlier
blocks; the pager plans, victims are evicted on the compute stream, the
page-ins are copied on a second stream while other work runs on the compute
stream, then committed.  The block table after each step must equal the
residency model's, and decode over the resident blocks must equal the
oracle's attention over exactly those tokens.
"""

import numpy as np
import pytest
import torch

from oracle.attention import decode_reference
from tests.gpu_harness import TOL
from tests.test_pager_cpu import Model

pytestmark = pytest.mark.gpu

L, HQ, HKV, D, BS, SLOTS, NLOG = 2, 8, 2, 128, 64, 12, 64


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import sliding_window_attention_kvc_gb300 as m
    return m


def test_pagein_then_decode_matches_resident_attention(kvc):
    d = kvc.make_desc("paged", "none", "bf16", L, 1, HQ, HKV, D, block_size=BS, num_blocks=SLOTS,
                      max_blocks_per_seq=NLOG)
    gen = torch.Generator().manual_seed(21)
    # host copy: [logical block][layer][K|V][kv head][row][D], pinned
    host = torch.randn((NLOG, L, 2, HKV, BS, D), generator=gen).to(torch.bfloat16).pin_memory()
    cache = kvc.alloc_cache(d, fill=float("nan"))
    ws = kvc.alloc_workspace(d)
    table = torch.full((1, NLOG), -1, dtype=torch.int32, device="cuda")
    valid = torch.zeros((SLOTS + 31) // 32, dtype=torch.int32, device="cuda")
    pager, model = kvc.Pager(SLOTS), Model(SLOTS)
    copy_stream = torch.cuda.Stream()
    rng = np.random.default_rng(4)
    t = NLOG * BS - 1
    window = list(range(NLOG - 4, NLOG))
    busy = torch.zeros(1 << 22, device="cuda")
    g = HQ // HKV
    for step in range(6):
        need = window + rng.choice(NLOG - 4, size=6, replace=False).tolist()
        pinned = [1] * 4 + [0] * 6
        ins, outs = pager.plan(need, pinned)
        assert (ins, outs) == model.plan(need, pinned)
        pager.evict(d, 0, outs, table, valid)
        pager.issue(d, cache, host, ins, copy_stream)
        busy.mul_(1.0001)                          # compute-stream work overlapping the copies
        pager.commit(d, 0, ins, table, valid)
        want = np.full(NLOG, -1)
        for s, lb in enumerate(model.block):
            if lb >= 0:
                want[lb] = s
        assert table[0].cpu().numpy().tolist() == want.tolist()
        q = torch.randn((1, HQ, D), generator=gen).to(torch.bfloat16)
        pos = torch.tensor([t], dtype=torch.int32, device="cuda")
        for layer in range(L):
            out = kvc.decode_attention(d, cache, layer, q.cuda(), pos, ws, block_table=table, valid_bits=valid)
            got = out.float().cpu().numpy()[0]
            resident = sorted(lb for lb in model.block if lb >= 0)
            ps = [lb * BS + r for lb in resident for r in range(BS)]
            for h in range(HKV):
                K = np.concatenate([host[lb, layer, 0, h].double().numpy() for lb in resident])
                V = np.concatenate([host[lb, layer, 1, h].double().numpy() for lb in resident])
                ref = decode_reference(q[0, h * g:(h + 1) * g].double().numpy(), K, V, ps, t, rope="none",
                                       storage="bf16")
                assert np.abs(got[h * g:(h + 1) * g] - ref).max() <= TOL["bf16"], (step, layer, h)
    assert kvc.get_error(ws) == 0
