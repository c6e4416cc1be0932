"""Chunked prefill (kvc_prefill) on the GPU against oracle.prefill.

The cache is first filled as it stands before the chunk (every position the
decode step at pos0 would attend, except pos0 itself), then one call prefills
T tokens per sequence.  Outputs are compared element by element with the
oracle (tolerance 2e-2, bf16 outputs); the cache the call leaves must equal
the cache after a plain kvc_append of the same chunk (so the ring slots the
chunk overwrites were read before they were overwritten).  Cases: ring with a
chunk across the first wrap and far past it, sink + ring, paged with shared
prefix blocks, a chunk that starts at position 0, ragged chunk lengths (not a
multiple of the 16 tokens a CTA takes), left padding, RoPE none, baked and read
at in-cache positions; INT8 caches (ring, sink + ring with baked and read-time
RoPE, paged, head_dim 128 and 256), whose keys and values are compared with the
oracle as the cache reads them back.
"""

import dataclasses

import numpy as np
import pytest
import torch

import bench
import kvc_synth
import oracle
from oracle.prefill import prefill_sequence
from tests.gpu_harness import TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import sliding_window_attention_kvc_gb300 as m
    return m


def _attended_fn(wl, b):
    if wl.layout == "window":
        return lambda t: oracle.window_attended(t, wl.sinks, wl.window)
    return lambda t: oracle.paged_attended(t, wl.block_table[b], wl.valid, wl.block_size)


def _run(kvc, wl, pos0, T, layer=0):
    """Prefill T tokens at pos0 [B]; returns (got [B, T, Hq, D], state, chunk q/k/v)."""
    # the cache as it stands before the chunk (no history before position 0)
    wl0 = dataclasses.replace(wl, positions=np.maximum(np.asarray(pos0, dtype=np.int64), 0))
    st = bench.DecodeState(wl0, 1, source="cpu")
    B, Hq, Hkv, D = wl.batch, wl.q_heads, wl.kv_heads, wl.head_dim
    q = torch.zeros((B, T, Hq, D), dtype=torch.bfloat16)
    k = torch.zeros((B, T, Hkv, D), dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    for b in range(B):
        ps = np.arange(pos0[b], pos0[b] + T)
        keep = ps >= 0
        kb, vb = wl.kv_history(layer, b, ps[keep])
        k[b, keep] = kb
        v[b, keep] = vb
        for i, t in enumerate(ps):
            if t >= 0:
                q[b, i] = wl.query(layer, b, int(t))
    ws = kvc.alloc_prefill_workspace(st.desc, T)
    ref_cache = st.cache.clone()
    pos_t = torch.from_numpy(np.asarray(pos0, dtype=np.int32)).cuda()
    out = kvc.prefill(st.desc, st.cache, layer, q.cuda(), k.cuda(), v.cuda(), pos_t, ws, block_table=st.table,
                      valid_bits=st.valid_bits)
    kvc.append(st.desc, ref_cache, layer, k.cuda(), v.cuda(), pos_t, ws, block_table=st.table)
    torch.cuda.synchronize()
    assert kvc.get_error(ws) == 0
    return out.float().cpu().numpy(), st, ref_cache, q, k, v


def _oracle(wl, b, pos0, T, q, layer=0):
    N = max(pos0 + T, 1)
    K, V = wl.kv_history(layer, b, np.arange(N))
    K, V = K.double().numpy(), V.double().numpy()
    if wl.dtype == "i8":
        # rows as an INT8 cache reads them back; baked keys are quantised after
        # rotation, inside the oracle
        V = oracle.quant.store_i8(V)
        if wl.rope != "baked":
            K = oracle.quant.store_i8(K)
    spec = dict(rope=wl.rope, base=wl.rope_base, storage=wl.dtype, sinks=wl.sinks, window=wl.window)
    return prefill_sequence(q[b].double().numpy(), K, V, pos0, _attended_fn(wl, b), **spec)


CASES = {
    # name: (workload, rope, pos0 per sequence, T)
    "ring_wrap": ("ring_bf16", "baked", [150, 190, 4300], 37),
    "ring_none_long": ("ring_bf16", "none", [0, 64, 1000], 70),
    "sink_baked": ("sink_window_bf16", "baked", [3, 180, 987600], 45),
    "sink_none": ("sink_window_bf16", "none", [100, 150, 50000], 33),
    # read-time RoPE (the sink workload's own mode): keys rotated at their
    # in-cache positions relative to each chunk token
    "sink_read": ("sink_window_bf16", "read_time", [3, 180, 987600], 45),
    "ring_read": ("ring_bf16", "read_time", [150, 190, 4300], 37),
    # head_dim 64 (the mma.sync kernel; 128 runs on tcgen05)
    "ring_d64": ("ring_bf16", "baked", [150, 190, 4300], 37, {"head_dim": 64}),
    "sink_read_d64": ("sink_window_bf16", "read_time", [3, 180, 987600], 45, {"head_dim": 64}),
    # several CTAs per (sequence, kv head) along the chunk
    "ring_long_chunk": ("ring_bf16", "baked", [150, 190, 4300], 130),
    # head_dim 256 (the long-context pool's head size)
    "ring_d256": ("ring_bf16", "baked", [150, 190, 4300], 37, {"head_dim": 256}),
    "sink_read_d256": ("sink_window_bf16", "read_time", [3, 180, 987600], 45, {"head_dim": 256}),
    # a chunk longer than the window: the pre-tile kernels take it
    "ring_chunk_past_window": ("ring_bf16", "baked", [150, 190, 4300], 230),
    # INT8 caches: cached keys expanded from codes in the kernel, the chunk's
    # own rows staged as the cache reads them back
    "ring_i8": ("ring_int8", "baked", [150, 190, 4300], 37),
    "ring_i8_none": ("ring_int8", "none", [0, 64, 1000], 70),
    "sink_i8_read": ("sink_window_int8", "read_time", [3, 180, 987600], 45),
    "sink_i8_baked": ("sink_window_int8", "baked", [3, 180, 987600], 45),
    "ring_i8_d256": ("ring_int8", "baked", [150, 190, 4300], 37, {"head_dim": 256}),
    # a capacity that is not a multiple of 4: tiles' row scales start off a
    # 16-byte boundary
    "ring_i8_odd_capacity": ("ring_int8", "baked", [150, 190, 4300], 37, {"window": 198}),
    "sink_i8_read_d256": ("sink_window_int8", "read_time", [3, 180, 987600], 45, {"head_dim": 256}),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_prefill_window_layouts(kvc, case):
    name, rope, pos0, T, *extra = CASES[case]
    wl = dataclasses.replace(kvc_synth.make_workload(name, small=True), rope=rope, **(extra[0] if extra else {}))
    got, st, ref_cache, q, _, _ = _run(kvc, wl, pos0, T)
    assert np.isfinite(got).all()
    for b in range(wl.batch):
        ref = _oracle(wl, b, pos0[b], T, q)
        err = float(np.abs(got[b] - ref).max())
        assert err <= TOL[wl.dtype], (case, b, err)
    a, r = st.cache.float(), ref_cache.float()
    same = (a == r) | (torch.isnan(a) & torch.isnan(r))
    assert bool(same.all())


@pytest.mark.parametrize("name", ["paged_shared_prefix_bf16", "paged_shared_prefix_int8"])
def test_prefill_paged_shared_prefix(kvc, name):
    wl = kvc_synth.make_workload(name, small=True)
    T = 29
    pos0 = [max(int(t) - T + 1, 0) for t in wl.positions]     # the chunk ends at each sequence's mapped tail
    got, st, ref_cache, q, _, _ = _run(kvc, wl, pos0, T)
    assert np.isfinite(got).all()
    for b in range(wl.batch):
        Tb = min(T, int(wl.positions[b]) + 1 - pos0[b])         # rows past the mapped tail are not compared
        ref = _oracle(wl, b, pos0[b], T, q)
        err = float(np.abs(got[b, :Tb] - ref[:Tb]).max())
        assert err <= TOL[wl.dtype], (b, err)


def test_prefill_left_padding(kvc):
    wl = kvc_synth.make_workload("ring_bf16", small=True)
    pos0, T = [-5, 10, -1], 21
    got, st, ref_cache, q, _, _ = _run(kvc, wl, pos0, T)
    for b in range(wl.batch):
        pad = max(0, -pos0[b])
        assert not got[b, :pad].any()
        ref = _oracle(wl, b, pos0[b], T, q)
        assert float(np.abs(got[b] - ref).max()) <= TOL["bf16"], b


def test_prefill_long_context_pool_d256(kvc):
    """The pool's shape (head_dim 256, 64-token blocks, valid mask): a chunk of
    96 tokens ending at the sequence's position, in its always-resident tail."""
    wl = kvc_synth.make_workload("long_context_pool_bf16", small=True)
    T = 96
    pos0 = [int(wl.positions[0]) - T + 1]
    got, st, ref_cache, q, _, _ = _run(kvc, wl, pos0, T)
    assert np.isfinite(got).all()
    ref = _oracle(wl, 0, pos0[0], T, q)
    assert float(np.abs(got[0] - ref).max()) <= TOL["bf16"]


def test_prefill_long_context_pool_int8_d256(kvc):
    """The pool's shape over an INT8 cache (head_dim 256, 64-token blocks, NaN
    scales in the non-resident slots)."""
    wl = kvc_synth.as_int8(kvc_synth.make_workload("long_context_pool_bf16", small=True), "long_context_pool_int8_small")
    T = 96
    pos0 = [int(wl.positions[0]) - T + 1]
    got, st, ref_cache, q, _, _ = _run(kvc, wl, pos0, T)
    assert np.isfinite(got).all()
    ref = _oracle(wl, 0, pos0[0], T, q)
    assert float(np.abs(got[0] - ref).max()) <= TOL["i8"]
