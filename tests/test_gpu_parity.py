"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

* cache placement after kvc_append: slot / block of every appended position
  bit-exact, values bit-exact (raw K, V) or within one bf16 ulp (RoPE baked);
* attended sets bit-exact, recovered through the real decode kernel with
  K = 0 and one-hot V rows;
* decode outputs element by element at small sizes (several tiles, ragged
  tails, before and after the first ring wrap) and on sampled sequences at
  the full workload sizes in the launch configuration bench.py times;
* edge cases: first token, empty attended set, more splits than rows,
  NaN-poisoned slots outside the attended set, device error bits.
Tolerances: max abs error 2e-3 for fp32 caches, 2e-2 for bf16 caches.
"""

import numpy as np
import pytest
import torch

import bench
import kvc_synth
import oracle
from tests.gpu_harness import TOL, attended, oracle_outputs, run_stepwise

pytestmark = pytest.mark.gpu

SMALL = ["ring_bf16", "sink_window_bf16", "paged_shared_prefix_bf16", "long_context_pool_bf16"]


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import sliding_window_attention_kvc_gb300 as m
    return m


def _maxerr(got, ref):
    return float(np.abs(np.asarray(got, dtype=np.float64) - ref).max())


# ---------------------------------------------------------------------------
# append: where every position lands, and what is stored
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", SMALL)
def test_append_places_rows_at_the_oracle_slot(kvc, name):
    wl = kvc_synth.make_workload(name, small=True)
    st = bench.DecodeState(wl, 1, source="cpu")
    cache = st.cache[0].float().cpu().numpy()          # [2, X, Hkv, R, D]
    for b in range(wl.batch):
        t = int(wl.positions[b])
        pos = attended(wl, b)
        pos = pos[pos < t]                              # the step's own token is appended by step()
        k, v = wl.kv_history(0, b, pos)
        k, v = k.double().numpy(), v.double().numpy()
        if wl.layout == "window":
            slots = oracle.window_slot(pos, wl.sinks, wl.window)
            gk = cache[0, b][:, slots].transpose(1, 0, 2)
            gv = cache[1, b][:, slots].transpose(1, 0, 2)
        else:
            phys = wl.block_table[b, pos // wl.block_size]
            rows = pos % wl.block_size
            gk = cache[0][phys, :, rows]
            gv = cache[1][phys, :, rows]
        assert np.array_equal(gv, v), "V must be stored unchanged"
        if wl.rope == "baked":
            ref = oracle.round_storage(oracle.rotate(k, pos[:, None], wl.rope_base), wl.dtype)
            # one bf16 ulp of the stored value, plus the fp32 rounding of the
            # rotation itself (it matters only where x1 cos - x2 sin cancels)
            half = wl.head_dim // 2
            pair = np.abs(k) + np.abs(np.concatenate([k[..., half:], k[..., :half]], axis=-1))
            tol = np.abs(ref) * 2.0 ** -7 + pair * 2.0 ** -21
            assert (np.abs(gk - ref) <= tol).all(), "baked K off by more than one bf16 ulp"
            assert (gk == ref).mean() > 0.99
        else:
            assert np.array_equal(gk, k), "read-time K must be stored raw"
    if wl.layout == "window":
        # slots no position has reached yet were never written
        for b in range(wl.batch):
            t = int(wl.positions[b])
            if t < wl.capacity:
                assert np.isnan(cache[:, b, :, t:]).all()


def test_bulk_append_keeps_only_survivors(kvc):
    """A bulk append longer than the window leaves the same cache as appending
    token by token ([ring] 3.3): later tokens win their slot."""
    wl = kvc_synth.make_workload("sink_window_bf16", small=True)
    d = bench.workload_desc(wl, layers=1)
    d.batch = 1
    n = 3 * wl.capacity + 17
    k, v = wl.kv_history(0, 0, np.arange(n))
    ws = kvc.alloc_workspace(d)
    c1 = kvc.alloc_cache(d, fill=float("nan"))
    kvc.append(d, c1, 0, k[None].cuda(), v[None].cuda(), torch.tensor([0], dtype=torch.int32, device="cuda"), ws)
    c2 = kvc.alloc_cache(d, fill=float("nan"))
    for p in range(n):
        kvc.append(d, c2, 0, k[p:p + 1][None].cuda(), v[p:p + 1][None].cuda(),
                   torch.tensor([p], dtype=torch.int32, device="cuda"), ws)
    torch.cuda.synchronize()
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))
    assert kvc.get_error(ws) == 0


# ---------------------------------------------------------------------------
# attended sets, bit-exact, through the decode kernel
# ---------------------------------------------------------------------------

def _probe_window(kvc, sinks, window, t, num_splits=0):
    C = sinks + window
    d = kvc.make_desc("sink_ring" if sinks else "ring", "none", "f32", 1, 1, 4, 1, 64, window=window,
                      sinks=sinks, num_splits=num_splits)
    cache = kvc.alloc_cache(d, fill=float("nan"))
    n_live = min(t + 1, C)
    cache[0, 0, 0, 0, :n_live] = 0.0                              # K = 0
    cache[0, 1, 0, 0, :n_live] = torch.eye(C, 64, device="cuda")[:n_live]   # V[slot] = e_slot
    ws = kvc.alloc_workspace(d)
    q = torch.randn(1, 4, 64, device="cuda")
    out = kvc.decode_attention(d, cache, 0, q, torch.tensor([t], dtype=torch.int32, device="cuda"), ws)
    return out[0].cpu().numpy()


@pytest.mark.parametrize("sinks,window", [(0, 64), (4, 60), (1, 31)])
def test_attended_set_window_bit_exact(kvc, sinks, window):
    C = sinks + window
    for t in (0, 1, 2, sinks, C - 2, C - 1, C, C + 1, 2 * C + 5, 10007, 123456):
        for ns in (0, 3):
            out = _probe_window(kvc, sinks, window, t, ns)
            A = oracle.window_attended(t, sinks, window)
            expect = np.zeros(64, dtype=np.float32)
            expect[oracle.window_slot(A, sinks, window)] = np.float32(1.0) / np.float32(len(A))
            for h in range(4):
                assert np.array_equal(out[h], expect), (sinks, window, t, ns)


def test_attended_set_paged_bit_exact(kvc):
    rng = np.random.default_rng(0)
    bs, nb, maxb, B = 4, 16, 12, 3
    d = kvc.make_desc("paged", "none", "f32", 1, B, 4, 1, 64, block_size=bs, num_blocks=nb,
                      max_blocks_per_seq=maxb)
    for trial in range(6):
        table = np.full((B, maxb), -1, dtype=np.int32)
        for b in range(B):
            phys = rng.permutation(nb)[:maxb]
            keep = rng.random(maxb) < 0.7
            table[b, keep] = phys[keep]
        valid = rng.random(nb) < 0.7
        pos = rng.integers(0, bs * maxb, size=B).astype(np.int32)
        cache = kvc.alloc_cache(d, fill=float("nan"))
        cache[0, 0] = 0.0
        cache[0, 1] = torch.eye(64, device="cuda").view(nb, 1, bs, 64)   # row (p, r) -> e_{4p + r}
        cache[0, :, torch.from_numpy(~valid).cuda()] = float("nan")
        ws = kvc.alloc_workspace(d)
        q = torch.randn(B, 4, 64, device="cuda")
        out = kvc.decode_attention(d, cache, 0, q, torch.from_numpy(pos).cuda(), ws,
                                   block_table=torch.from_numpy(table).cuda(),
                                   valid_bits=kvc.pack_valid_bits(torch.from_numpy(valid)).cuda())
        out = out.cpu().numpy()
        for b in range(B):
            A = oracle.paged_attended(int(pos[b]), table[b], valid, bs)
            expect = np.zeros(64, dtype=np.float32)
            if len(A):
                ids = table[b, A // bs] * bs + A % bs
                expect[ids] = np.float32(1.0) / np.float32(len(A))
            for h in range(4):
                assert np.array_equal(out[b, h], expect), (trial, b)
        assert kvc.get_error(ws) == 0


# ---------------------------------------------------------------------------
# decode outputs
# ---------------------------------------------------------------------------

def test_tiny_ring_sink_f32_all_256_steps(kvc):
    wl = kvc_synth.make_workload("tiny_ring_sink_f32")
    outs = run_stepwise(wl, steps=range(wl.steps))
    worst = 0.0
    for t, got in outs.items():
        ref = oracle_outputs(wl, 0, positions=np.array([t]))[0]
        worst = max(worst, _maxerr(got, ref))
    assert worst <= TOL["f32"], worst


def test_decode_step_f32_through_the_first_wrap(kvc):
    """kvc_decode_step on an fp32 cache (kvc_append, then the attention, on
    the same stream) from an empty cache past the first wrap of the window:
    outputs within the fp32 tolerance of the oracle at every step, and the
    cache bit-identical to one filled by kvc_append alone."""
    wl = kvc_synth.make_workload("tiny_ring_sink_f32")
    d = bench.workload_desc(wl, layers=1)
    cache = kvc.alloc_cache(d, fill=float("nan"))
    ref_cache = kvc.alloc_cache(d, fill=float("nan"))
    ws = kvc.alloc_workspace(d)
    worst = 0.0
    for t in range(72):
        k, v = wl.kv_history(0, 0, [t])                     # [1, kv_heads, D]
        k, v = k.contiguous().cuda(), v.contiguous().cuda()
        pos = torch.tensor([t], dtype=torch.int32, device="cuda")
        q = wl.query(0, 0, t)[None].contiguous().cuda()
        out = kvc.decode_step(d, cache, 0, q, k, v, pos, ws)
        kvc.append(d, ref_cache, 0, k[None], v[None], pos, ws)
        ref = oracle_outputs(wl, 0, positions=np.array([t]))[0]
        worst = max(worst, _maxerr(out[0].float().cpu().numpy(), ref))
    assert worst <= TOL["f32"], worst
    assert torch.equal(torch.nan_to_num(cache, nan=7.0), torch.nan_to_num(ref_cache, nan=7.0))
    assert kvc.get_error(ws) == 0


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("num_splits", [0, 1, 7])
def test_decode_small_elementwise(kvc, name, num_splits):
    wl = kvc_synth.make_workload(name, small=True)
    st = bench.DecodeState(wl, 1, source="cpu", num_splits=num_splits)
    got = st.step(0).float().cpu().numpy()
    ref = oracle_outputs(wl, 0)
    assert np.isfinite(got).all()
    err = _maxerr(got, ref)
    assert err <= TOL[wl.dtype], (name, num_splits, err)
    assert kvc.get_error(st.ws) == 0


@pytest.mark.parametrize("name,seqs,kw", [
    ("ring_bf16", [0, 5, 7], {}),
    ("sink_window_bf16", [0, 13, 31], {}),
    ("paged_shared_prefix_bf16", [0, 9, 40, 63], {}),
    ("long_context_pool_bf16", [0], {}),
    # the pool's valid-density sweep (0.25 and every slot valid)
    ("long_context_pool_bf16", [0], {"density": 0.25}),
    ("long_context_pool_bf16", [0], {"density": 1.0}),
])
def test_decode_full_size_sampled(kvc, name, seqs, kw):
    """Full workload sizes, bench.py's launch configuration, sampled sequences."""
    wl = kvc_synth.make_workload(name, **kw)
    st = bench.DecodeState(wl, 1, source="cpu")
    got = st.step(0).float().cpu().numpy()
    assert np.isfinite(got).all()
    ref = oracle_outputs(wl, 0, seqs=seqs)
    err = _maxerr(got[seqs], ref)
    assert err <= TOL[wl.dtype], (name, err)
    assert kvc.get_error(st.ws) == 0


@pytest.mark.parametrize("name", SMALL)
def test_decode_step_three_steps_and_cache(kvc, name):
    """kvc_decode_step (fused append for bf16 ring layouts) over three
    consecutive positions: outputs match the oracle, and the cache holds what
    the separate kvc_append writes (one bf16 ulp for RoPE baked into K)."""
    wl = kvc_synth.make_workload(name, small=True)
    st = bench.DecodeState(wl, 1, source="cpu")
    ref_cache = st.cache.clone()
    # paged: the next positions may need blocks the table does not map yet
    for step in range(3 if wl.layout == "window" else 1):
        pos = wl.positions + step
        q = wl.queries(0, pos).contiguous().cuda()
        kn, vn = wl.new_kv(0, pos)
        kn, vn = kn.contiguous().cuda(), vn.contiguous().cuda()
        pos_t = torch.from_numpy(pos.astype(np.int32)).cuda()
        out = kvc.decode_step(st.desc, st.cache, 0, q, kn, vn, pos_t, st.ws, block_table=st.table,
                              valid_bits=st.valid_bits)
        kvc.append(st.desc, ref_cache, 0, kn, vn, pos_t, st.ws, block_table=st.table)
        got = out.float().cpu().numpy()
        ref = oracle_outputs(wl, 0, positions=pos)
        assert np.isfinite(got).all()
        assert _maxerr(got, ref) <= TOL[wl.dtype], (name, step, _maxerr(got, ref))
        a, r = st.cache.float(), ref_cache.float()
        both_nan = torch.isnan(a) & torch.isnan(r)
        diff = (a - r).abs().masked_fill(both_nan, 0.0)
        assert (diff <= r.abs().masked_fill(both_nan, 0.0) * 2.0 ** -7 + 1e-6).all()
        assert (diff == 0).float().mean() > 0.999
    assert kvc.get_error(st.ws) == 0


def test_shared_prefix_outputs_depend_on_own_tail(kvc):
    """[share] 3.3: sequences sharing prefix blocks but with different tails
    must give different outputs (no cross-talk through the shared blocks)."""
    wl = kvc_synth.make_workload("paged_shared_prefix_bf16", small=True)
    st = bench.DecodeState(wl, 1, source="cpu")
    got = st.step(0).float().cpu().numpy()
    ref = oracle_outputs(wl, 0)
    for b in range(1, wl.batch):
        if wl.group[b] == wl.group[b - 1]:
            assert not np.allclose(got[b], got[b - 1])
    assert _maxerr(got, ref) <= TOL["bf16"]


# ---------------------------------------------------------------------------
# edge cases and device errors
# ---------------------------------------------------------------------------

def test_first_token_returns_its_value(kvc):
    d = kvc.make_desc("ring", "baked", "f32", 1, 2, 4, 2, 128, window=32)
    cache = kvc.alloc_cache(d, fill=float("nan"))
    ws = kvc.alloc_workspace(d)
    k = torch.randn(2, 1, 2, 128, device="cuda")
    v = torch.randn(2, 1, 2, 128, device="cuda")
    pos = torch.zeros(2, dtype=torch.int32, device="cuda")
    kvc.append(d, cache, 0, k, v, pos, ws)
    out = kvc.decode_attention(d, cache, 0, torch.randn(2, 4, 128, device="cuda"), pos, ws)
    expect = v[:, 0].repeat_interleave(2, dim=1)
    assert torch.equal(out, expect)


def test_fully_masked_sequence_gives_zeros(kvc):
    d = kvc.make_desc("paged", "baked", "bf16", 1, 2, 8, 2, 128, block_size=16, num_blocks=8,
                      max_blocks_per_seq=4)
    cache = kvc.alloc_cache(d, fill=1.0)
    ws = kvc.alloc_workspace(d)
    table = torch.tensor([[0, 1, 2, 3], [4, 5, -1, -1]], dtype=torch.int32, device="cuda")
    valid = torch.tensor([True, True, True, True, False, False, True, True])
    out = kvc.decode_attention(d, cache, 0, torch.randn(2, 8, 128, device="cuda").bfloat16(),
                               torch.tensor([50, 20], dtype=torch.int32, device="cuda"), ws,
                               block_table=table, valid_bits=kvc.pack_valid_bits(valid).cuda())
    assert torch.equal(out[1].float(), torch.zeros(8, 128, device="cuda"))
    assert torch.allclose(out[0].float(), torch.ones(8, 128, device="cuda"))


def test_device_errors_are_reported_not_faulted(kvc):
    d = kvc.make_desc("paged", "baked", "bf16", 1, 1, 4, 1, 128, block_size=16, num_blocks=4,
                      max_blocks_per_seq=4)
    cache = kvc.alloc_cache(d, fill=0.0)
    ws = kvc.alloc_workspace(d)
    # block id beyond the pool: skipped, KVC_DEV_BAD_BLOCK
    table = torch.tensor([[0, 9, 1, -1]], dtype=torch.int32, device="cuda")
    q = torch.randn(1, 4, 128, device="cuda").bfloat16()
    out = kvc.decode_attention(d, cache, 0, q, torch.tensor([40], dtype=torch.int32, device="cuda"), ws,
                               block_table=table)
    assert kvc.get_error(ws) == kvc.KVC_DEV_BAD_BLOCK
    assert torch.isfinite(out.float()).all()
    # append into an unmapped block: skipped, KVC_DEV_UNMAPPED_APPEND
    k = torch.randn(1, 1, 1, 128, device="cuda").bfloat16()
    kvc.append(d, cache, 0, k, k, torch.tensor([50], dtype=torch.int32, device="cuda"), ws, block_table=table)
    assert kvc.get_error(ws) == kvc.KVC_DEV_UNMAPPED_APPEND
    assert kvc.get_error(ws) == 0


def test_block_table_and_valid_writes(kvc):
    rng = np.random.default_rng(3)
    B, maxb, nb = 5, 9, 70
    d = kvc.make_desc("paged", "baked", "bf16", 1, B, 4, 1, 128, block_size=16, num_blocks=nb,
                      max_blocks_per_seq=maxb)
    ws = kvc.alloc_workspace(d)
    table = torch.full((B, maxb), -1, dtype=torch.int32, device="cuda")
    valid = torch.zeros((nb + 31) // 32, dtype=torch.int32, device="cuda")
    ref_t = np.full((B, maxb), -1)
    ref_v = np.zeros(nb, dtype=bool)
    idx = rng.permutation(B * maxb)[:30]
    seq, lb = (idx // maxb).astype(np.int32), (idx % maxb).astype(np.int32)
    phys = rng.integers(-1, nb, size=30).astype(np.int32)
    kvc.block_table_write(d, table, torch.from_numpy(seq).cuda(), torch.from_numpy(lb).cuda(),
                          torch.from_numpy(phys).cuda(), ws, valid_bits=valid)
    ref_t[seq, lb] = phys
    ref_v[phys[phys >= 0]] = True
    slots = rng.integers(0, nb, size=20).astype(np.int32)
    vals = (rng.random(20) < 0.5).astype(np.int32)
    # apply one value per slot (duplicate slots in one call would race)
    slots, first = np.unique(slots, return_index=True)
    vals = vals[first]
    kvc.valid_write(d, valid, torch.from_numpy(slots).cuda(), torch.from_numpy(vals).cuda(), ws)
    ref_v[slots] = vals.astype(bool)
    assert np.array_equal(table.cpu().numpy(), ref_t)
    w = valid.cpu().numpy().view(np.uint32)
    got_v = np.array([(w[k // 32] >> (k % 32)) & 1 for k in range(nb)], dtype=bool)
    assert np.array_equal(got_v, ref_v)
    # out-of-range entry: flagged, skipped
    kvc.block_table_write(d, table, torch.tensor([B], dtype=torch.int32, device="cuda"),
                          torch.tensor([0], dtype=torch.int32, device="cuda"),
                          torch.tensor([1], dtype=torch.int32, device="cuda"), ws)
    assert kvc.get_error(ws) == kvc.KVC_DEV_BAD_ENTRY
    assert np.array_equal(table.cpu().numpy(), ref_t)
