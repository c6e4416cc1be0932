"""Attended sets, bit-exact, through the kernels that run the bf16 and INT8
workloads (tensor-core decode with its copy-warp runs, ring-wrap and
sink/window cuts, stream-K shares and paged work plan; the fused append of
kvc_decode_step; the chunked-prefill kernels' per-tile masks).

The probe (tests/attended_probe.py) gives every attended row the same weight
and one-hot V rows by id slice, with NaN in every row outside the attended
sets, so each output entry is exactly unit(|A|) or 0 and the passes recover
each sequence's attended set exactly.  Expected sets: the oracle's closed
forms for the ring ([ring] 2.2, 3.1, 6: A(t) = {t-W+1 .. t}), the sink cache
([sink] cache-set equation: {0 .. S-1} U window) and the paged cache ([pool]
"kernel forgets absent blocks": mapped and valid blocks only).
"""

import numpy as np
import pytest
import torch

import kvc_synth
import oracle
from tests.attended_probe import NAN, Probe, paged_probe, run_decode, unit, window_probe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import sliding_window_attention_kvc_gb300 as m
    return m


def _positions(S, C):
    # before, at and after the sinks, the first wrap, and far past it
    return [0, 1, S, C - 2, C - 1, C, C + 1, 2 * C + 5, 987654]


# geometry per head_dim: (q heads, kv heads, window of a ring); D 128 is the
# statement's ring / sink shape (32 q / 8 kv heads, 4096 slots)
GEOM = {64: (8, 2, 512), 128: (32, 8, 4096), 256: (16, 4, 1024)}
WINDOW_CASES = [("bf16", 64), ("bf16", 128), ("bf16", 256), ("i8", 128), ("i8", 256)]


@pytest.mark.parametrize("dtype,D", WINDOW_CASES)
@pytest.mark.parametrize("sinks", [0, 4])
@pytest.mark.parametrize("num_splits", [0, 1, 7])
@pytest.mark.parametrize("fused", [False, True])
def test_window_attended_sets_exact(kvc, dtype, D, sinks, num_splits, fused):
    Hq, Hkv, C = GEOM[D]
    W = C - sinks
    t = _positions(sinks, C)
    p = window_probe(kvc, dtype=dtype, B=len(t), Hq=Hq, Hkv=Hkv, D=D, sinks=sinks, window=W, t=t,
                     num_splits=num_splits, fused=fused)
    run_decode(kvc, p, t)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("i8", 128), ("i8", 256)])
@pytest.mark.parametrize("sinks", [0, 4])
@pytest.mark.parametrize("num_splits,fused", [(0, False), (0, True), (7, False), (7, True)])
def test_window_read_time_sets_exact(kvc, dtype, D, sinks, num_splits, fused):
    """Read-time RoPE ([sink] "RoPE cache position shifting"): the rotating
    paths (bf16 rows rotated in place, INT8 rows dequantised and rotated into
    a bf16 tile) see exactly the attended sets."""
    Hq, Hkv, C = GEOM[D]
    W = C - sinks
    t = _positions(sinks, C)
    p = window_probe(kvc, dtype=dtype, B=len(t), Hq=Hq, Hkv=Hkv, D=D, sinks=sinks, window=W, t=t,
                     num_splits=num_splits, fused=fused, rope="read_time")
    run_decode(kvc, p, t)


@pytest.mark.parametrize("name", ["ring_bf16", "sink_window_bf16", "ring_int8", "sink_window_int8"])
@pytest.mark.parametrize("num_splits,fused", [(0, False), (0, True), (1, False), (7, True)])
def test_window_workload_sets_exact(kvc, name, num_splits, fused):
    """The full workload shapes, positions and RoPE modes (bench.py's launch
    configuration at num_splits 0)."""
    wl = kvc_synth.make_workload(name)
    t = wl.positions
    p = window_probe(kvc, dtype=wl.dtype, B=wl.batch, Hq=wl.q_heads, Hkv=wl.kv_heads, D=wl.head_dim,
                     sinks=wl.sinks, window=wl.window, t=t, num_splits=num_splits, fused=fused, rope=wl.rope)
    run_decode(kvc, p, t)


def _random_paged(rng, B, bs, maxb, nb, share=True, empty=True, p_valid=0.75):
    """A block table with a shared prefix (sequences 0..2 map the same first
    blocks), random private blocks, unmapped holes, invalid slots, and (empty)
    one sequence whose every block is unmapped or invalid."""
    perm = rng.permutation(nb)
    table = np.full((B, maxb), -1, dtype=np.int32)
    nxt = 0
    pre = 3
    prefix = perm[nxt:nxt + pre]
    nxt += pre
    for b in range(B):
        n = maxb
        own = perm[nxt:nxt + n]
        nxt += n
        table[b] = own
        if share and b < 3:
            table[b, :pre] = prefix
        holes = rng.random(maxb) < 0.15
        holes[:pre] = False
        table[b, holes] = -1
    valid = rng.random(nb) < p_valid
    valid[prefix] = True
    t = rng.integers(0, bs * maxb, size=B)
    t[0] = bs * pre - 1                  # on the last row of the shared prefix
    t[1] = bs * pre                      # first row after it
    if empty:
        valid[table[B - 1][table[B - 1] >= 0]] = False
    return table, valid, t


@pytest.mark.parametrize("dtype,D,bs", [("bf16", 128, 16), ("bf16", 256, 64), ("bf16", 64, 16),
                                        ("i8", 128, 16), ("i8", 256, 64)])
@pytest.mark.parametrize("num_splits", [0, 1, 7])
def test_paged_attended_sets_exact(kvc, dtype, D, bs, num_splits):
    rng = np.random.default_rng(11 + D + bs + num_splits)
    Hq, Hkv, _ = GEOM[D]
    B, maxb = 9, 12
    nb = 3 + B * maxb + 5
    table, valid, t = _random_paged(rng, B, bs, maxb, nb)
    t[B - 2] = -1                        # no position: nothing attended, zeros
    p = paged_probe(kvc, dtype=dtype, Hq=Hq, Hkv=Hkv, D=D, bs=bs, num_blocks=nb, table=table, valid=valid, t=t,
                    num_splits=num_splits, fused=False)
    # t < 0 sets the bad-position bit; everything else must be exact
    d = p.d
    ws = kvc.alloc_workspace(d)
    pos = torch.from_numpy(t.astype(np.int32)).cuda()
    q = torch.randn((B, Hq, D), generator=torch.Generator().manual_seed(3)).bfloat16().cuda()
    for ps in range(p.passes):
        p.fill(ps)
        out = kvc.decode_attention(d, p.cache, 0, q, pos, ws, block_table=p.table, valid_bits=p.valid_bits)
        p.compare(out, ps, f"paged pass {ps}")
    assert kvc.get_error(ws) == kvc.KVC_DEV_BAD_POSITION


@pytest.mark.parametrize("dtype,D,bs", [("bf16", 128, 16), ("bf16", 256, 64), ("i8", 128, 16)])
@pytest.mark.parametrize("num_splits", [0, 7])
def test_paged_decode_step_sets_exact(kvc, dtype, D, bs, num_splits):
    """kvc_decode_step: the plan kernel appends each sequence's token, the
    decode kernel must attend it (its row is NaN before the call)."""
    rng = np.random.default_rng(5 + D + num_splits)
    Hq, Hkv, _ = GEOM[D]
    B, maxb = 8, 10
    nb = 3 + B * maxb + 5
    table, valid, t = _random_paged(rng, B, bs, maxb, nb, share=False, empty=False)
    for b in range(B):                   # the new token's block: mapped and resident
        if table[b, t[b] // bs] < 0:
            t[b] = int(np.flatnonzero(table[b] >= 0)[-1]) * bs + bs // 2
        valid[table[b, t[b] // bs]] = True
    p = paged_probe(kvc, dtype=dtype, Hq=Hq, Hkv=Hkv, D=D, bs=bs, num_blocks=nb, table=table, valid=valid, t=t,
                    num_splits=num_splits, fused=True)
    run_decode(kvc, p, t)


@pytest.mark.parametrize("name,kw,num_splits,fused", [
    ("paged_shared_prefix_bf16", {}, 0, False),
    ("paged_shared_prefix_bf16", {}, 0, True),
    ("paged_shared_prefix_bf16", {}, 7, False),
    ("paged_shared_prefix_int8", {}, 0, False),
    ("paged_shared_prefix_int8", {}, 1, True),
    ("long_context_pool_bf16", {}, 0, False),
    ("long_context_pool_bf16", {}, 0, True),
    ("long_context_pool_bf16", {}, 7, False),
    ("long_context_pool_bf16", {"density": 0.25}, 0, False),
    ("long_context_pool_bf16", {"density": 1.0}, 1, False),
])
def test_paged_workload_sets_exact(kvc, name, kw, num_splits, fused):
    """The full paged workloads: shared-prefix tables (ids = positions, shared
    rows sit at one position in every sequence of a group) and the 256K pool
    with its valid mask (ids = row ranks)."""
    wl = kvc_synth.make_workload(name, **kw)
    mode = "rank" if wl.batch == 1 else "position"
    p = paged_probe(kvc, dtype=wl.dtype, Hq=wl.q_heads, Hkv=wl.kv_heads, D=wl.head_dim, bs=wl.block_size,
                    num_blocks=wl.num_blocks, table=wl.block_table, valid=wl.valid, t=wl.positions,
                    num_splits=num_splits, fused=fused, id_mode=mode)
    run_decode(kvc, p, wl.positions)


def test_probe_reports_a_planted_missing_row(kvc):
    """The probe itself: an attended row missing from the expected set
    (a mistake planted on the host side) is reported."""
    t = [5000]
    p = window_probe(kvc, dtype="bf16", B=1, Hq=8, Hkv=2, D=128, sinks=0, window=256, t=t)
    p.sets = [p.sets[0][1:]]             # drop one attended slot from the expectation
    with pytest.raises(AssertionError):
        run_decode(kvc, p, t)
    assert unit(4096, "bf16") == float(torch.tensor(1.0 / 4096))
    assert not np.isnan(unit(3, "i8"))


# ---------------------------------------------------------------------------
# chunked prefill: per-tile causal, window, sink and mask edges
# ---------------------------------------------------------------------------

def _prefill_probe(kvc, d, cache, sets_of, cached_rows, chunk_id, B, T):
    """Probe over a prefill call: `sets_of[b][i]` the ids chunk token i of
    sequence b attends, `cached_rows` the ids of cache rows (X, R) live before
    the call, chunk_id [B, T] the ids of the chunk's own rows (-1: padding)."""
    sets = [sets_of[b][i] for b in range(B) for i in range(T)]
    p = Probe(kvc, d, cache, cached_rows, sets)
    p.chunk_id = chunk_id
    return p


def _run_prefill(kvc, p, pos0, T, table=None, valid_bits=None):
    d = p.d
    B, Hq, Hkv, D = d.batch, d.q_heads, d.kv_heads, d.head_dim
    ws = kvc.alloc_prefill_workspace(d, T)
    q = torch.randn((B, T, Hq, D), generator=torch.Generator().manual_seed(9)).bfloat16().cuda()
    k = torch.zeros((B, T, Hkv, D), dtype=torch.bfloat16, device="cuda")
    pos = torch.from_numpy(np.asarray(pos0, dtype=np.int32)).cuda()
    # the chunk's one-hot V: 127/128 on an INT8 cache, which stores it as the
    # code 127 of scale 2^-7 and reads it back exactly, like the cached rows
    one = 127.0 / 128.0 if p.dtype == "i8" else 1.0
    for ps in range(p.passes):
        p.fill(ps)
        v = torch.zeros((B, T, Hkv, D), dtype=torch.bfloat16)
        for b in range(B):
            for i in range(T):
                e = int(p.chunk_id[b, i])
                if e < 0:
                    continue
                h = e // D - ps * Hkv
                if 0 <= h < Hkv:
                    v[b, i, h, e % D] = one
        out = kvc.prefill(d, p.cache, 0, q, k, v.cuda(), pos, ws, block_table=table, valid_bits=valid_bits)
        p.compare(out.view(B * T, Hq, D), ps, f"prefill pass {ps}")
    assert kvc.get_error(ws) == 0


@pytest.mark.parametrize("D,rope,sinks,dtype", [(128, "baked", 0, "bf16"), (128, "read_time", 4, "bf16"),
                                                (64, "none", 0, "bf16"), (64, "read_time", 4, "bf16"),
                                                (256, "baked", 0, "bf16"), (256, "read_time", 4, "bf16"),
                                                (128, "baked", 0, "i8"), (128, "read_time", 4, "i8"),
                                                (256, "read_time", 4, "i8")])
def test_prefill_window_sets_exact(kvc, D, rope, sinks, dtype):
    """Ring and sink+ring chunks before, across and far past the first wrap,
    with left padding; ids: sinks keep their position, window positions count
    from the oldest one any chunk token can see."""
    Hq, Hkv, C = GEOM[D]
    W = C - sinks
    T = 128
    pos0 = np.array([-5, 0, 100, C - 64, C + 3, 3 * C + 77, 987654 - T], dtype=np.int64)
    B = len(pos0)
    d = kvc.make_desc("sink_ring" if sinks else "ring", rope, dtype, 1, B, Hq, Hkv, D, window=W, sinks=sinks)
    cache = kvc.alloc_cache(d, fill=NAN)
    ids = np.full((B, C), -1, dtype=np.int64)
    chunk_id = np.full((B, T), -1, dtype=np.int64)
    sets_of = []
    for b in range(B):
        base = max(sinks, int(pos0[b]) - W)

        def idp(p):
            p = np.asarray(p, dtype=np.int64)
            return np.where(p < sinks, p, sinks + (p - base))
        row_sets, cached = [], set()
        for i in range(T):
            t = int(pos0[b]) + i
            if t < 0:
                row_sets.append(np.zeros(0, np.int64))
                continue
            A = oracle.window_attended(t, sinks, W)
            row_sets.append(idp(A))
            cached |= set(A[A < pos0[b]].tolist())
            chunk_id[b, i] = int(idp(t))
        sets_of.append(row_sets)
        if cached:
            cp = np.array(sorted(cached), dtype=np.int64)
            ids[b, oracle.window_slot(cp, sinks, W)] = idp(cp)
    p = _prefill_probe(kvc, d, cache, sets_of, ids, chunk_id, B, T)
    _run_prefill(kvc, p, pos0, T)


@pytest.mark.parametrize("D,bs,dtype", [(128, 16, "bf16"), (64, 16, "bf16"), (256, 64, "bf16"), (128, 32, "bf16"),
                                        (128, 16, "i8"), (256, 64, "i8")])
def test_prefill_paged_sets_exact(kvc, D, bs, dtype):
    """Paged chunks over a table with a shared prefix, holes and invalid
    blocks; the chunk's own blocks mapped and resident; ids = positions."""
    rng = np.random.default_rng(21 + D + bs)
    Hq, Hkv, _ = GEOM[D]
    B, maxb, T = 6, 24 * 16 // bs, 96
    nb = 3 + B * maxb + B * (T // bs + 2)   # room for private blocks under the chunks
    table, valid, _ = _random_paged(rng, B, bs, maxb, nb, share=True, empty=False)
    pos0 = np.array([-7, 0, 5, 40, 150, bs * maxb - T], dtype=np.int64)
    # every block a chunk writes: mapped, private to its sequence, resident
    used = set(int(x) for x in table[table >= 0].ravel())
    free = [x for x in range(nb) if x not in used]
    for b in range(B):
        for lb in range(max(0, pos0[b]) // bs, (pos0[b] + T - 1) // bs + 1):
            shared = b < 3 and lb < 3
            if table[b, lb] < 0 or shared:
                table[b, lb] = free.pop()
            valid[table[b, lb]] = True
    d = kvc.make_desc("paged", "baked", dtype, 1, B, Hq, Hkv, D, block_size=bs, num_blocks=nb,
                      max_blocks_per_seq=maxb)
    cache = kvc.alloc_cache(d, fill=NAN)
    ids = np.full((nb, bs), -1, dtype=np.int64)
    chunk_id = np.full((B, T), -1, dtype=np.int64)
    sets_of = []
    for b in range(B):
        row_sets = []
        for i in range(T):
            t = int(pos0[b]) + i
            if t < 0:
                row_sets.append(np.zeros(0, np.int64))
                continue
            A = oracle.paged_attended(t, table[b], valid, bs)
            row_sets.append(A)
            chunk_id[b, i] = t
            old = A[A < pos0[b]]
            ph, r = table[b, old // bs], old % bs
            assert ((ids[ph, r] < 0) | (ids[ph, r] == old)).all()
            ids[ph, r] = old
        sets_of.append(row_sets)
    p = _prefill_probe(kvc, d, cache, sets_of, ids, chunk_id, B, T)
    _run_prefill(kvc, p, pos0, T, table=torch.from_numpy(table).cuda(),
                 valid_bits=kvc.pack_valid_bits(torch.from_numpy(valid)).cuda())


def test_prefill_full_paged_workload_sets_exact(kvc):
    """The full shared-prefix batch: 64 chunks of 128 tokens ending at each t_b
    (bench.py's prefill case), ids = positions."""
    wl = kvc_synth.make_workload("paged_shared_prefix_bf16")
    B, T, bs = wl.batch, 128, wl.block_size
    pos0 = np.maximum(wl.positions - T + 1, 0)
    table, valid = wl.block_table, wl.valid
    d = kvc.make_desc("paged", "baked", "bf16", 1, B, wl.q_heads, wl.kv_heads, wl.head_dim, block_size=bs,
                      num_blocks=wl.num_blocks, max_blocks_per_seq=wl.max_blocks_per_seq)
    cache = kvc.alloc_cache(d, fill=NAN)
    ids = np.full((wl.num_blocks, bs), -1, dtype=np.int64)
    chunk_id = np.full((B, T), -1, dtype=np.int64)
    sets_of = []
    for b in range(B):
        tb = int(wl.positions[b])
        A_last = oracle.paged_attended(tb, table[b], valid, bs)
        assert pos0[b] + T - 1 == tb         # every length is >= T: the chunk ends at t_b
        row_sets = []
        for i in range(T):
            t = int(pos0[b]) + i
            row_sets.append(A_last[A_last <= t])
            chunk_id[b, i] = t
        old = A_last[A_last < pos0[b]]
        ids[table[b, old // bs], old % bs] = old
        sets_of.append(row_sets)
    p = _prefill_probe(kvc, d, cache, sets_of, ids, chunk_id, B, T)
    _run_prefill(kvc, p, pos0, T, table=torch.from_numpy(table).cuda())


@pytest.mark.parametrize("num_splits,fused", [(0, False), (0, True), (7, False)])
def test_paged_batch_over_64_sequences_sets_exact(kvc, num_splits, fused):
    """A batch of more sequences than the decode CTAs keep rows for in
    registers (64): the rest are reloaded per 32 when a CTA cuts its shares;
    shared prefix, holes, invalid slots and an empty sequence as above."""
    rng = np.random.default_rng(41)
    B, bs, maxb = 70, 16, 64
    nb = 3 + B * maxb
    table, valid, t = _random_paged(rng, B, bs, maxb, nb, share=not fused, empty=not fused)
    if fused:
        for b in range(B):               # the new token's block: mapped and resident
            if table[b, t[b] // bs] < 0:
                t[b] = int(np.flatnonzero(table[b] >= 0)[-1]) * bs + bs // 2
            valid[table[b, t[b] // bs]] = True
    p = paged_probe(kvc, dtype="bf16", Hq=8, Hkv=2, D=128, bs=bs, num_blocks=nb, table=table, valid=valid, t=t,
                    num_splits=num_splits, fused=fused)
    run_decode(kvc, p, t)


def test_paged_one_sequence_long_table_sets_exact(kvc):
    """One sequence whose table has more entries than the decode CTAs plan
    themselves (the plan kernel's single-sequence path): ids = row ranks."""
    rng = np.random.default_rng(31)
    bs, maxb, nb = 16, 6000, 300
    table = np.full((1, maxb), -1, dtype=np.int32)
    t = 95000
    lbs = np.sort(rng.choice(t // bs, size=nb - 1, replace=False))
    slots = rng.permutation(nb)
    table[0, lbs] = slots[:-1]
    table[0, t // bs] = slots[-1]
    valid = rng.random(nb) < 0.6
    valid[slots[-1]] = True
    for fused in (False, True):
        p = paged_probe(kvc, dtype="bf16", Hq=8, Hkv=2, D=128, bs=bs, num_blocks=nb, table=table, valid=valid,
                        t=[t], fused=fused)
        run_decode(kvc, p, [t])


@pytest.mark.parametrize("dtype", ["bf16", "i8"])
def test_one_sequence_step_writes_a_token_whose_block_is_not_resident(kvc, dtype):
    """kvc_decode_step on one paged sequence whose new token's block is mapped
    but not valid: the token is written (as kvc_append writes it) and not
    attended; an unmapped block sets KVC_DEV_UNMAPPED_APPEND."""
    D, Hq, Hkv, bs, nb = 128, 8, 2, 16, 8
    d = kvc.make_desc("paged", "baked", dtype, 1, 1, Hq, Hkv, D, block_size=bs, num_blocks=nb,
                      max_blocks_per_seq=nb)
    g = torch.Generator().manual_seed(4)
    table = torch.from_numpy(np.array([[5, 2, 7, 0, 1, 3, 6, 4]], dtype=np.int32)).cuda()
    t = 50                                    # logical block 3 -> physical block 0
    valid = np.ones(nb, dtype=bool)
    valid[0] = False
    vb = kvc.pack_valid_bits(torch.from_numpy(valid)).cuda()
    ws = kvc.alloc_workspace(d)
    cache = kvc.alloc_cache(d, fill=0.0)
    k = torch.randn((1, t, Hkv, D), generator=g).bfloat16().cuda()
    v = torch.randn((1, t, Hkv, D), generator=g).bfloat16().cuda()
    kvc.append(d, cache, 0, k, v, torch.tensor([0], dtype=torch.int32, device="cuda"), ws, block_table=table)
    ref = cache.clone()
    q = torch.randn((1, Hq, D), generator=g).bfloat16().cuda()
    kn = torch.randn((1, Hkv, D), generator=g).bfloat16().cuda()
    vn = torch.randn((1, Hkv, D), generator=g).bfloat16().cuda()
    pos = torch.tensor([t], dtype=torch.int32, device="cuda")
    out = kvc.decode_step(d, cache, 0, q, kn, vn, pos, ws, block_table=table, valid_bits=vb)
    kvc.append(d, ref, 0, kn[:, None], vn[:, None], pos, ws, block_table=table)
    want = kvc.decode_attention(d, ref, 0, q, pos, ws, block_table=table, valid_bits=vb)
    torch.cuda.synchronize()
    assert torch.equal(cache, ref), "the token's rows differ from kvc_append's"
    assert torch.equal(out, want)
    assert kvc.get_error(ws) == 0
    # the block of the next token unmapped: reported, nothing written
    table2 = table.clone()
    table2[0, 3] = -1
    kvc.decode_step(d, cache, 0, q, kn, vn, pos, ws, block_table=table2, valid_bits=vb)
    assert kvc.get_error(ws) == kvc.KVC_DEV_UNMAPPED_APPEND
