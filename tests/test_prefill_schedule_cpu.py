"""The tile schedule of the chunked-prefill kernels (prefill_tc_kernel: 128
(token, q head) rows per CTA; prefill_kernel: 64), restated on the CPU and
checked against the oracle's attended sets for window layouts.

Per CTA the kernels visit the sink keys [0, min(S, t_hi + 1)) and the window
keys [max(S, t_lo - W + 1), t_hi] in tiles of 64 keys, mask each key of a tile
per row (key inside the tile's range, p <= t, p a sink or p > t - W), and skip
the mask on interior tiles -- window tiles that lie inside every row's window
and below every row's position.  The keys a row keeps must be exactly
A(t) = oracle.window_attended(t, S, W), and every interior tile must need no
mask for any row of its CTA.
"""

import numpy as np
import pytest

import oracle

KEYS = 64


def _cta_keys(i0, tq, T, pos0, S, W, G):
    """{row -> kept keys} for one CTA of tq tokens from chunk index i0."""
    i_last = min(i0 + tq, T) - 1
    t_hi, t_lo = pos0 + i_last, max(pos0 + i0, 0)
    all_rows = pos0 + i0 >= 0 and i0 + tq <= T
    r0e = r1b = r1e = 0
    if i_last >= i0 and t_hi >= 0:
        r0e, r1b, r1e = min(S, t_hi + 1), max(S, t_lo - W + 1), t_hi + 1
    n0 = (r0e + KEYS - 1) // KEYS
    ntiles = n0 + ((r1e - r1b + KEYS - 1) // KEYS if r1e > r1b else 0)
    rows = [(i0 + tl, pos0 + i0 + tl) for tl in range(tq) if i0 + tl < T]
    kept = {i: set() for i, _ in rows}
    for k in range(ntiles):
        base = k * KEYS if k < n0 else r1b + (k - n0) * KEYS
        end = r0e if k < n0 else r1e
        interior = all_rows and k >= n0 and base + KEYS <= r1e and base + KEYS - 1 <= t_lo and base >= t_hi - W + 1
        for i, t in rows:
            for pk in range(base, base + KEYS):
                ok = 0 <= pk < end
                masked = ok and pk <= t and (pk < S or pk > t - W)
                if interior:
                    assert masked, (i0, k, pk, t)       # the shortcut must lose nothing
                if (interior and ok) or (not interior and masked):
                    kept[i].add(pk)
    return kept


@pytest.mark.parametrize("rows_per_cta", [128, 64])
def test_tile_schedule_keeps_exactly_the_attended_set(rows_per_cta):
    rng = np.random.default_rng(77)
    for _ in range(60):
        S = int(rng.choice([0, 1, 4]))
        W = int(rng.choice([1, 7, 60, 64, 100, 200]))
        G = int(rng.choice([1, 2, 3, 4, 6, 8]))
        T = int(rng.integers(1, 140))
        pos0 = int(rng.choice([-20, -1, 0, 3, 63, 64, 150, 4300]))
        tq = rows_per_cta // G
        for i0 in range(0, T, tq):
            kept = _cta_keys(i0, tq, T, pos0, S, W, G)
            for i, keys in kept.items():
                t = pos0 + i
                want = set(oracle.window_attended(t, S, W).tolist()) if t >= 0 else set()
                assert keys == want, (S, W, G, T, pos0, i0, i)


def _cta_keys_paged(i0, tq, T, pos0, table, valid, bs):
    """{row -> kept keys} for one CTA on a paged cache: keys [0, t_hi] in
    64-key tiles, a key kept when its block is mapped and valid (the row
    source) and, outside interior tiles, when p <= t."""
    i_last = min(i0 + tq, T) - 1
    t_hi, t_lo = pos0 + i_last, max(pos0 + i0, 0)
    all_rows = pos0 + i0 >= 0 and i0 + tq <= T
    r1e = t_hi + 1 if (i_last >= i0 and t_hi >= 0) else 0
    ntiles = (r1e + KEYS - 1) // KEYS
    rows = [(i0 + tl, pos0 + i0 + tl) for tl in range(tq) if i0 + tl < T]
    kept = {i: set() for i, _ in rows}
    for k in range(ntiles):
        base = k * KEYS
        interior = all_rows and base + KEYS <= r1e and base + KEYS - 1 <= t_lo
        for pk in range(base, base + KEYS):
            lb = pk // bs
            phys = table[lb] if (pk < r1e and lb < len(table)) else -1
            ok = phys >= 0 and bool(valid[phys])
            for i, t in rows:
                if interior:
                    assert not ok or pk <= t
                if ok and (interior or pk <= t):
                    kept[i].add(pk)
    return kept


@pytest.mark.parametrize("rows_per_cta", [128, 64])
def test_paged_tile_schedule_keeps_exactly_the_attended_set(rows_per_cta):
    rng = np.random.default_rng(78)
    for _ in range(40):
        bs = int(rng.choice([1, 16, 64]))
        nlog, nphys = 40, 48
        table = rng.permutation(nphys)[:nlog].astype(np.int64)
        table[rng.random(nlog) < 0.2] = -1                      # unmapped blocks
        valid = rng.random(nphys) < 0.7
        G = int(rng.choice([1, 2, 3, 4, 8]))
        T = int(rng.integers(1, 100))
        pos0 = int(rng.choice([-5, 0, 7, 64, 300]))
        pos0 = min(pos0, nlog * bs - T)                         # the chunk stays inside the table
        tq = rows_per_cta // G
        for i0 in range(0, T, tq):
            kept = _cta_keys_paged(i0, tq, T, pos0, table, valid, bs)
            for i, keys in kept.items():
                t = pos0 + i
                want = set(oracle.paged_attended(t, table, valid, bs).tolist()) if t >= 0 else set()
                assert keys == want, (bs, G, T, pos0, i0, i)
