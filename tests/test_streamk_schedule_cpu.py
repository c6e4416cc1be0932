"""The stream-K work split of the bf16 decode step, restated on the CPU.

Window layouts (the copy warp of decode_mma_kernel): sequence b counts
U_b = max(1, ceil(n_b / 16)) + 4 units (n_b = attended rows, 4 units charged
for a segment's start); all sequences' units are cut into G = min(total,
splits) shares [floor(x total / G), floor((x + 1) total / G)); the part of
share x inside sequence b is one segment, which writes partial slot x + b and
streams the rows of its units past the 4 charged ones.  The combine of
sequence b merges slots fx + b .. lx + b, fx and lx the shares of its first
and last unit.

Paged layouts (plan_count_kernel / plan_items_kernel): rows, not units, are
cut into G = min(R, CTAs) shares (at least one); the part of share x inside
sequence b is work item x + b, and a sequence with no rows gets one empty
item.

Checked for random batches: every share non-empty, every sequence's rows
covered exactly once, a sequence's segments are exactly the shares it
overlaps, and slots are unique and below G + B (the workspace's partial and
item arrays).
"""

import numpy as np
import pytest

SEQ_UNITS = 4


def share_of(u, total, G):
    return ((u + 1) * G - 1) // total


def window_split(nl, splits):
    st = [(n + 15) // 16 if n > 0 else 1 for n in nl]
    st = [s + SEQ_UNITS for s in st]
    total = sum(st)
    G = min(total, splits)
    off = np.concatenate([[0], np.cumsum(st)]).tolist()
    segs = []                                      # (share, b, r0, r1)
    for x in range(G):
        lo, hi = x * total // G, (x + 1) * total // G
        assert hi > lo
        for b in range(len(nl)):
            Ob, Sb = off[b], st[b]
            if Ob >= hi or Ob + Sb <= lo:
                continue
            u0, u1 = max(lo, Ob) - Ob, min(hi, Ob + Sb) - Ob
            r0 = max(0, u0 - SEQ_UNITS) * 16
            r1 = min(max(0, u1 - SEQ_UNITS) * 16, nl[b])
            segs.append((x, b, r0, r1))
    firsts = [(share_of(off[b], total, G), share_of(off[b] + st[b] - 1, total, G)) for b in range(len(nl))]
    return G, segs, firsts


def paged_split(rows, ctas):
    R = sum(rows)
    G = (R if R > 0 else 1) if R < ctas else ctas
    off = np.concatenate([[0], np.cumsum(rows)]).tolist()
    items = []                                     # (share, b, s0, s1): sequence-local rows
    firsts = []
    for b, Rb in enumerate(rows):
        Ob = off[b]
        if Rb > 0:
            fx, lx = share_of(Ob, R, G), share_of(Ob + Rb - 1, R, G)
            for x in range(fx, lx + 1):
                lo, hi = x * R // G, (x + 1) * R // G
                s0, s1 = max(lo, Ob) - Ob, min(hi, Ob + Rb) - Ob
                assert s1 > s0
                items.append((x, b, s0, s1))
        else:
            fx = lx = share_of(min(Ob, R - 1), R, G) if R > 0 else 0
            items.append((fx, b, 0, 0))
        firsts.append((fx, lx))
    return G, items, firsts


def _check(B, G, parts, firsts, lengths):
    slots = [x + b for x, b, _, _ in parts]
    assert len(set(slots)) == len(slots) and max(slots) < G + B and min(slots) >= 0
    for b in range(B):
        mine = sorted((x, r0, r1) for x, bb, r0, r1 in parts if bb == b)
        fx, lx = firsts[b]
        assert [x for x, _, _ in mine] == list(range(fx, lx + 1))       # the combine's slot range
        covered = [(r0, r1) for _, r0, r1 in mine if r1 > r0]
        pos = 0
        for r0, r1 in covered:                                          # contiguous, in order, once
            assert r0 == pos
            pos = r1
        assert pos == lengths[b]


@pytest.mark.parametrize("seed", range(6))
def test_window_split_covers_every_row_once(seed):
    rng = np.random.default_rng(seed)
    for _ in range(80):
        B = int(rng.integers(1, 70))
        C = int(rng.choice([1, 15, 16, 64, 200, 4096]))
        t = rng.integers(-3, 3 * C + 2, size=B)
        t[rng.random(B) < 0.2] = -1                                     # empty sequences
        nl = [0 if tb < 0 else min(int(tb) + 1, C) for tb in t]
        splits = int(rng.choice([1, 2, 7, 152, 304, 1000]))
        G, segs, firsts = window_split(nl, splits)
        _check(B, G, segs, firsts, nl)


@pytest.mark.parametrize("seed", range(6))
def test_paged_plan_covers_every_row_once(seed):
    rng = np.random.default_rng(100 + seed)
    for _ in range(80):
        B = int(rng.integers(1, 70))
        rows = rng.integers(0, 3000, size=B).tolist()
        if rng.random() < 0.3:
            rows = [r if rng.random() < 0.5 else 0 for r in rows]      # fully masked sequences
        ctas = int(rng.choice([1, 3, 152, 304, 456]))
        G, items, firsts = paged_split(rows, ctas)
        _check(B, G, items, firsts, rows)
