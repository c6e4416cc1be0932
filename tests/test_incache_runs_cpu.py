"""Read-time RoPE positions in the bf16 decode step's copy warp, restated on
the CPU.

The copy warp cuts a segment's slots [r0, r1) into runs of at most 16 x (free
stages) rows that never straddle the sink/window boundary or the ring's wrap
(the slot of the token being decoded).  Each run carries the in-cache position
of its first slot, computed exactly at a segment start, at those boundaries,
after a partial run and every 32 runs, and otherwise carried on from the
previous run (position + rows).  Rows of a run take consecutive positions.

Checked for random t, S, W and cuts: every row's position equals the oracle's
in-cache position ([sink] "RoPE cache position shifting") of the token its
slot holds, and no run crosses a boundary.
"""

import numpy as np
import pytest

import oracle


def incache_of_slot(s, t, S, W, C):
    if s < S:
        return s
    p = t - ((t - s) % W)
    shift = t - C + 1
    return p - shift if shift > 0 else p


def runs(r0, r1, t, S, W, rooms):
    C = S + W
    h_slot = t if t < S else S + (t - S) % W
    out, ip_next, prev_n, since, r, k = [], 0, 0, 0, r0, 0
    while r < r1:
        n = min(16 * rooms[k % len(rooms)], r1 - r)
        k += 1
        seg_end = S if r < S else (h_slot + 1 if r <= h_slot else C)
        n = min(n, seg_end - r)
        exact = r == r0 or r == S or r == h_slot + 1 or (prev_n & 15) != 0 or since >= 32
        if exact:
            ip0, since = incache_of_slot(r, t, S, W, C), 0
        else:
            ip0 = ip_next
        since += 1
        ip_next, prev_n = ip0 + n, n
        out.append((r, n, ip0))
        r += n
    return out, h_slot


@pytest.mark.parametrize("seed", range(5))
def test_run_positions_match_the_oracle(seed):
    rng = np.random.default_rng(seed)
    for _ in range(150):
        S = int(rng.choice([1, 4, 7]))
        W = int(rng.choice([5, 60, 100, 4092]))
        C = S + W
        t = int(rng.choice([int(rng.integers(0, C)), int(rng.integers(C, 50 * C))]))
        nl = min(t + 1, C)
        r0 = int(rng.integers(0, nl))
        r1 = int(rng.integers(r0 + 1, nl + 1))
        rooms = rng.integers(1, 7, size=int(rng.integers(1, 5))).tolist()
        out, h_slot = runs(r0, r1, t, S, W, rooms)
        assert out[0][0] == r0 and sum(n for _, n, _ in out) == r1 - r0
        for r, n, ip0 in out:
            assert n >= 1
            assert not (r < S < r + n) and not (r <= h_slot < r + n - 1)     # no boundary inside a run
            for j in range(n):
                s = r + j
                p = s if s < S else t - ((t - s) % W)                          # the token slot s holds
                assert ip0 + j == oracle.incache_position(p, t, S, W), (S, W, t, s)
