"""The pool pager's residency policy (kvc_pager_plan, host code) against a
plain Python model of its documented rules ([pool] "KV cache paging":
least-recently-used residency; blocks inside a sliding window pinned)."""

import numpy as np
import pytest

import sliding_window_attention_kvc_gb300 as kvc


class Model:
    def __init__(self, slots):
        self.block = [-1] * slots
        self.last = [-1] * slots
        self.pinned = [False] * slots
        self.step = 0

    def plan(self, need, pinned=None):
        S = len(self.block)
        where = {b: s for s, b in enumerate(self.block) if b >= 0}
        needed = {where[b] for b in need if b in where}
        missing = []
        for b in need:
            if b not in where and b not in missing:
                missing.append(b)
        keep = len(needed | {s for s in range(S) if self.block[s] >= 0 and self.pinned[s]})
        if keep + len(missing) > S:
            raise ValueError("does not fit")
        self.step += 1
        ins, outs = [], []
        for b in missing:
            free = [s for s in range(S) if self.block[s] < 0]
            if free:
                s = free[0]
            else:
                cand = [s for s in range(S) if s not in needed and not self.pinned[s]]
                s = min(cand, key=lambda x: (self.last[x], x))
                outs.append((self.block[s], s))
            self.block[s] = b
            self.pinned[s] = False
            needed.add(s)
            where[b] = s
            ins.append((b, s))
        for i, b in enumerate(need):
            s = where[b]
            self.last[s] = self.step
            if pinned is not None:
                self.pinned[s] = bool(pinned[i])
        return ins, outs


@pytest.fixture(scope="module")
def lib():
    return kvc.lib()


def test_lru_fixed_cases(lib):
    pg, m = kvc.Pager(3), Model(3)
    for need in ([0, 1], [2], [3], [1, 4], [0]):
        assert pg.plan(need) == m.plan(need)
    # the first plan fills free slots in order; [3] evicts block 0 (least recent)
    assert Model(3).plan([0, 1]) == ([(0, 0), (1, 1)], [])


def test_pinned_blocks_stay_until_unpinned(lib):
    pg, m = kvc.Pager(2), Model(2)
    assert pg.plan([7], [1]) == m.plan([7], [1])
    assert pg.plan([1]) == m.plan([1])
    got = pg.plan([2])                        # block 7 is pinned: block 1 goes
    assert got == m.plan([2]) and got[1] == [(1, 1)]
    assert pg.plan([7], [0]) == m.plan([7], [0])
    assert pg.plan([3]) == m.plan([3])
    with pytest.raises(kvc.KvcError):
        pg.plan([4, 5, 6])                    # more than the pool holds


def test_lru_random_steps_match_the_model(lib):
    rng = np.random.default_rng(3)
    for slots in (4, 16):
        pg, m = kvc.Pager(slots), Model(slots)
        for _ in range(300):
            n = int(rng.integers(1, slots + 1))
            need = rng.choice(3 * slots, size=n, replace=False).tolist()
            pinned = (rng.random(n) < 0.2).tolist()
            try:
                want = m.plan(need, pinned)
            except ValueError:
                with pytest.raises(kvc.KvcError):
                    pg.plan(need, pinned)
                continue
            assert pg.plan(need, pinned) == want


def test_pagein_issue_rejects_bad_entries_before_any_copy(lib):
    """A bad (block, slot) anywhere in the list is refused before any CUDA
    call, so no copy of the list's good entries is issued either."""
    import ctypes
    d = kvc.make_desc("paged", "baked", "bf16", 2, 1, 8, 2, 128, block_size=16, num_blocks=8,
                      max_blocks_per_seq=32)
    pg = kvc.Pager(8)
    A = 1 << 20                                   # fake addresses: never dereferenced on this path
    arr = ctypes.c_int32 * 2
    for blocks, slots in (([0, 32], [1, 2]), ([0, 3], [1, 8]), ([0, -1], [1, 2]), ([0, 3], [-1, 2])):
        rc = lib.kvc_pagein_issue(pg._p, ctypes.byref(d), A, A, 2, arr(*blocks), arr(*slots), None, None)
        assert rc == kvc.KVC_ERR_ARG, (blocks, slots, rc)
    d8 = kvc.make_desc("paged", "baked", "i8", 2, 1, 8, 2, 128, block_size=16, num_blocks=8, max_blocks_per_seq=32)
    assert lib.kvc_pagein_issue(pg._p, ctypes.byref(d8), A, A, 1, arr(0, 0), arr(1, 0), None, None) == \
        kvc.KVC_ERR_UNSUPPORTED
    pg.close()
