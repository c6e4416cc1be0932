"""Pins for oracle.blocks (the paged cache's block manager) against what the
[share] page fixes: copy-on-write before writing into a shared block (§3.2,
§5.1), reference counts raised by prefix sharing and dropped on release,
reclaim only at zero (§6.1), and sharing that never lets one sequence's
write reach another (§3.2's bug, §7)."""

import numpy as np
import pytest

from oracle import blocks
from oracle.blocks import BlockManager


class Pool:
    """Contents of the physical blocks: token ids, -1 = empty."""

    def __init__(self, num_blocks, bs):
        self.rows = np.full((num_blocks, bs), -1, dtype=np.int64)

    def copy(self, src, dst, n):
        self.rows[dst, :n] = self.rows[src, :n]


def step(bm, pool, hist, positions, token_of):
    """One decode step: prepare, then write each sequence's new token."""
    bm.prepare(positions, copy=pool.copy)
    for b, t in enumerate(positions):
        if t < 0:
            continue
        phys = bm.table[b, t // bm.bs]
        if phys >= 0:
            pool.rows[phys, t % bm.bs] = token_of(b, t)
            hist[b][t] = token_of(b, t)


def visible(bm, pool, b, t):
    out = {}
    for p in range(t + 1):
        phys = bm.table[b, p // bm.bs]
        if phys >= 0:
            out[p] = int(pool.rows[phys, p % bm.bs])
    return out


def _worked_scenario(cls):
    # block size 4, pool of 8; sequence 0 writes 6 tokens, sequence 1 takes
    # its 6-token prefix (2 blocks), then both write token 6 into the shared,
    # partly filled second block
    bm, pool = cls(8, 4, batch=2, max_blocks=4), Pool(8, 4)
    hist = [{}, {}]
    for t in range(6):
        step(bm, pool, hist, [t, -1], lambda b, p: 100 * b + p)
    assert bm.table[0, :2].tolist() == [7, 6]          # stack: top first
    bm.share(src=0, dst=1, nblocks=2)
    for p in range(6):
        hist[1][p] = hist[0][p]
    assert bm.ref[[7, 6]].tolist() == [2, 2]
    copies = bm.prepare([6, 6], copy=pool.copy)
    # sequence 0 is served first and copies (count 2 > 1); sequence 1 then
    # sees a count of 1 and keeps the original
    assert copies == [(0, 6, 5, 2)]
    assert bm.table[0, :2].tolist() == [7, 5] and bm.table[1, :2].tolist() == [7, 6]
    assert bm.ref[[7, 6, 5]].tolist() == [2, 1, 1]
    assert bm.free == [0, 1, 2, 3, 4]
    for b in range(2):
        pool.rows[bm.table[b, 1], 2] = 1000 + b
        hist[b][6] = 1000 + b
    for b in range(2):
        assert visible(bm, pool, b, 6) == hist[b]       # no cross-talk
    assert bm.check_invariants()
    bm.release([0])
    assert bm.ref[[7, 6, 5]].tolist() == [1, 1, 0] and bm.free == [0, 1, 2, 3, 4, 5]
    bm.release([1])
    assert bm.free == [0, 1, 2, 3, 4, 5, 6, 7] and bm.check_invariants()
    assert not bm.valid.any()


def test_worked_scenario_share_cow_release():
    _worked_scenario(BlockManager)


def _new_block_rule(cls):
    bm = cls(2, 4, batch=3, max_blocks=2)
    bm.prepare([0, 5, -1])
    assert bm.errors == [(1, blocks.ERR_UNMAPPED)] and bm.table[0, 0] == 1
    bm.prepare([4, 0, 0])
    assert bm.table[0, 1] == 0 and (2, blocks.ERR_NO_FREE) in bm.errors and bm.table[2, 0] == -1
    bm.prepare([8, -1, -1])
    assert (0, blocks.ERR_POSITION) in bm.errors
    assert bm.check_invariants()


def test_new_block_only_at_a_block_start_and_exhaustion():
    _new_block_rule(BlockManager)


def _three_sharers(cls):
    # a block shared by 3 sequences, all three writing: the first two copy,
    # the third writes in place (count r - k seen by the k-th)
    bm, pool = cls(6, 4, batch=3, max_blocks=2), Pool(6, 4)
    hist = [{}, {}, {}]
    for t in range(2):
        step(bm, pool, hist, [t, -1, -1], lambda b, p: p)
    bm.share(0, 1, 1)
    bm.share(0, 2, 1)
    assert bm.ref[5] == 3
    copies = bm.prepare([2, 2, 2], copy=pool.copy)
    assert [c[0] for c in copies] == [0, 1] and bm.table[2, 0] == 5
    assert bm.check_invariants()


def test_three_sharers_two_copies():
    _three_sharers(BlockManager)


def _churn(bm, pool, rng, steps, do_cow=True, careful_release=True):
    B = bm.table.shape[0]
    t = np.full(B, -1)
    hist = [dict() for _ in range(B)]
    for _ in range(steps):
        op = rng.random()
        if op < 0.15:
            # a fresh sequence takes a prefix of a live one
            live = [b for b in range(B) if t[b] >= 0]
            dead = [b for b in range(B) if t[b] < 0]
            if live and dead:
                src, dst = rng.choice(live), rng.choice(dead)
                n = int(rng.integers(1, t[src] + 2))            # tokens 0 .. n-1
                nb = (n + bm.bs - 1) // bm.bs
                bm.share(src, dst, nb)
                hist[dst] = {p: hist[src][p] for p in range(nb * bm.bs) if p in hist[src] and p < n}
                t[dst] = n - 1
                # the shared last block may hold src tokens past n-1: they are
                # overwritten by dst's next tokens (after copy-on-write)
        elif op < 0.25:
            b = int(rng.integers(B))
            if t[b] >= 0:
                if careful_release:
                    bm.release([b])
                else:       # planted: reclaim without looking at the counts
                    for lb in range(bm.table.shape[1]):
                        phys = bm.table[b, lb]
                        if phys >= 0:
                            bm.ref[phys] = 0
                            bm.free.append(int(phys))
                            bm.table[b, lb] = -1
                t[b] = -1
                hist[b] = {}
        else:
            nxt = np.where(t >= 0, t + 1, -1)
            start = rng.integers(0, 2, size=B).astype(bool) & (t < 0)
            nxt[start] = 0
            if do_cow:
                bm.prepare(nxt.tolist(), copy=pool.copy)
            else:           # planted: map new blocks but write shared ones in place
                for b, p in enumerate(nxt):
                    if p >= 0 and bm.table[b, p // bm.bs] < 0 and p % bm.bs == 0:
                        f = bm._take()
                        if f is not None:
                            bm.table[b, p // bm.bs] = f
            for b, p in enumerate(nxt):
                if p < 0 or p // bm.bs >= bm.table.shape[1]:
                    continue
                phys = bm.table[b, p // bm.bs]
                if phys < 0:
                    continue
                tok = int(rng.integers(1 << 30))
                pool.rows[phys, p % bm.bs] = tok
                hist[b][p] = tok
                t[b] = p
        yield t, hist


def test_random_churn_keeps_invariants_and_isolation():
    rng = np.random.default_rng(7)
    bm, pool = BlockManager(64, 4, batch=6, max_blocks=8), Pool(64, 4)
    for t, hist in _churn(bm, pool, rng, 400):
        assert bm.check_invariants()
        for b in range(len(t)):
            if t[b] >= 0:
                assert visible(bm, pool, b, t[b]) == {p: v for p, v in hist[b].items() if p <= t[b]}


@pytest.mark.parametrize("mistake", ["no_cow", "release_ignores_counts"])
def test_planted_mistakes_are_caught(mistake):
    rng = np.random.default_rng(7)
    bm, pool = BlockManager(64, 4, batch=6, max_blocks=8), Pool(64, 4)
    caught = False
    for t, hist in _churn(bm, pool, rng, 400, do_cow=mistake != "no_cow",
                          careful_release=mistake != "release_ignores_counts"):
        if not bm.check_invariants():
            caught = True
            break
        for b in range(len(t)):
            if t[b] >= 0 and visible(bm, pool, b, t[b]) != {p: v for p, v in hist[b].items() if p <= t[b]}:
                caught = True
        if caught:
            break
    assert caught


# Mistakes planted in copies of the oracle (subclasses, on the CPU): each is a
# plausible slip in the block manager, and each must fail one of the pins above.
class _ShortCopy(BlockManager):            # copy-on-write brings one row too few
    def prepare(self, positions, copy=None):
        short = (lambda s, d, r: copy(s, d, max(r - 1, 0))) if copy else None
        return super().prepare(positions, copy=short)


class _CopyKeepsCount(BlockManager):       # the shared block's count not dropped after its copy
    def prepare(self, positions, copy=None):
        copies = super().prepare(positions, copy=copy)
        for _, src, _, _ in copies:
            self.ref[src] += 1
        return copies


class _FifoFreeList(BlockManager):         # free list taken from the bottom, not the top
    def _take(self):
        if not self.free:
            return None
        f = self.free.pop(0)
        self.ref[f] = 1
        self.valid[f] = True
        return f


class _MidBlockAllocation(BlockManager):   # a new block taken mid-block instead of an error
    def prepare(self, positions, copy=None):
        for b, t in enumerate(positions):
            if t >= 0 and t // self.bs < self.table.shape[1] and self.table[b, t // self.bs] < 0 and t % self.bs:
                f = self._take()
                if f is not None:
                    self.table[b, t // self.bs] = f
        return super().prepare(positions, copy=copy)


class _ShareWithoutCounts(BlockManager):   # prefix sharing maps blocks without raising counts
    def share(self, src, dst, nblocks):
        before = self.ref.copy()
        super().share(src, dst, nblocks)
        self.ref[:] = before


class _ReleaseDescending(BlockManager):    # freed blocks pushed in descending id
    def release(self, seqs):
        n = len(self.free)
        super().release(seqs)
        self.free[n:] = sorted(self.free[n:], reverse=True)


def _churn_catches(cls):
    rng = np.random.default_rng(7)
    bm, pool = cls(64, 4, batch=6, max_blocks=8), Pool(64, 4)
    for t, hist in _churn(bm, pool, rng, 400):
        if not bm.check_invariants():
            return True
        for b in range(len(t)):
            if t[b] >= 0 and visible(bm, pool, b, t[b]) != {p: v for p, v in hist[b].items() if p <= t[b]}:
                return True
    return False


@pytest.mark.parametrize("cls", [_ShortCopy, _CopyKeepsCount, _FifoFreeList, _MidBlockAllocation,
                                 _ShareWithoutCounts, _ReleaseDescending], ids=lambda c: c.__name__.strip("_"))
def test_planted_block_manager_mistakes_fail_a_pin(cls):
    failed = []
    for pin in (_worked_scenario, _new_block_rule, _three_sharers):
        try:
            pin(cls)
        except AssertionError:
            failed.append(pin.__name__)
    if _churn_catches(cls):
        failed.append("churn")
    assert failed, cls.__name__
