"""Block manager of a paged KV cache: allocation, prefix sharing with reference
counts, copy-on-write, release.  TEST INFRASTRUCTURE ONLY (see oracle/__init__).

Follows [share] "Shared state, isolated problems: KV cache and batching":
  §3.1 / §5.1  blocks come from a free list and are mapped through a block
               table; a new block is taken when a sequence's current block
               is full;
  §3.2 / §5.1  prefix sharing points another sequence's table at the same
               physical blocks and raises their reference counts; a block
               referenced more than once is read-only, and a sequence about
               to write into it first copies it (copy-on-write);
  §6.1         when a sequence ends its blocks' counts drop by one, and a
               block is reclaimed only when its count reaches zero.

Readings where the page is silent (the same on the GPU):
  * the free list is a stack: allocation takes the top, in ascending
    sequence order within one call;
  * sequences preparing the same shared block in one call are served in
    ascending order: the k-th of them (k = 0, 1, ...) copies while the
    count it sees, r - k, is above one; the last one may write in place;
  * a copy brings the rows before the appended token (rows 0 .. t mod bs - 1)
    of every layer, K and V, every kv head;
  * blocks freed by one release call are pushed in ascending block id;
  * a new block is taken only at a block's first row (t mod bs == 0);
    appending into the middle of an unmapped block is an error;
  * sharing requires the destination's blocks to be unmapped.
"""

from __future__ import annotations

import numpy as np

# error codes of the model (the GPU reports the same conditions as bits)
ERR_NO_FREE = "no free block"
ERR_UNMAPPED = "append into the middle of an unmapped block"
ERR_POSITION = "position past the block table"
ERR_SHARE = "share into mapped blocks"


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, batch: int, max_blocks: int, free=None):
        self.num_blocks = num_blocks
        self.bs = block_size
        self.table = np.full((batch, max_blocks), -1, dtype=np.int64)
        self.ref = np.zeros(num_blocks, dtype=np.int64)
        self.valid = np.zeros(num_blocks, dtype=bool)
        self.free = list(range(num_blocks)) if free is None else list(free)   # stack; top = last
        self.errors = []

    # -- allocation ----------------------------------------------------------
    def _take(self):
        if not self.free:
            return None
        f = self.free.pop()
        self.ref[f] = 1
        self.valid[f] = True
        return f

    def prepare(self, positions, copy=None):
        """Make the block of each sequence's next token (position t_b; t_b < 0:
        none) mapped, private and resident.  `copy(src, dst, rows)` moves the
        first `rows` rows of a block (all layers, K and V, all kv heads).
        Returns the list of (seq, src, dst, rows) copies, in sequence order."""
        copies = []
        for b, t in enumerate(positions):
            t = int(t)
            if t < 0:
                continue
            lb, r = t // self.bs, t % self.bs
            if lb >= self.table.shape[1]:
                self.errors.append((b, ERR_POSITION))
                continue
            phys = int(self.table[b, lb])
            if phys < 0:
                if r != 0:
                    self.errors.append((b, ERR_UNMAPPED))
                    continue
                f = self._take()
                if f is None:
                    self.errors.append((b, ERR_NO_FREE))
                    continue
                self.table[b, lb] = f
            elif self.ref[phys] > 1:
                f = self._take()
                if f is None:
                    self.errors.append((b, ERR_NO_FREE))
                    continue
                if copy is not None:
                    copy(phys, f, r)
                copies.append((b, phys, f, r))
                self.ref[phys] -= 1
                self.table[b, lb] = f
        return copies

    # -- sharing ---------------------------------------------------------------
    def share(self, src: int, dst: int, nblocks: int):
        """dst's logical blocks 0 .. nblocks-1 point at src's; counts rise."""
        if np.any(self.table[dst, :nblocks] >= 0):
            self.errors.append((dst, ERR_SHARE))
            return
        for lb in range(nblocks):
            phys = int(self.table[src, lb])
            if phys >= 0:
                self.table[dst, lb] = phys
                self.ref[phys] += 1

    # -- release ---------------------------------------------------------------
    def release(self, seqs):
        """Sequences end: every mapped block's count drops by one and the entry
        is unmapped; blocks reaching zero go back to the free list (ascending
        id) and lose their residency bit."""
        freed = set()
        for b in seqs:
            for lb in range(self.table.shape[1]):
                phys = int(self.table[b, lb])
                if phys < 0:
                    continue
                self.ref[phys] -= 1
                self.table[b, lb] = -1
                if self.ref[phys] == 0:
                    freed.add(phys)
        for phys in sorted(freed):
            self.free.append(phys)
            self.valid[phys] = False

    # -- checks ------------------------------------------------------------------
    def check_invariants(self):
        """Counts equal table references; free and referenced blocks partition
        the pool; a referenced block is resident ([share] §7: sharing must be
        verifiable)."""
        refs = np.zeros(self.num_blocks, dtype=np.int64)
        for phys in self.table[self.table >= 0]:
            refs[phys] += 1
        if not np.array_equal(refs, self.ref):
            return False
        free = set(self.free)
        if len(free) != len(self.free):
            return False
        used = set(np.nonzero(self.ref > 0)[0].tolist())
        if free & used or (free | used) != set(range(self.num_blocks)):
            return False
        return bool(np.all(self.valid[list(used)])) if used else True
