"""Slot maps, attended sets and layout models of the three cache layouts.

Closed forms (used for any size) and step-by-step models (pure Python, small
cases only) that keep each slot's original position beside its K/V, as the
pages ask ([ring] 3.2, 5.1 and 7: "position cache beside the KV cache").

Readings of the pages taken here:
* The window includes the current token: token t attends t-W+1 .. t
  ([ring] 2.2, 3.1, 6 and the 4.3 demo trace; [sink] cache-set equation).
  [ring] 1.2's "token 5 sees tokens 1-4" is the one sentence that excludes
  self; the rest of the page, its demo output and [sink] include it.
* Append happens before attention, so t is in its own attended set ([ring]
  4.3 demo: append, then attend).
* The pinned-sink cache is written as a ring after its S sink slots:
  slot(p) = p for p < S, else S + ((p - S) mod W).  [sink]'s manager compacts
  by concatenation instead; both hold the same set of tokens, and before the
  first wrap they hold them in the same order.
* RoPE at read time uses a token's index in [sink]'s compacted cache
  ("cache position shifting"): sinks keep 0..S-1, window token p sits at
  p - max(0, t - C + 1) with C = S + W, and the query at min(t, C - 1).
"""

from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

def window_slot(p, sinks: int, window: int):
    """Physical slot of position p.  Ring ([ring] 3.2, 3.3, 5.1): slot = p mod W.
    With S pinned sinks: p for p < S, else S + ((p - S) mod W)."""
    p = np.asarray(p, dtype=np.int64)
    return np.where(p < sinks, p, sinks + np.mod(p - sinks, window))


def window_attended(t: int, sinks: int, window: int) -> np.ndarray:
    """Positions attended by the token at t, ascending.

    Ring ([ring] 2.2, 6): t-W+1 .. t clipped at 0.  With sinks ([sink]
    cache-set equation): {0 .. S-1} U {t-W+1 .. t}, each clipped to 0 .. t.
    """
    sinks_part = np.arange(0, min(sinks, t + 1), dtype=np.int64)
    lo = max(sinks, t - window + 1)
    return np.concatenate([sinks_part, np.arange(lo, t + 1, dtype=np.int64)])


def incache_position(p, t: int, sinks: int, window: int):
    """Index of position p in [sink]'s compacted cache at time t (RoPE cache
    position shifting): sinks keep their index, window tokens shift left by
    max(0, t - C + 1), C = S + W.  The query's own index is incache_position(t, t)."""
    p = np.asarray(p, dtype=np.int64)
    shift = max(0, t - (sinks + window) + 1)
    return np.where(p < sinks, p, p - shift)


def paged_attended(t: int, table_row, valid, block_size: int) -> np.ndarray:
    """Positions p <= t whose logical block is mapped (table entry >= 0) and whose
    physical slot is resident (valid bit set; `valid` None = all resident).
    [share] 3.1 (block table), [pool] "kernel forgets absent blocks"."""
    table_row = np.asarray(table_row)
    p = np.arange(t + 1, dtype=np.int64)
    phys = table_row[p // block_size]
    keep = phys >= 0
    if valid is not None:
        valid = np.asarray(valid, dtype=bool)
        keep &= valid[np.where(phys >= 0, phys, 0)]
    return p[keep]


# ---------------------------------------------------------------------------
# step-by-step layout models (small cases)
# ---------------------------------------------------------------------------

class RingKV:
    """Fixed-size ring of W slots with a head pointer ([ring] 4.2).

    Each slot keeps key, value, original position and write sequence number.
    append() writes slot `head` then advances head = (head + 1) mod W ([ring]
    3.3); visible() lists the live slots oldest first, starting at head - size.
    """

    def __init__(self, window: int):
        self.window = window
        self.keys = [None] * window
        self.values = [None] * window
        self.positions = [None] * window
        self.insert_seq = [None] * window
        self.head = 0
        self.size = 0
        self.num_writes = 0

    def append(self, key, value, position: int):
        self.keys[self.head] = key
        self.values[self.head] = value
        self.positions[self.head] = position
        self.insert_seq[self.head] = self.num_writes
        self.num_writes += 1
        self.head = (self.head + 1) % self.window
        self.size = min(self.size + 1, self.window)

    def visible(self):
        start = self.head - self.size
        out = []
        for i in range(self.size):
            slot = (start + i) % self.window
            out.append({"key": self.keys[slot], "value": self.values[slot],
                        "position": self.positions[slot], "insert_seq": self.insert_seq[slot],
                        "slot": slot})
        return out


class StreamingKV:
    """Compacting StreamingLLM cache ([sink] cache manager).

    Appending concatenates the new token; once longer than S + W the cache keeps
    its first S entries and its last W entries, in chronological order.  The
    index of an entry in this list is its in-cache position.
    """

    def __init__(self, sinks: int, window: int):
        self.sinks = sinks
        self.window = window
        self.entries = []

    def append(self, key, value, position: int):
        self.entries.append({"key": key, "value": value, "position": position})
        if len(self.entries) > self.sinks + self.window:
            self.entries = self.entries[: self.sinks] + self.entries[-self.window:]

    def visible(self):
        return [dict(e, incache=i) for i, e in enumerate(self.entries)]


class SinkRingKV:
    """Physical cache of C = S + W slots: S pinned sink slots, then a ring.

    Slot of position p: p for p < S, else S + ((p - S) mod W); each slot keeps
    the position it holds.  visible() lists the live slots in chronological
    order of the positions they hold.
    """

    def __init__(self, sinks: int, window: int):
        self.sinks = sinks
        self.window = window
        C = sinks + window
        self.keys = [None] * C
        self.values = [None] * C
        self.positions = [None] * C

    def slot_of(self, position: int) -> int:
        if position < self.sinks:
            return position
        return self.sinks + (position - self.sinks) % self.window

    def append(self, key, value, position: int):
        s = self.slot_of(position)
        self.keys[s] = key
        self.values[s] = value
        self.positions[s] = position

    def visible(self):
        live = [s for s in range(len(self.positions)) if self.positions[s] is not None]
        live.sort(key=lambda s: self.positions[s])
        return [{"key": self.keys[s], "value": self.values[s], "position": self.positions[s],
                 "slot": s} for s in live]


class PagedKV:
    """Pool of fixed-size blocks addressed through per-sequence block tables
    ([share] 3.1, 5.1) with a residency bit per pool slot ([pool] "kernel
    forgets absent blocks").  Token p of sequence b lives at row p mod bs of
    physical block table[b][p // bs]."""

    def __init__(self, num_blocks: int, block_size: int, table, valid=None):
        self.block_size = block_size
        self.table = np.array(table, dtype=np.int64)
        self.valid = np.ones(num_blocks, dtype=bool) if valid is None else np.array(valid, dtype=bool)
        self.keys = [[None] * block_size for _ in range(num_blocks)]
        self.values = [[None] * block_size for _ in range(num_blocks)]
        self.positions = [[None] * block_size for _ in range(num_blocks)]

    def append(self, b: int, key, value, position: int):
        phys = int(self.table[b][position // self.block_size])
        if phys < 0:
            raise IndexError("append into an unmapped logical block")
        r = position % self.block_size
        self.keys[phys][r] = key
        self.values[phys][r] = value
        self.positions[phys][r] = position

    def visible(self, b: int, t: int):
        """Tokens p <= t of sequence b in mapped, resident blocks, in logical order."""
        out = []
        for lb in range((t // self.block_size) + 1):
            phys = int(self.table[b][lb])
            if phys < 0 or not self.valid[phys]:
                continue
            for r in range(self.block_size):
                p = lb * self.block_size + r
                if p > t:
                    break
                out.append({"key": self.keys[phys][r], "value": self.values[phys][r],
                            "position": self.positions[phys][r], "block": phys, "row": r})
        return out
