"""The five decode workloads, as seeded synthetic inputs.

Each builder returns a `Workload`: cache geometry, the current position t_b of
every sequence, and for the paged layouts the block table and residency mask.
Positions, tables and masks are drawn with numpy's PCG64 from the workload
seed; K/V/Q values come from `generator.randn`.  `small=True` gives a
same-shaped case that the oracle finishes in seconds (several tiles plus a
ragged tail, positions before and after the first ring wrap).

Token values and prefix sharing: token p of sequence b belongs to its group's
shared prefix when p < shared_tokens[b]; such tokens have the same K/V for every
member of the group (they are one token stored once).  All other tokens belong
to the sequence itself.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from .generator import POSITION_BLOCK, randn

STREAM_K, STREAM_V, STREAM_Q = 1, 2, 3
OWNER_SEQ, OWNER_GROUP = 0, 1


@dataclass
class Workload:
    name: str
    layout: str                 # "window" (ring, or ring with pinned sinks) | "paged"
    dtype: str                  # cache storage: "f32" | "bf16" | "i8" (int8 codes + fp32 row scales, bf16 values)
    rope: str                   # "none" | "baked" | "read_time"
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    positions: np.ndarray       # int64 [batch]: position t_b of the token being decoded
    layers: int = 1
    window: int = 0
    sinks: int = 0
    block_size: int = 0
    num_blocks: int = 0
    max_blocks_per_seq: int = 0
    rope_base: float = 10000.0
    seed: int = 0
    steps: int = 1              # decode steps from an empty cache (tiny workload)
    block_table: np.ndarray | None = None   # int32 [batch, max_blocks_per_seq], -1 = unmapped
    valid: np.ndarray | None = None         # bool [num_blocks]; None = every slot resident
    group: np.ndarray = field(default=None)          # int64 [batch]
    shared_tokens: np.ndarray = field(default=None)  # int64 [batch]
    notes: str = ""

    def __post_init__(self):
        self.positions = np.asarray(self.positions, dtype=np.int64)
        if self.group is None:
            self.group = np.arange(self.batch, dtype=np.int64)
        if self.shared_tokens is None:
            self.shared_tokens = np.zeros(self.batch, dtype=np.int64)

    # ---- geometry -----------------------------------------------------------
    @property
    def capacity(self) -> int:
        """Slots per (sequence, kv head) of a window layout."""
        return self.window + self.sinks

    @property
    def group_size(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def value_dtype(self) -> str:
        """Type of the drawn values (q, K, V inputs): bf16 for an INT8 cache."""
        return "bf16" if self.dtype == "i8" else self.dtype

    @property
    def elt_bytes(self) -> int:
        """Bytes of one stored cache element (an INT8 code: 1)."""
        return {"f32": 4, "bf16": 2, "i8": 1}[self.dtype]

    @property
    def row_scale_bytes(self) -> int:
        """Bytes stored per cache row besides its elements (INT8: the fp32 scale)."""
        return 4 if self.dtype == "i8" else 0

    @property
    def value_bytes(self) -> int:
        return 4 if self.value_dtype == "f32" else 2

    def cache_shape(self, layers: int | None = None) -> tuple:
        """[layers, 2, batch, kv_heads, capacity, D] or [layers, 2, num_blocks, kv_heads, bs, D]."""
        L = self.layers if layers is None else layers
        if self.layout == "window":
            return (L, 2, self.batch, self.kv_heads, self.capacity, self.head_dim)
        return (L, 2, self.num_blocks, self.kv_heads, self.block_size, self.head_dim)

    # ---- values -------------------------------------------------------------
    def _owner(self, b: int, p: np.ndarray):
        shared = p < self.shared_tokens[b]
        kind = np.where(shared, OWNER_GROUP, OWNER_SEQ)
        ident = np.where(shared, self.group[b], b)
        return kind, ident

    def kv_history(self, layer: int, b: int, positions, device: str = "cpu"):
        """Pre-RoPE K and V of sequence b at `positions`: two [n, kv_heads, D] tensors."""
        p = np.asarray(positions, dtype=np.int64).reshape(-1)
        n = p.shape[0]
        H, D = self.kv_heads, self.head_dim
        out_k = torch.empty((n, H, D), dtype=torch.float32).to(_td(self.value_dtype))
        out_v = torch.empty_like(out_k)
        if n == 0:
            return out_k.to(device), out_v.to(device)
        kind, ident = self._owner(b, p)
        blk = p // POSITION_BLOCK
        off = p % POSITION_BLOCK
        keys = np.stack([kind, ident, blk], axis=1)
        uniq, inv = np.unique(keys, axis=0, return_inverse=True)
        inv = inv.reshape(-1)
        for u, (kd, idn, bk) in enumerate(uniq):
            sel = np.nonzero(inv == u)[0]
            base = (self.seed, layer, int(kd), int(idn), int(bk))
            kb = randn(base + (STREAM_K,), (POSITION_BLOCK, H, D), self.value_dtype)
            vb = randn(base + (STREAM_V,), (POSITION_BLOCK, H, D), self.value_dtype)
            idx = torch.from_numpy(off[sel])
            sel_t = torch.from_numpy(sel)
            out_k[sel_t] = kb[idx]
            out_v[sel_t] = vb[idx]
        return out_k.to(device), out_v.to(device)

    def query(self, layer: int, b: int, t: int | None = None) -> torch.Tensor:
        """Pre-RoPE query of sequence b for the token at position t (default t_b): [q_heads, D]."""
        t = int(self.positions[b]) if t is None else int(t)
        return randn((self.seed, layer, OWNER_SEQ, b, t, STREAM_Q), (self.q_heads, self.head_dim), self.value_dtype)

    def queries(self, layer: int, positions=None) -> torch.Tensor:
        pos = self.positions if positions is None else np.asarray(positions)
        return torch.stack([self.query(layer, b, int(pos[b])) for b in range(self.batch)])

    def new_kv(self, layer: int, positions=None):
        """K/V of the token being decoded at t_b for every sequence: two [batch, kv_heads, D]."""
        pos = self.positions if positions is None else np.asarray(positions)
        ks, vs = [], []
        for b in range(self.batch):
            k, v = self.kv_history(layer, b, [int(pos[b])])
            ks.append(k[0])
            vs.append(v[0])
        return torch.stack(ks), torch.stack(vs)


def _td(name: str) -> torch.dtype:
    return torch.float32 if name == "f32" else torch.bfloat16


# ---------------------------------------------------------------------------
# builders
# ---------------------------------------------------------------------------

def tiny_ring_sink_f32(small: bool = True, layers: int = 1) -> Workload:
    """fp32, batch 1, 1 layer, 4 q / 1 kv heads, D 64, 4 sinks + 60 window slots
    (capacity 64), 256 decode steps from empty, RoPE base 1e4 baked at absolute
    position.  Already small: `small` is accepted for a uniform interface."""
    steps = 256
    return Workload(
        name="tiny_ring_sink_f32", layout="window", dtype="f32", rope="baked",
        batch=1, q_heads=4, kv_heads=1, head_dim=64, layers=layers,
        window=60, sinks=4, seed=1, steps=steps, positions=[steps - 1],
        notes="256 decode steps from an empty cache; seed 1",
    )


def ring_bf16(small: bool = False, layers: int = 1) -> Workload:
    """bf16 ring: batch 8, 32 q / 8 kv heads, D 128, W 4096 (slot = t mod W, no
    sinks), t_b ~ U[4096, 65536], RoPE baked into K at the original position."""
    if small:
        W = 200
        pos = [W - 51, W - 1, 4321]       # before, at, and long after the first wrap
        return Workload(
            name="ring_bf16_small", layout="window", dtype="bf16", rope="baked",
            batch=3, q_heads=8, kv_heads=2, head_dim=128, layers=layers,
            window=W, sinks=0, seed=2, positions=pos,
        )
    rng = np.random.Generator(np.random.PCG64(2))
    pos = rng.integers(4096, 65536, size=8, endpoint=True)
    return Workload(
        name="ring_bf16", layout="window", dtype="bf16", rope="baked",
        batch=8, q_heads=32, kv_heads=8, head_dim=128, layers=layers,
        window=4096, sinks=0, seed=2, positions=pos,
        notes="t_b ~ U[4096, 65536] (seed 2): every ring is full",
    )


def sink_window_bf16(small: bool = False, layers: int = 1) -> Workload:
    """bf16 StreamingLLM cache: batch 32, 32 q / 8 kv heads, D 128, 4 pinned sink
    slots + 4092-slot rolling window, t_b ~ U[4096, 1e6], K stored pre-RoPE and
    rotated at read time from its position inside the cache."""
    if small:
        S, W = 4, 188
        pos = [100, S + W - 1, 987654]
        return Workload(
            name="sink_window_bf16_small", layout="window", dtype="bf16", rope="read_time",
            batch=3, q_heads=8, kv_heads=2, head_dim=128, layers=layers,
            window=W, sinks=S, seed=3, positions=pos,
        )
    rng = np.random.Generator(np.random.PCG64(3))
    pos = rng.integers(4096, 1_000_000, size=32, endpoint=True)
    return Workload(
        name="sink_window_bf16", layout="window", dtype="bf16", rope="read_time",
        batch=32, q_heads=32, kv_heads=8, head_dim=128, layers=layers,
        window=4092, sinks=4, seed=3, positions=pos,
        notes="t_b ~ U[4096, 1,000,000] (seed 3)",
    )


def _paged_prefix_tables(lengths, group, prefix_tokens, bs, max_blocks, rng):
    """Block tables for sequences that share their group's prefix.

    Token p of sequence b is a shared prefix token when p < min(prefix, t_b):
    the token being decoded (t_b = len_b - 1) is always the sequence's own.
    A logical block made only of shared tokens maps to the group's physical
    block; every other block is private to the sequence (for t_b inside the
    prefix, its block is a private copy holding the earlier shared tokens)."""
    B = len(lengths)
    t = lengths - 1
    shared_tokens = np.minimum(prefix_tokens, t)
    nblk = t // bs + 1
    shared_full = shared_tokens // bs
    alloc = 0
    group_blocks = {}
    for g in np.unique(group):
        n = int(shared_full[group == g].max())
        group_blocks[int(g)] = np.arange(alloc, alloc + n)
        alloc += n
    table = np.full((B, max_blocks), -1, dtype=np.int64)
    for b in range(B):
        sf = int(shared_full[b])
        table[b, :sf] = group_blocks[int(group[b])][:sf]
        n_priv = int(nblk[b]) - sf
        table[b, sf:nblk[b]] = np.arange(alloc, alloc + n_priv)
        alloc += n_priv
    perm = rng.permutation(alloc)
    mapped = table >= 0
    table[mapped] = perm[table[mapped]]
    return table.astype(np.int32), shared_tokens.astype(np.int64), alloc


def paged_shared_prefix_bf16(small: bool = False, layers: int = 1) -> Workload:
    """bf16 paged cache: 64 sequences, 16-token blocks, lengths ~ U[512, 8192],
    physical blocks a seeded random permutation, the first 2048 tokens shared by
    groups of 8 sequences through the same physical blocks, 32 q / 8 kv heads,
    D 128, RoPE baked at the absolute position, no residency mask."""
    rng = np.random.Generator(np.random.PCG64(4))
    if small:
        B, gs, bs, prefix, lo, hi, maxb = 8, 4, 16, 128, 40, 400, 25
        Hq, Hkv = 8, 2
    else:
        B, gs, bs, prefix, lo, hi, maxb = 64, 8, 16, 2048, 512, 8192, 512
        Hq, Hkv = 32, 8
    lengths = rng.integers(lo, hi, size=B, endpoint=True)
    if small:
        lengths[0] = 100                   # t_b inside the shared prefix
        lengths[1] = 2 * bs                # t_b on the last row of a block
    group = np.arange(B) // gs
    table, shared, nb = _paged_prefix_tables(lengths, group, prefix, bs, maxb, rng)
    return Workload(
        name="paged_shared_prefix_bf16" + ("_small" if small else ""), layout="paged",
        dtype="bf16", rope="baked", batch=B, q_heads=Hq, kv_heads=Hkv, head_dim=128,
        layers=layers, block_size=bs, num_blocks=nb, max_blocks_per_seq=maxb, seed=4,
        positions=lengths - 1, block_table=table, valid=None, group=group.astype(np.int64),
        shared_tokens=shared,
        notes="len_b ~ U[512, 8192] (seed 4) counts the new token; groups of 8 share 2048 tokens",
    )


def long_context_pool_bf16(small: bool = False, layers: int = 1, density: float = 0.5) -> Workload:
    """bf16 fixed pool: 1 sequence at t = 262143, 64-token blocks, a pool of 1024
    resident slots holding the last 64 logical blocks plus 960 seeded earlier
    ones in a seeded slot order, valid bit ~ Bernoulli(density) per slot (forced
    on for the last 4096 tokens), 16 q / 4 kv heads, D 256, RoPE baked."""
    rng = np.random.Generator(np.random.PCG64(5))
    if small:
        t, bs, pool, tail_blocks, Hq, Hkv = 20479, 64, 48, 4, 4, 1
    else:
        t, bs, pool, tail_blocks, Hq, Hkv = 262143, 64, 1024, 64, 16, 4
    nlog = t // bs + 1
    tail = np.arange(nlog - tail_blocks, nlog)
    early = rng.choice(nlog - tail_blocks, size=pool - tail_blocks, replace=False)
    resident = np.concatenate([np.sort(early), tail])
    slots = rng.permutation(pool)
    table = np.full((1, nlog), -1, dtype=np.int32)
    table[0, resident] = slots
    valid = rng.random(pool) < density
    valid[slots[-tail_blocks:]] = True
    return Workload(
        name="long_context_pool_bf16" + ("_small" if small else ""), layout="paged",
        dtype="bf16", rope="baked", batch=1, q_heads=Hq, kv_heads=Hkv, head_dim=256,
        layers=layers, block_size=bs, num_blocks=pool, max_blocks_per_seq=nlog, seed=5,
        positions=[t], block_table=table, valid=valid,
        notes=f"valid density {density} (seed 5); last {tail_blocks * bs} tokens always resident",
    )


def as_int8(wl: Workload, name: str) -> Workload:
    """The same workload (sizes, positions, seed, drawn values) over an INT8
    cache; read-time RoPE becomes baked (INT8 rows hold rotated keys)."""
    import dataclasses
    return dataclasses.replace(wl, name=name, dtype="i8", rope="none" if wl.rope == "none" else "baked",
                               notes=(wl.notes + "; " if wl.notes else "") + "INT8 cache, per-row fp32 scales")


def ring_int8(small: bool = False, layers: int = 1) -> Workload:
    """ring_bf16's sizes, positions and values over an INT8 cache."""
    return as_int8(ring_bf16(small, layers), "ring_int8" + ("_small" if small else ""))


def sink_window_int8(small: bool = False, layers: int = 1) -> Workload:
    """sink_window_bf16's sizes, positions and values over an INT8 cache that
    keeps its keys raw and rotates them at read time (in-cache positions)."""
    import dataclasses
    wl = as_int8(sink_window_bf16(small, layers), "sink_window_int8" + ("_small" if small else ""))
    return dataclasses.replace(wl, rope="read_time",
                               notes=wl.notes.replace("INT8 cache", "INT8 cache, raw keys rotated at read time"))


def paged_shared_prefix_int8(small: bool = False, layers: int = 1) -> Workload:
    """paged_shared_prefix_bf16's sizes, tables and values over an INT8 cache."""
    return as_int8(paged_shared_prefix_bf16(small, layers), "paged_shared_prefix_int8" + ("_small" if small else ""))


WORKLOAD_NAMES = {
    "tiny_ring_sink_f32": tiny_ring_sink_f32,
    "ring_bf16": ring_bf16,
    "sink_window_bf16": sink_window_bf16,
    "paged_shared_prefix_bf16": paged_shared_prefix_bf16,
    "long_context_pool_bf16": long_context_pool_bf16,
    "ring_int8": ring_int8,
    "sink_window_int8": sink_window_int8,
    "paged_shared_prefix_int8": paged_shared_prefix_int8,
}


def make_workload(name: str, small: bool = False, layers: int = 1, **kw) -> Workload:
    return WORKLOAD_NAMES[name](small=small, layers=layers, **kw)
