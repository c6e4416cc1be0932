"""Bit-exact recovery of attended sets through the real kernels (GPU helper).

Every key row an attended set may contain holds K = 0, so every attended
score is exactly 0 and every attended row gets the same softmax weight.  Each
live row carries an integer id.  In pass `ps`, kv head h looks at the id slice
j = ps * kv_heads + h, the ids [j D, (j + 1) D): a live V row whose id lies in
it is one-hot at column id - j D (value 1, or 127/128 = 127 codes of scale 2^-7
in an INT8 cache), every other live V row is zero.  Rows outside every
attended set hold NaN (bf16 K and V, or the INT8 row scales), so a kernel that
reads one gives NaN.  Output column c of every q head of kv head h is then
exactly unit(|A|) when the row with id j D + c is attended and exactly 0
otherwise, where

    bf16 cache: unit(n) = bf16(fp32(1) / fp32(n))
    INT8 cache: unit(n) = bf16(fp32(127/128) * (fp32(1) / fp32(n)))

(the kernels sum the equal weights exactly in fp32 and multiply the summed
output by the reciprocal of the summed weights).  The passes together recover
each sequence's attended set of ids exactly; a dropped, extra or wrong row
changes a column.  Expected sets come from the oracle's closed forms
(`oracle.window_attended`, `oracle.window_slot`, `oracle.paged_attended`)."""

from __future__ import annotations

import numpy as np
import torch

import oracle

NAN = float("nan")


def unit(n: int, dtype: str) -> float:
    one = np.float32(1.0) / np.float32(n)
    if dtype == "i8":
        one = np.float32(127.0 / 128.0) * one
    return float(torch.tensor(float(one), dtype=torch.float32).to(torch.bfloat16).float())


def window_live(t, sinks, window):
    """Attended positions of each sequence and their slots ([ring] 2.2, 3.1; [sink])."""
    pos = [oracle.window_attended(int(tb), sinks, window) if tb >= 0 else np.zeros(0, np.int64) for tb in t]
    slots = [oracle.window_slot(p, sinks, window) if len(p) else np.zeros(0, np.int64) for p in pos]
    return pos, slots


class Probe:
    """One cache (layer 0 of a one-layer descriptor) set up for the probe.

    ids      int64 [X, R] on the host: the id of each (X = sequence or block,
             R = slot or row) row that is live before the call, -1 for a row
             that must never be read (NaN).
    sets     per sequence, the ids its output must attend (after the call's
             own append, for a decode step).
    new_ids  decode step only: per sequence, the id of the token the call
             appends (its row is dead before the call), or None."""

    def __init__(self, kvc, d, cache, ids, sets, new_ids=None):
        self.kvc, self.d, self.cache = kvc, d, cache
        self.ids = torch.from_numpy(np.asarray(ids, dtype=np.int64)).cuda()
        self.sets = [np.asarray(s, dtype=np.int64) for s in sets]
        self.new_ids = new_ids
        self.D, self.Hkv = d.head_dim, d.kv_heads
        self.g = d.q_heads // d.kv_heads
        self.dtype = {0: "f32", 1: "bf16", 2: "i8"}[d.dtype]
        top = max([int(ids.max()) if ids.size else -1] + [int(s.max()) for s in self.sets if len(s)])
        self.passes = max(1, -(-(top + 1) // (self.D * self.Hkv)))

    def fill(self, ps):
        """K = 0 and V of pass ps on live rows, NaN elsewhere."""
        D, ids = self.D, self.ids
        live = ids >= 0
        col = torch.where(live, ids % D, torch.zeros_like(ids))
        if self.dtype == "i8":
            codes, scales = self.kvc.int8_views(self.d, self.cache)
            codes[0].zero_()
            for kv in (0, 1):
                sc = scales[0, kv]                          # [X, Hkv, R]
                sc.fill_(NAN)
                sc.transpose(1, 2)[live] = 0.0
            for h in range(self.Hkv):
                j = ps * self.Hkv + h
                sel = live & (ids // D == j)
                xi, ri = sel.nonzero(as_tuple=True)
                codes[0, 1, :, h][xi, ri, col[xi, ri]] = 127
                scales[0, 1, :, h][xi, ri] = 2.0 ** -7
        else:
            K, V = self.cache[0, 0], self.cache[0, 1]      # [X, Hkv, R, D]
            K.fill_(NAN)
            K.transpose(1, 2)[live] = 0.0
            for h in range(self.Hkv):
                j = ps * self.Hkv + h
                Vh = V[:, h]
                Vh.fill_(NAN)
                Vh[live] = 0.0
                sel = live & (ids // D == j)
                xi, ri = sel.nonzero(as_tuple=True)
                Vh[xi, ri, col[xi, ri]] = 1.0

    def new_rows(self, ps):
        """k_new = 0 and v_new of pass ps for the appended tokens ([B, Hkv, D], bf16)."""
        B, D = len(self.new_ids), self.D
        dt = torch.float32 if self.dtype == "f32" else torch.bfloat16
        k = torch.zeros((B, self.Hkv, D), dtype=dt)
        v = torch.zeros((B, self.Hkv, D), dtype=dt)
        one = 127.0 / 128.0 if self.dtype == "i8" else 1.0
        for b, e in enumerate(self.new_ids):
            for h in range(self.Hkv):
                if e is not None and e // D == ps * self.Hkv + h:
                    v[b, h, e % D] = one
        return k.cuda(), v.cuda()

    def expected(self, ps, rows=None):
        """Expected output of pass ps, [len(sets), q_heads, D] fp32."""
        D, g = self.D, self.g
        out = torch.zeros((len(self.sets), self.Hkv * g, D), dtype=torch.float32)
        for b, s in enumerate(self.sets):
            if not len(s):
                continue
            u = unit(len(s), self.dtype)
            for h in range(self.Hkv):
                j = ps * self.Hkv + h
                c = s[(s // D) == j] - j * D
                out[b, h * g:(h + 1) * g][:, torch.from_numpy(c)] = u
        return out

    def compare(self, got, ps, what):
        """got [len(sets), q_heads, D] (device or host) against the expected sets."""
        got = got.float().cpu()
        exp = self.expected(ps)
        if torch.equal(got, exp):
            return
        D, g = self.D, self.g
        msgs = []
        for b, s in enumerate(self.sets):
            for h in range(self.Hkv):
                j = ps * self.Hkv + h
                gb = got[b, h * g:(h + 1) * g]
                eb = exp[b, h * g:(h + 1) * g]
                if torch.equal(gb, eb):
                    continue
                nz = set((j * D + torch.nonzero(gb[0] != 0).flatten()).tolist())
                want = set(s[(s // D) == j].tolist())
                vals = sorted(set(gb[gb != 0].flatten().tolist()))[:4]
                msgs.append(f"seq {b} kv head {h} pass {ps}: missing {sorted(want - nz)[:8]}, "
                            f"extra {sorted(nz - want)[:8]}, values {vals} (want {unit(max(1, len(s)), self.dtype)}), "
                            f"nan {bool(torch.isnan(gb).any())}")
                if len(msgs) >= 6:
                    break
        raise AssertionError(f"{what}: attended set differs\n" + "\n".join(msgs))


def window_probe(kvc, *, dtype, B, Hq, Hkv, D, sinks, window, t, num_splits=0, fused=False, rope="none"):
    """Ring / sink+ring cache: ids are slots.  Live rows: the attended slots at
    t_b (at t_b without slot(t_b) for a decode step, whose kernel appends t_b).
    K = 0 rotates to 0, so any RoPE mode leaves the expected sets unchanged;
    read-time RoPE takes the kernels' rotating paths (runs cut at the
    sink/window boundary and the ring's wrap)."""
    t = np.asarray(t, dtype=np.int64)
    C = sinks + window
    layout = "sink_ring" if sinks else "ring"
    d = kvc.make_desc(layout, rope, dtype, 1, len(t), Hq, Hkv, D, window=window, sinks=sinks,
                      num_splits=num_splits)
    cache = kvc.alloc_cache(d, fill=NAN)
    ids = np.full((len(t), C), -1, dtype=np.int64)
    pos, slots = window_live(t, sinks, window)
    new_ids = []
    for b in range(len(t)):
        sl = slots[b]
        if fused:
            new = int(oracle.window_slot(np.array([t[b]]), sinks, window)[0])
            sl = sl[sl != new]
            new_ids.append(new)
        ids[b, sl] = sl
    return Probe(kvc, d, cache, ids, slots, new_ids if fused else None)


def paged_probe(kvc, *, dtype, Hq, Hkv, D, bs, num_blocks, table, valid, t, num_splits=0, fused=False,
                id_mode="rank"):
    """Paged cache.  Live rows: every (block, row) some sequence attends.
    id_mode "position": a row's id is its logical position (rows shared by
    several sequences sit at the same position in each); "rank": rows are
    numbered in (block, row) order."""
    t = np.asarray(t, dtype=np.int64)
    table = np.asarray(table, dtype=np.int32)
    B = len(t)
    d = kvc.make_desc("paged", "none", dtype, 1, B, Hq, Hkv, D, block_size=bs, num_blocks=num_blocks,
                      max_blocks_per_seq=table.shape[1], num_splits=num_splits)
    cache = kvc.alloc_cache(d, fill=NAN)
    att = [oracle.paged_attended(int(tb), table[b], valid, bs) if tb >= 0 else np.zeros(0, np.int64)
           for b, tb in enumerate(t)]
    rows = [(table[b, a // bs].astype(np.int64), a % bs) for b, a in enumerate(att)]
    pos_of = np.full((num_blocks, bs), -1, dtype=np.int64)
    for b, a in enumerate(att):
        ph, r = rows[b]
        prev = pos_of[ph, r]
        assert ((prev < 0) | (prev == a) | (id_mode == "rank")).all(), "a row shared at two positions"
        pos_of[ph, r] = a
    live = pos_of >= 0
    if id_mode == "position":
        idmap = pos_of.copy()
    else:
        idmap = np.full((num_blocks, bs), -1, dtype=np.int64)
        idmap[live] = np.arange(int(live.sum()))
    sets = [idmap[ph, r] for (ph, r) in rows]
    ids = idmap.copy()
    new_ids = None
    if fused:
        new_ids = []
        for b, tb in enumerate(t):
            ph, r = int(table[b, tb // bs]), int(tb % bs)
            assert ph >= 0, f"sequence {b}: the new token's block is unmapped"
            new_ids.append(int(idmap[ph, r]))
            ids[ph, r] = -1                  # written by the call itself
    p = Probe(kvc, d, cache, ids, sets, new_ids)
    p.table = torch.from_numpy(table).cuda()
    p.valid_bits = kvc.pack_valid_bits(torch.from_numpy(np.asarray(valid))).cuda() if valid is not None else None
    return p


def run_decode(kvc, p, t, ws=None):
    """Every pass of a probe through kvc_decode_attention (or kvc_decode_step
    when the probe has new tokens); raises on the first differing pass."""
    d = p.d
    ws = kvc.alloc_workspace(d) if ws is None else ws
    pos = torch.from_numpy(np.asarray(t, dtype=np.int32)).cuda()
    table = getattr(p, "table", None)
    valid = getattr(p, "valid_bits", None)
    g = torch.Generator().manual_seed(7)
    dt = torch.float32 if p.dtype == "f32" else torch.bfloat16
    q = torch.randn((d.batch, d.q_heads, d.head_dim), generator=g).to(dt).cuda()
    for ps in range(p.passes):
        p.fill(ps)
        if p.new_ids is None:
            out = kvc.decode_attention(d, p.cache, 0, q, pos, ws, block_table=table, valid_bits=valid)
        else:
            kn, vn = p.new_rows(ps)
            out = kvc.decode_step(d, p.cache, 0, q, kn, vn, pos, ws, block_table=table, valid_bits=valid)
        p.compare(out, ps, f"decode pass {ps}")
    err = kvc.get_error(ws)
    assert err == 0, f"device error bits {err:#x}"
