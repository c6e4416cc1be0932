"""One decode step of attention over a KV cache, fp64 with exact sums.

Definition followed ([primer] 2.2 and 4.2; [sink] softmax equations; [ring]
4.3 demo): for a new query q and the attended keys/values,

    s_j = (q . k_j) / sqrt(D)
    A_j = exp(s_j - max s) / sum_m exp(s_m - max s)      (sum_j A_j = 1)
    out = sum_j A_j v_j

Grouped-query attention ([share] 2.2, 4.1): q head h reads kv head
floor(h / g), g = q_heads / kv_heads (contiguous grouping is the reading taken;
the pages only say that several q heads share one kv head).

Every sum is math.fsum (exactly rounded), so the result depends on the set of
attended (k, v) pairs and not on the order they are visited in: a ring read in
physical slot order, a compacted cache and a masked full history give the
same bits.  An empty attended set gives zeros (not stated by the pages; only a
fully masked paged sequence reaches it).
"""

from __future__ import annotations

import math

import numpy as np

from .layouts import incache_position
from .rope import rotate
from .storage import round_storage


def _fsum_rows(m: np.ndarray) -> np.ndarray:
    """Exactly rounded sum along the last axis of a 2-D array."""
    return np.array([math.fsum(row) for row in m.tolist()], dtype=np.float64)


def attend(q, K, V, scale: float):
    """q [g, D], K [n, D], V [n, D] (fp64, already rotated) -> (out [g, D], A [g, n])."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    g, D = q.shape
    n = K.shape[0]
    if n == 0:
        return np.zeros((g, D)), np.zeros((g, 0))
    out = np.empty((g, D))
    A = np.empty((g, n))
    for h in range(g):
        s = _fsum_rows(q[h][None, :] * K) * scale          # [n]
        w = np.exp(s - s.max())
        A[h] = w / math.fsum(w.tolist())
        out[h] = _fsum_rows((A[h][:, None] * V).T)           # [D]
    return out, A


def _rotated_operands(q, K, positions, t, rope, base, storage, sinks, window):
    """Apply the RoPE mode to the query and the cached keys.

    baked     ([primer] 4.5, [pool] "RoPE baked into K rows"): K is rotated at
              its absolute position before it is stored, so the stored row is
              the rotated value rounded to the storage type; q rotated at t.
    read_time ([sink] "RoPE cache position shifting"): K is stored raw and
              rotated when read, at its in-cache position; q at its own.
    none      no rotation.
    """
    if rope == "baked":
        return rotate(q, t, base), round_storage(rotate(K, positions, base), storage)
    if rope == "read_time":
        ip = incache_position(positions, t, sinks, window)
        iq = int(incache_position(t, t, sinks, window))
        return rotate(q, iq, base), rotate(K, ip, base)
    if rope == "none":
        return np.asarray(q, dtype=np.float64), np.asarray(K, dtype=np.float64)
    raise ValueError(rope)


def decode_reference(q, K, V, positions, t: int, *, rope: str = "none", base: float = 10000.0,
                     storage: str = "f32", sinks: int = 0, window: int = 0, scale=None):
    """Decode output for one kv head's query group.

    q [g, D] pre-RoPE query heads; K, V [n, D] pre-RoPE cached rows (values as
    stored, i.e. already in the storage type) of the attended `positions` [n].
    Returns out [g, D].
    """
    q = np.asarray(q, dtype=np.float64)
    D = q.shape[-1]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    positions = np.asarray(positions, dtype=np.int64)
    qr, Kr = _rotated_operands(q, K, positions, t, rope, base, storage, sinks, window)
    out, _ = attend(qr, Kr, V, scale)
    return out


def decode_masked_history(q, K_hist, V_hist, t: int, mask, *, rope: str = "none",
                          base: float = 10000.0, storage: str = "f32", sinks: int = 0,
                          window: int = 0, scale=None):
    """The same step computed over the full history 0..t with a score mask.

    K_hist, V_hist [t+1, D] hold every position 0..t; `mask` [t+1] marks the
    attended ones.  Masked scores are -inf (weight exactly 0), the way a
    prefill-style masked kernel handles a window ([ring] 3.1, 5.2).
    """
    q = np.asarray(q, dtype=np.float64)
    D = q.shape[-1]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    mask = np.asarray(mask, dtype=bool)
    positions = np.arange(t + 1, dtype=np.int64)
    if not mask.any():
        return np.zeros_like(q)
    qr, Kr = _rotated_operands(q, K_hist, positions, t, rope, base, storage, sinks, window)
    V = np.asarray(V_hist, dtype=np.float64)
    out = np.empty_like(qr)
    for h in range(qr.shape[0]):
        s = _fsum_rows(qr[h][None, :] * Kr) * scale
        s = np.where(mask, s, -np.inf)
        w = np.exp(s - s.max())
        A = w / math.fsum(w.tolist())
        out[h] = _fsum_rows((A[:, None] * V).T)
    return out


def decode_sequence(q, K, V, positions, t: int, **spec):
    """All q heads of one sequence: q [Hq, D], K/V [n, Hkv, D] at `positions` [n].

    q head h uses kv head floor(h / g), g = Hq / Hkv.  Returns out [Hq, D]."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Hq, Hkv = q.shape[0], K.shape[1]
    g = Hq // Hkv
    out = np.empty_like(q)
    for h in range(Hkv):
        out[h * g:(h + 1) * g] = decode_reference(q[h * g:(h + 1) * g], K[:, h], V[:, h],
                                                  positions, t, **spec)
    return out
