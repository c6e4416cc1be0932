"""Rotary position embedding, fp64.

The pages use RoPE without defining it ([ring] 3.2, 3.4 and 8 defer the
formula; [primer] 4.5 and [pool] "RoPE baked into K rows" only say that the
rotation is applied to K, not V, before the row is cached).  Reading taken:
the usual rotate-half form.  For head_dim D and i in [0, D/2), the pair
(x[i], x[i + D/2]) is rotated by the angle pos * theta_i, with
theta_i = base ** (-2 i / D):

    y[i]       = x[i] cos(a) - x[i + D/2] sin(a)
    y[i + D/2] = x[i] sin(a) + x[i + D/2] cos(a),     a = pos * theta_i

The query is rotated the same way, so a score depends only on the position
difference: <R(a) q, R(b) k> = <q, R(b - a) k>.
"""

import numpy as np


def inv_freq(head_dim: int, base: float = 10000.0) -> np.ndarray:
    """theta_i = base ** (-2 i / D), i = 0 .. D/2 - 1, fp64."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(np.float64(base), -2.0 * i / head_dim)


def rotate(x, pos, base: float = 10000.0) -> np.ndarray:
    """Rotate the last axis of `x` ([..., D]) at integer positions `pos` (broadcast to x[..., 0])."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    half = D // 2
    theta = inv_freq(D, base)
    pos = np.asarray(pos, dtype=np.float64)[..., None]
    a = pos * theta                      # [..., D/2]
    c, s = np.cos(a), np.sin(a)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)
