"""Chunked prefill over the three cache layouts.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[pool] "the real cost of long context" and "paging": prefill runs in chunks
of 128-256 tokens, sharing one mechanism with the paged pool; [ring] 3.1 and
5.2 describe the window as a mask on the score matrix during prefill.

Reading taken (the pages fix the chunk size and the masks, not the call): a
chunk holds T consecutive tokens of a sequence, at positions pos0 .. pos0+T-1,
with their q, k and v.  Token i of the chunk gets exactly the output that a
decode step at t = pos0 + i would give after the chunk's tokens up to i have
been appended: attention of q_i over the attended set A(t) of the layout
(window, sinks + window, or mapped and valid blocks), whose keys are the
sequence's rows at those positions -- the chunk's own rows for positions
>= pos0, the rows already cached for earlier positions.  After the call the
cache holds the chunk's tokens as T appends would leave it.  Positions below
0 are left padding: no output (zeros), nothing appended.
"""

from __future__ import annotations

import numpy as np

from .attention import decode_sequence


def prefill_sequence(q_chunk, K_hist, V_hist, pos0: int, attended, **spec):
    """Outputs of one sequence's chunk.

    q_chunk [T, Hq, D] pre-RoPE queries of the chunk; K_hist, V_hist
    [N, Hkv, D] the sequence's rows at positions 0 .. N-1 (N >= pos0 + T; the
    chunk's own rows among them), as stored (pre-RoPE values in the storage
    type); attended(t) the layout's attended positions of token t; spec as for
    decode_sequence (rope, base, storage, sinks, window, scale).
    Returns out [T, Hq, D] (fp64).
    """
    q_chunk = np.asarray(q_chunk, dtype=np.float64)
    K_hist = np.asarray(K_hist, dtype=np.float64)
    V_hist = np.asarray(V_hist, dtype=np.float64)
    T = q_chunk.shape[0]
    out = np.zeros_like(q_chunk)
    for i in range(T):
        t = pos0 + i
        if t < 0:
            continue
        ps = np.asarray(attended(t), dtype=np.int64)
        out[i] = decode_sequence(q_chunk[i], K_hist[ps], V_hist[ps], ps, t, **spec)
    return out
