"""Per-row INT8 storage of the KV cache.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[primer] 5.1, "memory is short" (the quantised-cache item and its table):
storing the cache in INT8 instead of 16-bit floats halves its memory; the page
adds that calibration keeps the accuracy loss in check, and gives no format.

Reading taken (the plainest one the page supports): symmetric quantisation
with one scale per stored row, a row being one token's K (or V) for one kv
head, head_dim values:

    s   = max_i |x_i| / 127
    c_i = round(x_i / s), ties to even, clamped to [-127, 127]
    x_i is read back as c_i * s

A row of zeros stores s = 0 and zero codes.  No calibration: it needs a
trained model, which is out of scope.

The codes are integers chosen by floating-point arithmetic, so the oracle
makes that choice in fp32, the precision of the stored scale: s is the
correctly rounded fp32 quotient of the fp32 maximum and 127, and c_i the
nearest integer to the correctly rounded fp32 quotient x_i / s.  The rows
are the fp32 values being stored (with baked RoPE: the rotated key rounded
to fp32).  Reading back, c_i * s is exact in fp64.
"""

from __future__ import annotations

import numpy as np

QMAX = 127


def quantize_rows(x):
    """Rows x [..., D] (fp32-representable) -> (codes int8 [..., D], scales fp32 [...])."""
    x32 = np.asarray(x, dtype=np.float32)
    a = np.max(np.abs(x32), axis=-1)
    s = (a / np.float32(QMAX)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (x32 / s[..., None]).astype(np.float32)
    c = np.where(s[..., None] > 0, np.clip(np.rint(r), -QMAX, QMAX), 0)
    return c.astype(np.int8), s


def dequantize_rows(codes, scales):
    """codes [..., D] int8, scales [...] -> the values read back, fp64."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[..., None]


def store_i8(x):
    """The value a row holds after it is stored in INT8 and read back (fp64)."""
    c, s = quantize_rows(np.asarray(x, dtype=np.float64).astype(np.float32))
    return dequantize_rows(c, s)
