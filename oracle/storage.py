"""Rounding a value to the cache's storage type.

The cache of the pages is a preallocated half-precision tensor ([ring] 5.1,
"kv_cache = torch.zeros(..., dtype=torch.float16)"; [primer] 4.4); the
workloads store bf16 or fp32.  A stored value is the real value rounded to the
nearest representable one, ties to even.
"""

import numpy as np


def round_bf16(x):
    """Nearest bfloat16 of fp64 `x` (ties to even), returned as fp64.

    bfloat16 keeps 8 significant bits.  With x = m * 2**e, 0.5 <= |m| < 1,
    the kept significand is m * 2**8 rounded to an integer (np.rint rounds
    halves to even).  Normal range only: the workloads draw N(0, 1) values,
    far from bf16's underflow and overflow.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def round_f32(x):
    """Nearest fp32 of fp64 `x` (numpy's cast rounds to nearest, ties to even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_storage(x, dtype: str):
    """The value read back after storing rows x [..., D] as "bf16" | "f32" |
    "i8" (per-row INT8 codes and an fp32 scale, `oracle.quant`)."""
    if dtype == "bf16":
        return round_bf16(x)
    if dtype == "f32":
        return round_f32(x)
    if dtype == "i8":
        from .quant import store_i8
        return store_i8(x)
    raise ValueError(dtype)
