"""Counter-keyed normal draws.

A draw is identified by an integer key tuple; numpy's SeedSequence hashes the
tuple into a 64-bit seed for a fresh torch generator.  Two calls with the same
key return the same tensor on the same device type; CPU draws are what the
oracle and the parity tests share.
"""

from __future__ import annotations

import numpy as np
import torch

# Positions are drawn in blocks of this many tokens: the values of a position
# depend only on (key, position), never on the range that asked for it.
POSITION_BLOCK = 256

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def to_dtype(name: str) -> torch.dtype:
    """Storage dtype name ("f32" | "bf16") -> torch dtype."""
    return _DTYPES[name]


def derive_seed(*key: int) -> int:
    """Hash an integer key tuple into a 63-bit generator seed."""
    words = [int(k) & 0xFFFFFFFF for k in key] + [(int(k) >> 32) & 0xFFFFFFFF for k in key]
    state = np.random.SeedSequence(words).generate_state(2, np.uint32)
    return int((int(state[0]) << 31) ^ int(state[1])) & ((1 << 63) - 1)


def randn(key: tuple, shape, dtype: str = "f32", device: str = "cpu") -> torch.Tensor:
    """N(0, 1) draws for `key`, rounded (round-to-nearest-even) to `dtype`."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(derive_seed(*key))
    x = torch.randn(tuple(shape), generator=gen, dtype=torch.float32, device=dev)
    return x.to(_DTYPES[dtype])
