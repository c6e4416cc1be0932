"""Pins of the oracle's per-row INT8 storage (oracle.quant) against closed
forms, a brute-force search and exactness properties ([primer] 5.1,
quantised cache: INT8 halves the memory; the per-row symmetric format is
the reading taken)."""

import math

import numpy as np
import pytest

from oracle import attention, quant


def test_worked_row_closed_form():
    # max |x| = 254 -> s = 2 exactly; the quotients are exact, so the codes
    # are the plain ties-to-even roundings of x / 2
    x = np.array([254.0, 1.0, -3.0, 5.0, -254.0, 0.0, 127.0, -0.5])
    c, s = quant.quantize_rows(x)
    assert s.dtype == np.float32 and float(s) == 2.0
    assert c.dtype == np.int8
    assert c.tolist() == [127, 0, -2, 2, -127, 0, 64, 0]
    assert quant.dequantize_rows(c, s).tolist() == [254.0, 0.0, -4.0, 4.0, -254.0, 0.0, 128.0, 0.0]


def test_zero_row_and_sign_of_the_maximum():
    c, s = quant.quantize_rows(np.zeros((2, 8)))
    assert s.tolist() == [0.0, 0.0] and not c.any()
    assert not quant.dequantize_rows(c, s).any()
    # the largest magnitude is negative: it still takes the full code range
    c, s = quant.quantize_rows(np.array([-508.0, 4.0, 2.0]))
    assert float(s) == 4.0 and c.tolist() == [-127, 1, 0]


def _nearest_even_search(r):
    """The integer k in [-127, 127] nearest to r, ties to the even one (search)."""
    best = None
    for k in range(-127, 128):
        d = abs(r - k)
        if best is None or d < best[0] or (d == best[0] and k % 2 == 0):
            best = (d, k)
    return best[1]


def test_codes_against_brute_force_search():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((6, 16)) * np.array([1e-3, 1.0, 3.0, 50.0, 1e4, 0.25])[:, None]).astype(np.float32)
    x[2, 5] = x[2, 5] * 0  # a zero entry in a nonzero row
    c, s = quant.quantize_rows(x)
    for i in range(x.shape[0]):
        si = np.float32(np.max(np.abs(x[i])) / np.float32(127))
        assert s[i] == si
        for j in range(x.shape[1]):
            r = float(np.float32(x[i, j] / si))
            assert c[i, j] == _nearest_even_search(r), (i, j)


def test_invariants_on_random_rows():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((200, 128)) * rng.uniform(1e-2, 1e2, size=(200, 1))
    x32 = x.astype(np.float32).astype(np.float64)
    c, s = quant.quantize_rows(x)
    assert np.abs(c.astype(np.int32)).max() <= 127
    # the largest magnitude of every row maps to +-127
    assert (np.abs(c.astype(np.int32)).max(axis=1) == 127).all()
    # read back within half a step (the fp32 quotient adds a relative 2^-24)
    err = np.abs(x32 - quant.dequantize_rows(c, s))
    assert (err <= s[:, None].astype(np.float64) * (0.5 + 1e-6)).all()
    # scaling a row by a power of two scales s and keeps the codes
    c2, s2 = quant.quantize_rows(x32 * 8.0)
    assert (c2 == c).all() and (s2 == s * np.float32(8)).all()


def test_integer_rows_are_stored_exactly_and_attention_is_unchanged():
    # rows of integers in [-127, 127] holding +-127 have s = 1: lossless
    rng = np.random.default_rng(9)
    K = rng.integers(-127, 128, size=(12, 16)).astype(np.float64)
    V = rng.integers(-127, 128, size=(12, 16)).astype(np.float64)
    K[:, 3] = 127
    V[:, 0] = -127
    assert (quant.store_i8(K) == K).all() and (quant.store_i8(V) == V).all()
    q = rng.standard_normal((4, 16)) * 0.05
    ps = list(range(12))
    want = attention.decode_reference(q, K, V, ps, 11)
    got = attention.decode_reference(q, quant.store_i8(K), quant.store_i8(V), ps, 11, storage="i8")
    assert (got == want).all()


def test_baked_keys_are_quantised_after_rotation():
    # with baked RoPE the stored key is the rotated row, quantised; at position
    # 0 the rotation is the identity, so a lossless integer row stays exact
    rng = np.random.default_rng(10)
    K = rng.integers(-127, 128, size=(1, 8)).astype(np.float64)
    K[0, 0] = 127
    V = rng.standard_normal((1, 8))
    q = rng.standard_normal((2, 8))
    out = attention.decode_reference(q, K, V, [0], 0, rope="baked", storage="i8")
    assert np.allclose(out, np.repeat(V, 2, axis=0), rtol=0, atol=0)
    # at a later position the rows differ from the unrotated ones, but each
    # still reads back within half a step of the rotated value
    from oracle.rope import rotate
    R = rotate(K, np.array([37]), 10000.0)
    c, s = quant.quantize_rows(R)
    assert np.abs(R - quant.dequantize_rows(c, s)).max() <= float(s[0]) * (0.5 + 1e-6) + 1e-6
    assert math.isclose(float(s[0]), float(np.abs(R.astype(np.float32)).max()) / 127, rel_tol=1e-6)


def test_read_time_keys_are_quantised_before_rotation():
    # read-time RoPE on an INT8 cache: the raw key is stored and the value read
    # back (code * scale) is rotated at its in-cache position.  Integer rows
    # holding +-127 are stored losslessly, so the INT8 result equals the
    # unquantised one exactly, past the cache's first shift; quantising the
    # rotated key instead (the baked rule) would not.
    rng = np.random.default_rng(12)
    S, W, t, D = 4, 7, 30, 16
    pos = np.concatenate([np.arange(S), np.arange(t - W + 1, t + 1)])
    K = rng.integers(-127, 128, size=(len(pos), D)).astype(np.float64)
    V = rng.integers(-127, 128, size=(len(pos), D)).astype(np.float64)
    K[:, 5] = -127
    V[:, 2] = 127
    q = rng.standard_normal((2, D)) * 0.05
    spec = dict(rope="read_time", sinks=S, window=W)
    want = attention.decode_reference(q, K, V, pos, t, storage="f32", **spec)
    got = attention.decode_reference(q, quant.store_i8(K), quant.store_i8(V), pos, t, storage="i8", **spec)
    assert (got == want).all()
    from oracle.layouts import incache_position
    from oracle.rope import rotate
    ip = incache_position(pos, t, S, W)
    rotated_then_stored = quant.store_i8(rotate(K, ip, 10000.0))
    assert not np.allclose(rotated_then_stored, rotate(K, ip, 10000.0), rtol=0, atol=1e-6)


@pytest.mark.parametrize("D", [128, 256])
def test_store_i8_matches_quantize_then_dequantize(D):
    rng = np.random.default_rng(D)
    x = rng.standard_normal((5, D))
    c, s = quant.quantize_rows(x.astype(np.float32))
    assert (quant.store_i8(x) == quant.dequantize_rows(c, s)).all()


# ---------------------------------------------------------------------------
# planted mistakes (in copies of the quantiser, on the CPU): each fails a pin
# ---------------------------------------------------------------------------

def _check_quantizer(qfn) -> bool:
    """The pins above, for a quantiser qfn(x) -> (codes, scales); False on the first failure."""
    try:
        c, s = qfn(np.array([254.0, 1.0, -3.0, 5.0, -254.0, 0.0, 127.0, -0.5]))
        assert float(s) == 2.0 and np.asarray(c).tolist() == [127, 0, -2, 2, -127, 0, 64, 0]
        c, s = qfn(np.array([-508.0, 4.0, 2.0]))
        assert float(s) == 4.0 and np.asarray(c).tolist() == [-127, 1, 0]
        rng = np.random.default_rng(7)
        x = (rng.standard_normal((6, 16)) * np.array([1e-3, 1.0, 3.0, 50.0, 1e4, 0.25])[:, None]).astype(np.float32)
        c, s = qfn(x)
        for i in range(x.shape[0]):
            si = np.float32(np.max(np.abs(x[i])) / np.float32(127))
            assert np.asarray(s)[i] == si
            for j in range(x.shape[1]):
                assert np.asarray(c)[i, j] == _nearest_even_search(float(np.float32(x[i, j] / si)))
        return True
    except AssertionError:
        return False


def _planted(scale_div=127.0, rounding=np.rint, per_tensor=False, signed_max=False):
    def qfn(x):
        x32 = np.asarray(x, dtype=np.float32)
        a = np.max(x32, axis=-1) if signed_max else np.max(np.abs(x32), axis=-1)
        if per_tensor:
            a = np.full_like(a, np.max(np.abs(x32)))
        s = (np.abs(a) / np.float32(scale_div)).astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            r = (x32 / s[..., None]).astype(np.float32)
        c = np.where(s[..., None] > 0, np.clip(rounding(r), -127, 127), 0)
        return c.astype(np.int8), s
    return qfn


def test_planted_quantizer_mistakes_fail_a_pin():
    assert _check_quantizer(quant.quantize_rows)
    assert _check_quantizer(_planted())                       # the planted form with no mistake passes
    assert not _check_quantizer(_planted(scale_div=128.0))    # scale from the wrong code maximum
    assert not _check_quantizer(_planted(rounding=np.trunc))  # truncation instead of rounding
    assert not _check_quantizer(_planted(rounding=lambda r: np.floor(r + 0.5)))   # ties away from the even code
    assert not _check_quantizer(_planted(per_tensor=True))    # one scale for the whole tensor, not per row
    assert not _check_quantizer(_planted(signed_max=True))    # scale from the signed maximum
