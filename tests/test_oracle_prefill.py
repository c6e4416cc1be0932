"""Pins of the chunked-prefill oracle (oracle.prefill) against torch's
scaled_dot_product_attention in fp64 with an explicit mask (the window as a
mask on the score matrix, [ring] 3.1 / 5.2), causal attention as the special
case of a window no shorter than the history, and the relative-position form
of read-time RoPE."""

import numpy as np
import pytest
import torch

from oracle import attention, layouts, prefill, rope, storage


def _sdpa_masked(q, K, V, mask):
    """q [T, D], K/V [N, D], mask [T, N] bool -> [T, D], torch fp64."""
    out = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, None], torch.from_numpy(K)[None, None], torch.from_numpy(V)[None, None],
        attn_mask=torch.from_numpy(mask)[None, None])
    return out[0, 0].numpy()


def _case(layout, rng):
    T, Hq, Hkv, D = 11, 4, 2, 16
    if layout == "ring":
        S, W, pos0 = 0, 9, 14
    elif layout == "sink":
        S, W, pos0 = 3, 7, 13
    else:
        S, W, pos0 = 0, 0, 21
    N = pos0 + T
    q = rng.standard_normal((T, Hq, D))
    K = rng.standard_normal((N, Hkv, D))
    V = rng.standard_normal((N, Hkv, D))
    if layout == "paged":
        bs, nb = 4, 16
        table = rng.permutation(nb)[:(N + bs - 1) // bs].astype(np.int64)
        table[2] = -1
        valid = rng.random(nb) < 0.7
        for lb in range(pos0 // bs, len(table)):           # the chunk's own blocks are mapped and valid
            if table[lb] < 0:
                table[lb] = nb - 1 - lb
            valid[table[lb]] = True
        att = lambda t: layouts.paged_attended(t, table, valid, bs)
    else:
        att = lambda t: layouts.window_attended(t, S, W)
    return T, Hq, Hkv, D, S, W, pos0, q, K, V, att


@pytest.mark.parametrize("layout", ["ring", "sink", "paged"])
@pytest.mark.parametrize("rope_mode", ["none", "baked"])
def test_prefill_matches_masked_sdpa(layout, rope_mode):
    rng = np.random.default_rng(30)
    T, Hq, Hkv, D, S, W, pos0, q, K, V, att = _case(layout, rng)
    got = prefill.prefill_sequence(q, K, V, pos0, att, rope=rope_mode, sinks=S, window=W)
    N = K.shape[0]
    g = Hq // Hkv
    mask = np.zeros((T, N), dtype=bool)
    for i in range(T):
        mask[i, att(pos0 + i)] = True
    t_rows = pos0 + np.arange(T)
    for h in range(Hq):
        kv = h // g
        qh, Kh = q[:, h], K[:, kv]
        if rope_mode == "baked":            # K is stored rotated, in the storage type (fp32 here)
            qh = rope.rotate(qh, t_rows)
            Kh = storage.round_storage(rope.rotate(Kh, np.arange(N)), "f32")
        want = _sdpa_masked(qh, Kh, V[:, kv], mask)
        assert np.allclose(got[:, h], want, rtol=0, atol=1e-12), (layout, rope_mode, h)


def test_prefill_from_zero_with_a_long_window_is_causal_attention():
    rng = np.random.default_rng(31)
    T, D = 12, 8
    q, K, V = (rng.standard_normal((T, 1, D)) for _ in range(3))
    got = prefill.prefill_sequence(q, K, V, 0, lambda t: layouts.window_attended(t, 0, 64))
    want = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q[:, 0])[None, None], torch.from_numpy(K[:, 0])[None, None],
        torch.from_numpy(V[:, 0])[None, None], is_causal=True)[0, 0].numpy()
    assert np.allclose(got[:, 0], want, rtol=0, atol=1e-12)


def test_prefill_read_time_rope_is_relative_to_each_token():
    # read-time RoPE: a window key sits at distance t - p from the query, a
    # sink key at min(t, C-1) - p ([sink] "RoPE cache position shifting"); the
    # scores are those of R(distance) q against the raw key
    rng = np.random.default_rng(32)
    T, Hq, Hkv, D, S, W, pos0, q, K, V, att = _case("sink", rng)
    C = S + W
    got = prefill.prefill_sequence(q, K, V, pos0, att, rope="read_time", sinks=S, window=W)
    g = Hq // Hkv
    for i in range(T):
        t = pos0 + i
        ps = att(t)
        for h in range(Hq):
            kv = h // g
            dist = np.where(ps < S, min(t, C - 1) - ps, t - ps)
            s = np.array([np.dot(rope.rotate(q[i, h], d), K[p, kv]) for d, p in zip(dist, ps)]) / np.sqrt(D)
            w = np.exp(s - s.max())
            want = (w / w.sum()) @ V[ps, kv]
            assert np.allclose(got[i, h], want, rtol=0, atol=1e-10), (i, h)


def test_chunks_compose_and_one_token_chunk_is_a_decode_step():
    rng = np.random.default_rng(33)
    T, Hq, Hkv, D, S, W, pos0, q, K, V, att = _case("ring", rng)
    spec = dict(rope="baked", sinks=S, window=W, storage="bf16")
    whole = prefill.prefill_sequence(q, K, V, pos0, att, **spec)
    a = prefill.prefill_sequence(q[:5], K, V, pos0, att, **spec)
    b = prefill.prefill_sequence(q[5:], K, V, pos0 + 5, att, **spec)
    assert np.array_equal(whole, np.concatenate([a, b]))
    t = pos0 + 3
    ps = att(t)
    one = attention.decode_sequence(q[3], K[ps], V[ps], ps, t, **spec)
    assert np.array_equal(whole[3], one)


def test_left_padding_rows_are_zero():
    rng = np.random.default_rng(34)
    T, D = 6, 8
    q, K, V = (rng.standard_normal((T, 1, D)) for _ in range(3))
    got = prefill.prefill_sequence(q, K, V, -2, lambda t: layouts.window_attended(t, 0, 4))
    assert not got[:2].any()
    want = prefill.prefill_sequence(q[2:], K, V, 0, lambda t: layouts.window_attended(t, 0, 4))
    assert np.array_equal(got[2:], want)


# ---------------------------------------------------------------------------
# planted mistakes (in copies of the prefill oracle, on the CPU): each fails
# the masked-SDPA pin for some layout and RoPE mode
# ---------------------------------------------------------------------------

def _check_prefill(pfn) -> bool:
    """test_prefill_matches_masked_sdpa for a prefill function pfn; False on the first failure."""
    for layout in ("ring", "sink", "paged"):
        for rope_mode in ("none", "baked"):
            rng = np.random.default_rng(30)
            T, Hq, Hkv, D, S, W, pos0, q, K, V, att = _case(layout, rng)
            got = pfn(q, K, V, pos0, att, rope=rope_mode, sinks=S, window=W)
            N, g = K.shape[0], Hq // Hkv
            mask = np.zeros((T, N), dtype=bool)
            for i in range(T):
                mask[i, att(pos0 + i)] = True
            t_rows = pos0 + np.arange(T)
            for h in range(Hq):
                qh, Kh = q[:, h], K[:, h // g]
                if rope_mode == "baked":
                    qh = rope.rotate(qh, t_rows)
                    Kh = storage.round_storage(rope.rotate(Kh, np.arange(N)), "f32")
                if not np.allclose(got[:, h], _sdpa_masked(qh, Kh, V[:, h // g], mask), rtol=0, atol=1e-12):
                    return False
    return True


def _planted_prefill(mistake):
    """A copy of the prefill oracle with one mistake planted ("none": a faithful copy)."""
    def pfn(q_chunk, K_hist, V_hist, pos0, attended, **spec):
        T = q_chunk.shape[0]
        out = np.zeros_like(q_chunk, dtype=np.float64)
        for i in range(T):
            t = pos0 + i
            ps = np.asarray(attended(t), dtype=np.int64)
            qi = q_chunk[i]
            if mistake == "causal_off_by_one":           # the next token is visible too
                nxt = np.asarray(attended(t + 1), dtype=np.int64)
                ps = nxt[nxt <= min(t + 1, K_hist.shape[0] - 1)]
            elif mistake == "rope_at_pos0" and spec.get("rope") == "baked":
                qi = rope.rotate(qi, pos0 - t)            # with the rotation at t: q rotated at pos0
            elif mistake == "no_chunk_keys":              # the chunk's own rows left out (self kept)
                ps = ps[(ps < pos0) | (ps == t)]
            elif mistake == "one_window_per_chunk":       # the last token's set for every token
                last = np.asarray(attended(pos0 + T - 1), dtype=np.int64)
                ps = last[last <= t]
            out[i] = attention.decode_sequence(qi, K_hist[ps], V_hist[ps], ps, t, **spec)
        return out
    return pfn


@pytest.mark.parametrize("mistake", ["causal_off_by_one", "rope_at_pos0", "no_chunk_keys", "one_window_per_chunk"])
def test_planted_prefill_mistakes_fail_the_pin(mistake):
    assert _check_prefill(prefill.prefill_sequence)
    assert _check_prefill(_planted_prefill("none"))
    assert not _check_prefill(_planted_prefill(mistake))
