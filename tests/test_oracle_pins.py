"""Pins of the CPU oracle to what the pages and the mathematics fix.

Each `check_*` helper returns True when an implementation passes the pin; the
pin tests assert it for the oracle, and `test_planted_mistakes_fail_a_pin`
asserts that plausible mistakes planted in copies of oracle functions fail at
least one pin.  Sources: the pages' printed examples (tests/golden/*.json,
each citing its page and section), closed forms, torch's fp64
scaled_dot_product_attention, and brute force on tiny inputs.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import layouts, rope, storage
from oracle.attention import attend, decode_masked_history, decode_reference, decode_sequence

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# index arithmetic: ring, sinks, pages
# ---------------------------------------------------------------------------

def check_capacity4_letters(slot_fn) -> bool:
    g = _golden("ring_capacity4_letters.json")
    W = g["capacity"]
    for n, expect in g["slots_after"].items():
        slots = [None] * W
        for p, letter in enumerate(g["writes"][: int(n)]):
            s = int(slot_fn(p, 0, W))
            if not 0 <= s < W:
                return False
            slots[s] = letter
        if slots != expect:
            return False
    return True


def test_capacity4_ring_letters():
    assert check_capacity4_letters(layouts.window_slot)
    g = _golden("ring_capacity4_letters.json")
    ring = layouts.RingKV(g["capacity"])
    for p, letter in enumerate(g["writes"]):
        ring.append(letter, letter, p)
        if str(p + 1) in g["slots_after"]:
            assert ring.keys == g["slots_after"][str(p + 1)]


def check_demo_trace(attended_fn) -> bool:
    g = _golden("ring_w4_demo.json")
    return all(list(attended_fn(t, 0, g["window"])) == vis
               for t, vis in enumerate(g["visible_positions"]))


def test_ring_demo_trace_matches_page():
    g = _golden("ring_w4_demo.json")
    W = g["window"]
    ring = layouts.RingKV(W)
    stream = layouts.StreamingKV(0, W)
    phys = layouts.SinkRingKV(0, W)
    for t in range(g["steps"]):
        for model in (ring, stream, phys):
            model.append(None, None, t)
        assert [e["position"] for e in ring.visible()] == g["visible_positions"][t]
        assert [e["position"] for e in stream.visible()] == g["visible_positions"][t]
        assert [e["position"] for e in phys.visible()] == g["visible_positions"][t]
        assert ring.size == g["slots_used"][t]
    assert [e["position"] for e in ring.visible()] == g["final_positions"]
    assert [e["insert_seq"] for e in ring.visible()] == g["final_insert_seq"]
    assert check_demo_trace(layouts.window_attended)


def test_tenth_token_attends_7_to_10():
    case = _golden("window_examples.json")["cases"][0]
    assert list(layouts.window_attended(case["t"], 0, case["window"])) == case["attended"]


def test_window_boundary_against_ring_model():
    # [ring] 6: earliest visible is t-W+1; cover t < W and t >= W.
    for W in range(1, 9):
        ring = layouts.RingKV(W)
        for t in range(3 * W + 2):
            ring.append(None, None, t)
            got = layouts.window_attended(t, 0, W)
            assert list(got) == [e["position"] for e in ring.visible()]
            assert len(got) == min(t + 1, W)
            assert got[0] == max(0, t - W + 1) and got[-1] == t


def check_sink_set(attended_fn) -> bool:
    for S in (0, 1, 4):
        for W in (1, 2, 5, 8):
            model = layouts.StreamingKV(S, W)
            for t in range(3 * (S + W) + 3):
                model.append(None, None, t)
                if list(attended_fn(t, S, W)) != [e["position"] for e in model.visible()]:
                    return False
    return True


def test_sink_set_matches_streaming_model_and_equation():
    assert check_sink_set(layouts.window_attended)
    # [sink] cache-set equation with 4 sinks, once the window has slid past them.
    S, W = 4, 6
    for t in range(S + W, 40):
        got = set(layouts.window_attended(t, S, W))
        assert got == set(range(4)) | set(range(t - W + 1, t + 1))
        assert len(got) == S + W            # memory stays (4 + W) slots


def test_sink_ring_slot_map():
    for S in (0, 1, 4):
        for W in (1, 3, 7):
            C = S + W
            comp = layouts.StreamingKV(S, W)
            phys = layouts.SinkRingKV(S, W)
            for t in range(4 * C):
                comp.append(None, None, t)
                phys.append(None, None, t)
                assert int(layouts.window_slot(t, S, W)) == phys.slot_of(t)
                cv, pv = comp.visible(), phys.visible()
                assert [e["position"] for e in cv] == [e["position"] for e in pv]
                if t < C:   # before the first wrap: slot order is chronological order
                    assert [e["slot"] for e in pv] == list(range(t + 1))


def check_incache(incache_fn) -> bool:
    for S in (0, 4):
        for W in (3, 7):
            comp = layouts.StreamingKV(S, W)
            for t in range(4 * (S + W)):
                comp.append(None, None, t)
                vis = comp.visible()
                pos = np.array([e["position"] for e in vis])
                if list(incache_fn(pos, t, S, W)) != [e["incache"] for e in vis]:
                    return False
                if int(incache_fn(t, t, S, W)) != len(vis) - 1:
                    return False
    return True


def test_incache_positions_match_compacted_cache():
    assert check_incache(layouts.incache_position)


def check_paged(attended_fn) -> bool:
    """The attended set of a paged sequence against the block-pool model
    (mapped and resident blocks, positions up to t) on random tables with
    unmapped entries and non-resident blocks."""
    rng = np.random.default_rng(0)
    bs, maxb, nb = 4, 6, 20
    for trial in range(20):
        table = np.full((2, maxb), -1)
        phys = rng.permutation(nb)[: 2 * maxb].reshape(2, maxb)
        keep = rng.random((2, maxb)) < 0.8
        table[keep] = phys[keep]
        valid = rng.random(nb) < 0.6
        pool = layouts.PagedKV(nb, bs, table, valid)
        for b in range(2):
            for p in range(bs * maxb):
                if table[b][p // bs] >= 0:
                    pool.append(b, None, None, p)
            for t in range(bs * maxb):
                got = attended_fn(t, table[b], valid, bs)
                if list(got) != [e["position"] for e in pool.visible(b, t)]:
                    return False
    return True


def test_paged_attended_matches_pool_model():
    assert check_paged(layouts.paged_attended)


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def check_rope(rotate_fn, inv_freq_fn) -> bool:
    ok = np.allclose(inv_freq_fn(4, 10000.0), [1.0, 0.01], rtol=1e-15, atol=0)
    for p in (0, 1, 2, 7, 1000, 262143):
        # D = 2, theta_0 = 1: a counter-clockwise rotation by p radians.
        ok &= np.allclose(rotate_fn(np.array([1.0, 0.0]), p), [math.cos(p), math.sin(p)], atol=1e-12)
        ok &= np.allclose(rotate_fn(np.array([0.0, 1.0]), p), [-math.sin(p), math.cos(p)], atol=1e-12)
    # rotate-half pairing: dim i mixes only with dim i + D/2, at angle p * theta_i.
    D = 8
    th = 10000.0 ** (-2.0 * np.arange(D // 2) / D)
    for i in range(D // 2):
        e = np.zeros(D)
        e[i] = 1.0
        y = rotate_fn(e, 5)
        expect = np.zeros(D)
        expect[i], expect[i + D // 2] = math.cos(5 * th[i]), math.sin(5 * th[i])
        ok &= np.allclose(y, expect, atol=1e-12)
    return bool(ok)


def test_rope_closed_forms():
    assert check_rope(rope.rotate, rope.inv_freq)
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 128))
    assert np.array_equal(rope.rotate(x, 0), x)
    assert np.allclose(np.linalg.norm(rope.rotate(x, 12345), axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    assert np.allclose(rope.rotate(rope.rotate(x, 300), 4000), rope.rotate(x, 4300), atol=1e-11)


def test_rope_scores_depend_only_on_distance():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for a, b in ((10, 3), (70000, 65536), (999999, 995908)):
        ref = rope.rotate(q, a) @ rope.rotate(k, b)
        for d in (1, 17, 4096, 250000):
            assert abs(rope.rotate(q, a + d) @ rope.rotate(k, b + d) - ref) < 1e-9
        assert abs(q @ rope.rotate(k, b - a) - ref) < 1e-9


# ---------------------------------------------------------------------------
# storage rounding
# ---------------------------------------------------------------------------

def check_round_bf16(round_fn) -> bool:
    """Round-to-nearest-even to bf16: torch's fp32 -> bf16 conversion on fp32
    values over 17 decades, and the tie cases written out."""
    rng = np.random.default_rng(3)
    x32 = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    ok = np.array_equal(round_fn(x32.astype(np.float64)), ref)
    # ties go to the even significand
    ok &= round_fn(1 + 2.0 ** -8) == 1.0
    ok &= round_fn(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    ok &= round_fn(-(1 + 2.0 ** -8)) == -1.0
    ok &= round_fn(0.0) == 0.0
    return bool(ok)


def test_round_bf16_matches_torch_on_fp32_values():
    assert check_round_bf16(storage.round_bf16)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def _sdpa(q, K, V, scale=None):
    """torch fp64 SDPA for q [Hq, D], K/V [n, Hkv, D] (one query position)."""
    qt = torch.from_numpy(np.asarray(q, dtype=np.float64))[None, :, None, :]
    kt = torch.from_numpy(np.asarray(K, dtype=np.float64)).permute(1, 0, 2)[None]
    vt = torch.from_numpy(np.asarray(V, dtype=np.float64)).permute(1, 0, 2)[None]
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale, enable_gqa=True)
    return out[0, :, 0, :].numpy()


def check_attention(seq_fn) -> bool:
    rng = np.random.default_rng(4)
    ok = True
    for Hq, Hkv, D, n in ((4, 1, 64, 37), (8, 2, 128, 300), (16, 4, 32, 5), (3, 3, 16, 1)):
        q = rng.standard_normal((Hq, D))
        K = rng.standard_normal((n, Hkv, D)) * 2
        V = rng.standard_normal((n, Hkv, D))
        got = seq_fn(q, K, V, np.arange(n), n - 1, rope="none")
        ok &= np.allclose(got, _sdpa(q, K, V), rtol=0, atol=1e-12)
    return bool(ok)


def test_attention_matches_torch_sdpa_fp64():
    assert check_attention(decode_sequence)


def test_softmax_weights_sum_to_one():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((4, 64))
    K = rng.standard_normal((500, 64)) * 3
    V = rng.standard_normal((500, 64))
    _, A = attend(q, K, V, 1 / 8)
    for h in range(4):
        assert abs(math.fsum(A[h].tolist()) - 1.0) < 1e-14
        assert (A[h] >= 0).all()


def test_special_cases():
    rng = np.random.default_rng(6)
    D = 64
    q = rng.standard_normal((4, D))
    v0 = rng.standard_normal((1, D))
    # t = 0: the only attended token is the new one, out = v_0 exactly.
    for mode in ("none", "baked", "read_time"):
        out = decode_reference(q, rng.standard_normal((1, D)), v0, [0], 0, rope=mode, sinks=4, window=60)
        assert np.array_equal(out, np.repeat(v0, 4, axis=0))
    # K = 0: uniform weights, out = mean of V over the attended set.
    n = 77
    V = rng.standard_normal((n, D))
    out = decode_reference(q, np.zeros((n, D)), V, np.arange(n), n - 1)
    assert np.allclose(out, V.mean(axis=0)[None], rtol=0, atol=1e-14)
    # W >= t + 1: the window changes nothing, plain causal attention.
    t = 20
    K = rng.standard_normal((t + 1, 1, D))
    V = rng.standard_normal((t + 1, 1, D))
    pos = layouts.window_attended(t, 0, t + 1)
    got = decode_sequence(q, K[pos], V[pos], pos, t, rope="none")
    assert np.allclose(got, _sdpa(q, K, V), atol=1e-12)


def _brute(q, hist_k, hist_v, visible, t, mode, S, W, base=10000.0):
    """Direct triple loop over scalars: rotate, score, softmax, weighted sum."""
    D = len(q)
    half = D // 2

    def rot(x, p):
        y = [0.0] * D
        for i in range(half):
            a = p * base ** (-2.0 * i / D)
            y[i] = x[i] * math.cos(a) - x[i + half] * math.sin(a)
            y[i + half] = x[i] * math.sin(a) + x[i + half] * math.cos(a)
        return y

    def shift(p):
        return p if p < S else p - max(0, t - (S + W) + 1)

    if mode == "baked":
        qq = rot(q, t)
        keys = [[float(storage.round_storage(x, "f32")) for x in rot(hist_k[p], p)] for p in visible]
    elif mode == "read_time":
        qq = rot(q, shift(t))
        keys = [rot(hist_k[p], shift(p)) for p in visible]
    else:
        qq = list(q)
        keys = [list(hist_k[p]) for p in visible]
    scores = [sum(qq[d] * k[d] for d in range(D)) / math.sqrt(D) for k in keys]
    m = max(scores)
    e = [math.exp(s - m) for s in scores]
    z = sum(e)
    return [sum(e[j] / z * hist_v[p][d] for j, p in enumerate(visible)) for d in range(D)]


def test_brute_force_tiny_window_layouts():
    rng = np.random.default_rng(7)
    D = 4
    for S, W in ((0, 4), (1, 3), (4, 4), (2, 6)):
        T = 3 * (S + W) + 2
        hk = rng.standard_normal((T, D))
        hv = rng.standard_normal((T, D))
        model = layouts.SinkRingKV(S, W)
        for t in range(T):
            model.append(hk[t], hv[t], t)
            q = rng.standard_normal(D)
            vis = [e["position"] for e in model.visible()]
            for mode in ("none", "baked", "read_time"):
                ref = _brute(q, hk, hv, vis, t, mode, S, W)
                got = decode_reference(q[None], hk[vis], hv[vis], vis, t, rope=mode,
                                       storage="f32", sinks=S, window=W)[0]
                assert np.allclose(got, ref, rtol=0, atol=1e-12), (S, W, t, mode)


def test_brute_force_tiny_paged():
    rng = np.random.default_rng(8)
    D, bs, maxb, nb = 4, 2, 4, 8
    table = np.array([[5, -1, 2, 7], [0, 3, -1, 6]])
    valid = np.array([1, 1, 1, 0, 1, 1, 1, 1], dtype=bool)
    pool = layouts.PagedKV(nb, bs, table, valid)
    hk = rng.standard_normal((2, bs * maxb, D))
    hv = rng.standard_normal((2, bs * maxb, D))
    for b in range(2):
        for p in range(bs * maxb):
            if table[b][p // bs] >= 0:
                pool.append(b, hk[b, p], hv[b, p], p)
        for t in range(bs * maxb):
            vis = [e["position"] for e in pool.visible(b, t)]
            if not vis:
                continue
            q = rng.standard_normal(D)
            ref = _brute(q, hk[b], hv[b], vis, t, "baked", 0, 1 << 30)
            got = decode_reference(q[None], hk[b][vis], hv[b][vis], vis, t, rope="baked", storage="f32")[0]
            assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_layout_model_and_masked_history_agree_bit_exactly():
    rng = np.random.default_rng(9)
    D = 16
    for S, W in ((0, 5), (4, 6), (2, 3)):
        T = 4 * (S + W)
        hk = storage.round_bf16(rng.standard_normal((T, D)))
        hv = storage.round_bf16(rng.standard_normal((T, D)))
        model = layouts.SinkRingKV(S, W)
        for t in range(T):
            model.append(hk[t], hv[t], t)
            q = rng.standard_normal((3, D))
            vis = model.visible()
            # physical slot order, not chronological: the sum must not care
            vis_phys = sorted(vis, key=lambda e: e["slot"])
            pos = np.array([e["position"] for e in vis_phys])
            K = np.array([e["key"] for e in vis_phys])
            V = np.array([e["value"] for e in vis_phys])
            mask = np.zeros(t + 1, dtype=bool)
            mask[layouts.window_attended(t, S, W)] = True
            for mode in ("none", "baked", "read_time"):
                spec = dict(rope=mode, storage="bf16", sinks=S, window=W)
                a = decode_reference(q, K, V, pos, t, **spec)
                b = decode_masked_history(q, hk[: t + 1], hv[: t + 1], t, mask, **spec)
                assert np.array_equal(a, b), (S, W, t, mode)


def test_paged_with_mask_equals_contiguous_resident_attention():
    # [pool]: masked blocks behave as if absent; output equals attention over the
    # resident set of the contiguous history, bit for bit.
    rng = np.random.default_rng(10)
    D, bs, nlog, pool_n = 32, 8, 12, 9
    t = nlog * bs - 3
    hk = storage.round_bf16(rng.standard_normal((t + 1, D)))
    hv = storage.round_bf16(rng.standard_normal((t + 1, D)))
    resident = np.sort(rng.choice(nlog, size=pool_n, replace=False))
    table = np.full((1, nlog), -1)
    table[0, resident] = rng.permutation(pool_n)
    valid = rng.random(pool_n) < 0.6
    pool = layouts.PagedKV(pool_n, bs, table, valid)
    for p in range(t + 1):
        if table[0][p // bs] >= 0:
            pool.append(0, hk[p], hv[p], p)
    vis = sorted(pool.visible(0, t), key=lambda e: (e["block"], e["row"]))   # pool order
    pos = np.array([e["position"] for e in vis])
    q = rng.standard_normal((4, D))
    a = decode_reference(q, np.array([e["key"] for e in vis]), np.array([e["value"] for e in vis]),
                         pos, t, rope="baked", storage="bf16")
    mask = np.zeros(t + 1, dtype=bool)
    mask[layouts.paged_attended(t, table[0], valid, bs)] = True
    b = decode_masked_history(q, hk, hv, t, mask, rope="baked", storage="bf16")
    assert np.array_equal(a, b)
    # fully masked sequence: empty attended set, zeros
    z = decode_masked_history(q, hk, hv, t, np.zeros(t + 1, dtype=bool))
    assert np.array_equal(z, np.zeros_like(q))


def test_read_time_equals_baked_before_the_shift():
    rng = np.random.default_rng(11)
    D, S, W = 64, 4, 20
    for t in (0, 5, S + W - 1):
        pos = layouts.window_attended(t, S, W)
        q = rng.standard_normal((2, D))
        K = rng.standard_normal((len(pos), D))
        V = rng.standard_normal((len(pos), D))
        a = decode_reference(q, K, V, pos, t, rope="read_time", sinks=S, window=W, storage="f32")
        b = decode_reference(q, K, V, pos, t, rope="baked", sinks=S, window=W, storage="f32")
        assert np.allclose(a, b, atol=1e-6)


# ---------------------------------------------------------------------------
# planted mistakes (in copies of oracle functions, on the CPU)
# ---------------------------------------------------------------------------

def test_rope_by_slot_instead_of_position_is_caught():
    # [ring] 3.4 and 6: using the physical slot as the RoPE position is wrong
    # once the ring has wrapped.
    rng = np.random.default_rng(12)
    D, W = 32, 8
    for t, wrapped in ((5, False), (29, True)):
        pos = layouts.window_attended(t, 0, W)
        K = rng.standard_normal((len(pos), D))
        V = rng.standard_normal((len(pos), D))
        q = rng.standard_normal((2, D))
        right = decode_reference(q, K, V, pos, t, rope="baked", storage="f32")
        slots = layouts.window_slot(pos, 0, W)
        wrong = decode_reference(q, K, V, slots, int(layouts.window_slot(t, 0, W)), rope="baked", storage="f32")
        assert (np.abs(right - wrong).max() > 1e-3) == wrapped


def test_planted_mistakes_fail_a_pin():
    # window off by one (t - W instead of t - W + 1)
    def attended_off_by_one(t, S, W):
        return np.concatenate([np.arange(0, min(S, t + 1)), np.arange(max(S, t - W), t + 1)])
    assert not check_demo_trace(attended_off_by_one)
    assert not check_sink_set(attended_off_by_one)

    # ring slot from the wrong modulus
    assert not check_capacity4_letters(lambda p, S, W: p % (W + 1))

    # sinks not pinned in the in-cache shift
    assert not check_incache(lambda p, t, S, W: np.asarray(p) - max(0, t - (S + W) + 1))

    # RoPE: wrong sign, interleaved pairing, wrong frequency exponent
    def rot_sign(x, pos, base=10000.0):
        return rope.rotate(x, -np.asarray(pos), base)

    def rot_interleaved(x, pos, base=10000.0):
        x = np.asarray(x, dtype=np.float64)
        D = x.shape[-1]
        th = base ** (-2.0 * np.arange(D // 2) / D)
        a = np.asarray(pos, dtype=np.float64)[..., None] * th
        y = np.empty_like(x)
        y[..., 0::2] = x[..., 0::2] * np.cos(a) - x[..., 1::2] * np.sin(a)
        y[..., 1::2] = x[..., 0::2] * np.sin(a) + x[..., 1::2] * np.cos(a)
        return y

    def freq_wrong(D, base=10000.0):
        return base ** (-np.arange(D // 2) / D)

    assert not check_rope(rot_sign, rope.inv_freq)
    assert not check_rope(rot_interleaved, rope.inv_freq)
    assert not check_rope(rope.rotate, freq_wrong)

    # attention: missing 1/sqrt(D), wrong GQA grouping, softmax without max
    # subtraction overflowing is not a plausible silent error; transposed V is.
    def no_scale(q, K, V, pos, t, **kw):
        return decode_sequence(q, K, V, pos, t, scale=1.0, **kw)

    def gqa_modulo(q, K, V, pos, t, **kw):
        q = np.asarray(q)
        Hq, Hkv = q.shape[0], K.shape[1]
        out = np.empty_like(q, dtype=np.float64)
        for h in range(Hq):
            out[h] = decode_reference(q[h:h + 1], K[:, h % Hkv], V[:, h % Hkv], pos, t, **kw)[0]
        return out

    def v_wrong_head(q, K, V, pos, t, **kw):
        return decode_sequence(q, K, V[:, ::-1], pos, t, **kw)

    assert not check_attention(no_scale)
    assert not check_attention(gqa_modulo)
    assert not check_attention(v_wrong_head)


def test_planted_paged_and_rounding_mistakes_fail_a_pin():
    # paged attended set: residency ignored, the whole block of t attended,
    # unmapped entries read as physical block 0
    def ignores_valid(t, row, valid, bs):
        return layouts.paged_attended(t, row, np.ones_like(valid), bs)

    def whole_last_block(t, row, valid, bs):
        end = (t // bs + 1) * bs
        return np.array([p for p in range(end) if row[p // bs] >= 0 and valid[row[p // bs]]], dtype=np.int64)

    def unmapped_as_block0(t, row, valid, bs):
        return layouts.paged_attended(t, np.where(np.asarray(row) < 0, 0, row), valid, bs)

    for fn in (ignores_valid, whole_last_block, unmapped_as_block0):
        assert not check_paged(fn), fn.__name__

    # bf16 storage: truncation toward zero, ties away from zero
    def bits(x):
        return np.atleast_1d(np.asarray(x, dtype=np.float64)).astype(np.float32).view(np.uint32)

    def from_bits(u, like):
        out = (u & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
        return out if np.ndim(like) else float(out[0])

    def truncate(x):
        return from_bits(bits(x), x)

    def ties_away(x):
        return from_bits(bits(x) + np.uint32(0x8000), x)

    for fn in (truncate, ties_away):
        assert not check_round_bf16(fn), fn.__name__


def check_read_time(decode_fn) -> bool:
    """[sink] "RoPE cache position shifting", written out: keep the compacting
    StreamingLLM cache of (key, value) pairs, rotate each kept key at its index
    in that cache and the query at the last index, and take fp64 SDPA. The
    read-time decode over the same attended positions must match, before and
    long after the cache first shifts (S = 0 and S = 4)."""
    rng = np.random.default_rng(21)
    D, n = 16, 60
    K_all, V_all = rng.standard_normal((n, D)), rng.standard_normal((n, D))
    q = rng.standard_normal((2, D))
    ok = True
    for S, W in ((4, 7), (0, 9)):
        comp = layouts.StreamingKV(S, W)
        for t in range(n):
            comp.append(K_all[t], V_all[t], t)
            kept = comp.visible()
            Kr = rope.rotate(np.stack([e["key"] for e in kept]), np.arange(len(kept)))
            V = np.stack([e["value"] for e in kept])
            ref = _sdpa(rope.rotate(q, len(kept) - 1), Kr[:, None, :], V[:, None, :])
            pos = np.array([e["position"] for e in kept])
            got = decode_fn(q, K_all[pos], V_all[pos], pos, t, rope="read_time", storage="f32", sinks=S, window=W)
            ok &= bool(np.allclose(got, ref, rtol=0, atol=1e-12))
    return ok


def test_read_time_rope_equals_attention_over_the_compacted_cache():
    assert check_read_time(decode_reference)
    # the layout-model route: one kv head, K and V [n, 1, D]
    assert check_read_time(lambda q, K, V, pos, t, **kw: decode_sequence(q, K[:, None], V[:, None], pos, t, **kw))


def test_planted_read_time_mistakes_fail_a_pin():
    def q_at_absolute(q, K, V, positions, t, *, sinks, window, **kw):
        # keys at their in-cache positions, the query left at t
        ip = layouts.incache_position(positions, t, sinks, window)
        out, _ = attend(rope.rotate(q, t), rope.rotate(K, ip), V, 1.0 / math.sqrt(q.shape[-1]))
        return out

    def keys_at_absolute(q, K, V, positions, t, *, sinks, window, **kw):
        # the query at its in-cache position, keys left at their absolute positions
        iq = int(layouts.incache_position(t, t, sinks, window))
        out, _ = attend(rope.rotate(q, iq), rope.rotate(K, positions), V, 1.0 / math.sqrt(q.shape[-1]))
        return out

    for fn in (q_at_absolute, keys_at_absolute):
        assert not check_read_time(fn), fn.__name__


def check_baked_shift_invariance(decode_fn) -> bool:
    """Baked RoPE scores depend only on t - p ([primer] 4.5, [pool] rows
    rotated at their absolute positions): moving every attended position and
    t by the same offset leaves the output unchanged, and at distance 0 from
    the query a key scores as without RoPE.  Tolerance 1e-6: keys are stored
    as fp32 after rotation (relative rounding 2^-24), so the output moves by
    ~3e-8 with the angles; a misplaced rotation moves it by O(1)."""
    rng = np.random.default_rng(22)
    D = 32
    q = rng.standard_normal((3, D))
    K, V = rng.standard_normal((9, D)), rng.standard_normal((9, D))
    pos = np.array([0, 3, 4, 5, 9, 10, 11, 12, 13])
    base = decode_fn(q, K, V, pos, 13, rope="baked", storage="f32")
    ok = True
    for shift in (1, 1000, 262131, 999986):
        got = decode_fn(q, K, V, pos + shift, 13 + shift, rope="baked", storage="f32")
        ok &= bool(np.allclose(got, base, rtol=0, atol=1e-6))
    one = decode_fn(q, K[-1:], V[-1:], pos[-1:], 13, rope="baked", storage="f32")
    ok &= bool(np.allclose(one, V[-1:].repeat(3, axis=0), rtol=0, atol=1e-12))   # a single key: its value
    two = decode_fn(q, K[-2:], V[-2:], pos[-2:] + 500, 513, rope="baked", storage="f32")
    ok &= bool(np.allclose(two, decode_fn(q, rope.rotate(K[-2:], [-1, 0]), V[-2:], pos[-2:], 13, rope="none",
                                          storage="f32"), rtol=0, atol=1e-6))
    return ok


def test_baked_rope_depends_only_on_distance():
    assert check_baked_shift_invariance(decode_reference)


def test_planted_baked_mistakes_fail_a_pin():
    def q_unrotated(q, K, V, positions, t, **kw):
        out, _ = attend(np.asarray(q, dtype=np.float64), rope.rotate(K, positions), V, 1.0 / math.sqrt(q.shape[-1]))
        return out if kw.get("rope") == "baked" else decode_reference(q, K, V, positions, t, **kw)

    def keys_reversed(q, K, V, positions, t, **kw):
        if kw.get("rope") != "baked":
            return decode_reference(q, K, V, positions, t, **kw)
        out, _ = attend(rope.rotate(q, t), rope.rotate(K, t - np.asarray(positions)), V, 1.0 / math.sqrt(q.shape[-1]))
        return out

    for fn in (q_unrotated, keys_reversed):
        assert not check_baked_shift_invariance(fn), fn.__name__
