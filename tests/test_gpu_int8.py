"""INT8 cache ([primer] 5.1, quantised cache): the CUDA path against the oracle.

* append: the code and scale of every stored row equal oracle.quant's for raw
  rows (both sides quantise the same bf16 values in fp32); with baked RoPE the
  two rotate with different sin/cos roundings, so codes may differ by one step;
* decode outputs element by element at small sizes (ring before, at and after
  the first wrap, no RoPE, baked and read-time; sink + ring, baked and
  read-time (raw keys dequantised and rotated at their in-cache positions);
  paged shared prefix; a
  single-sequence pool at head_dim 256 with NaN scales in its non-resident
  slots) and on sampled sequences of the full ring_int8 workload in the launch
  configuration bench.py times, against the oracle over the rows as the INT8
  cache stores them;
* kvc_decode_step's fused INT8 append over consecutive steps: outputs, and the
  cache it leaves equal to what kvc_append writes.
Tolerance: max abs error 2e-2 on the bf16 outputs, as for bf16 caches.
"""

import dataclasses

import numpy as np
import pytest
import torch

import bench
import kvc_synth
import oracle
from oracle.quant import dequantize_rows, quantize_rows
from tests.gpu_harness import TOL, attended, oracle_outputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import sliding_window_attention_kvc_gb300 as m
    return m


def _small(case):
    if case == "ring":
        return kvc_synth.make_workload("ring_int8", small=True)
    if case == "ring_none":
        return dataclasses.replace(kvc_synth.make_workload("ring_int8", small=True), rope="none")
    if case == "sink_baked":
        return kvc_synth.as_int8(kvc_synth.make_workload("sink_window_bf16", small=True), "sink_window_int8_small")
    if case == "sink_read":
        return kvc_synth.make_workload("sink_window_int8", small=True)
    if case == "ring_read":
        return dataclasses.replace(kvc_synth.make_workload("ring_int8", small=True), rope="read_time")
    if case == "ring_d256_read":
        return dataclasses.replace(kvc_synth.as_int8(kvc_synth.make_workload("ring_bf16", small=True),
                                                     "ring_int8_d256_small"), rope="read_time", head_dim=256,
                                   q_heads=8, kv_heads=2)
    if case == "paged":
        return kvc_synth.make_workload("paged_shared_prefix_int8", small=True)
    if case == "pool_d256":
        return kvc_synth.as_int8(kvc_synth.make_workload("long_context_pool_bf16", small=True),
                                 "long_context_pool_int8_small")
    raise ValueError(case)


CASES = ["ring", "ring_none", "sink_baked", "sink_read", "ring_read", "ring_d256_read", "paged", "pool_d256"]


def _maxerr(got, ref):
    return float(np.abs(np.asarray(got, dtype=np.float64) - ref).max())


@pytest.mark.parametrize("rope", ["none", "baked"])
def test_int8_append_codes_and_scales(kvc, rope):
    wl = dataclasses.replace(kvc_synth.make_workload("ring_int8", small=True), rope=rope)
    st = bench.DecodeState(wl, 1, source="cpu")
    codes, scales = kvc.int8_views(st.desc, st.cache)
    codes = codes[0].cpu().numpy()             # [2, B, Hkv, C, D]
    scales = scales[0].cpu().numpy()           # [2, B, Hkv, C]
    checked = 0
    for b in range(wl.batch):
        t = int(wl.positions[b])
        pos = attended(wl, b)
        pos = pos[pos < t]                      # the step's own token is appended by step()
        k, v = wl.kv_history(0, b, pos)
        k, v = k.double().numpy(), v.double().numpy()
        slots = oracle.window_slot(pos, wl.sinks, wl.window)
        for h in range(wl.kv_heads):
            gk, gsk = codes[0, b, h, slots], scales[0, b, h, slots]
            gv, gsv = codes[1, b, h, slots], scales[1, b, h, slots]
            cv, sv = quantize_rows(v[:, h])
            assert np.array_equal(gv, cv) and np.array_equal(gsv, sv), (b, h)
            if rope == "none":
                ck, sk = quantize_rows(k[:, h])
                assert np.array_equal(gk, ck) and np.array_equal(gsk, sk), (b, h)
            else:
                R = oracle.rotate(k[:, h], pos, wl.rope_base)
                ck, sk = quantize_rows(R)
                assert np.allclose(gsk, sk, rtol=2e-6, atol=0), (b, h)
                assert np.abs(gk.astype(np.int32) - ck.astype(np.int32)).max() <= 1, (b, h)
                assert (gk == ck).mean() > 0.99
                err = np.abs(dequantize_rows(gk, gsk) - R).max(axis=-1)
                assert (err <= gsk * (0.5 + 1e-3) + 1e-7).all(), (b, h)
            checked += len(pos)
    assert checked > 0
    assert kvc.get_error(st.ws) == 0


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("num_splits", [0, 1, 7])
def test_int8_decode_small_elementwise(kvc, case, num_splits):
    wl = _small(case)
    st = bench.DecodeState(wl, 1, source="cpu", num_splits=num_splits)
    got = st.step(0).float().cpu().numpy()
    ref = oracle_outputs(wl, 0)
    assert np.isfinite(got).all()
    err = _maxerr(got, ref)
    assert err <= TOL["i8"], (case, num_splits, err)
    assert kvc.get_error(st.ws) == 0


def test_int8_decode_full_size_sampled(kvc):
    """ring_int8 at full size, bench.py's launch configuration, sampled sequences."""
    wl = kvc_synth.make_workload("ring_int8")
    seqs = [0, 5, 7]
    st = bench.DecodeState(wl, 1, source="cpu")
    got = st.step(0).float().cpu().numpy()
    assert np.isfinite(got).all()
    ref = oracle_outputs(wl, 0, seqs=seqs)
    err = _maxerr(got[seqs], ref)
    assert err <= TOL["i8"], err
    assert kvc.get_error(st.ws) == 0


@pytest.mark.parametrize("case", ["ring", "sink_baked", "sink_read", "paged"])
def test_int8_decode_step_fused_append(kvc, case):
    """kvc_decode_step over consecutive positions: the fused INT8 append (in
    the decode kernel for ring layouts, in the plan kernel for paged) leaves
    the cache kvc_append writes, and the outputs match the oracle."""
    wl = _small(case)
    st = bench.DecodeState(wl, 1, source="cpu")
    ref_cache = st.cache.clone()
    for step in range(3 if wl.layout == "window" else 1):
        pos = wl.positions + step
        q = wl.queries(0, pos).contiguous().cuda()
        kn, vn = wl.new_kv(0, pos)
        kn, vn = kn.contiguous().cuda(), vn.contiguous().cuda()
        pos_t = torch.from_numpy(pos.astype(np.int32)).cuda()
        out = kvc.decode_step(st.desc, st.cache, 0, q, kn, vn, pos_t, st.ws, block_table=st.table,
                              valid_bits=st.valid_bits)
        kvc.append(st.desc, ref_cache, 0, kn, vn, pos_t, st.ws, block_table=st.table)
        got = out.float().cpu().numpy()
        ref = oracle_outputs(wl, 0, positions=pos)
        assert np.isfinite(got).all()
        assert _maxerr(got, ref) <= TOL["i8"], (case, step, _maxerr(got, ref))
        ca, sa = kvc.int8_views(st.desc, st.cache)
        cr, sr = kvc.int8_views(st.desc, ref_cache)
        dc = (ca.int() - cr.int()).abs()
        assert int(dc.max()) <= 1 and float((dc == 0).float().mean()) > 0.999
        both_nan = torch.isnan(sa) & torch.isnan(sr)
        ds = (sa - sr).abs().masked_fill(both_nan, 0.0)
        assert bool((ds <= sr.abs().masked_fill(both_nan, 0.0) * 2e-6).all())
    assert kvc.get_error(st.ws) == 0
