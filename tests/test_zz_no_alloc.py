"""kvc_decode_attention_noalloc against kvc_decode_attention.

The no-allocation entry point serves callers that cannot call cudaMalloc once
they are running (a serving loop with device memory fixed at start-up, a
plugin inside a framework that owns all device memory): it keeps its split-K
partials, counters and work plan in the library's own fixed scratch array
instead of a caller workspace.  These tests call it through the C ABI twice in
a row (the second call finds the scratch as the first left it), and in an
interleaved order of workloads with different layouts, batches and split
counts, and check every output against the ordinary entry point on the same
inputs: within the tolerances of the other GPU tests, and bit for bit, since
both run the same kernels.  It sits in its own file, collected last,
and passes both alone in a fresh process and after the other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

import bench
import kvc_synth
from tests.gpu_harness import TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import sliding_window_attention_kvc_gb300 as m
    return m


def _noalloc(kvc, st, out):
    d = st.desc
    rc = kvc.lib().kvc_decode_attention_noalloc(
        ctypes.byref(d), st.cache.data_ptr(), 0, st.q[0].data_ptr(), st.pos.data_ptr(),
        st.table.data_ptr() if st.table is not None else None,
        st.valid_bits.data_ptr() if st.valid_bits is not None else None,
        out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, kvc.strerror(rc)


NAMES = ["ring_bf16", "sink_window_bf16", "paged_shared_prefix_bf16", "long_context_pool_bf16"]


def _workspace_reference(kvc, st):
    """The ordinary entry point (caller workspace) on the same inputs, after
    the step's token was appended."""
    st.step(0)
    return kvc.decode_attention(st.desc, st.cache, 0, st.q[0], st.pos, st.ws, block_table=st.table,
                                valid_bits=st.valid_bits).clone()


def _check(kvc, st, ref, name):
    out = torch.full_like(st.out, float("nan"))
    _noalloc(kvc, st, out)
    torch.cuda.synchronize()
    got = out.float()
    assert torch.isfinite(got).all(), name
    err = float((got - ref.float()).abs().max())
    assert err <= TOL[st.wl.dtype], (name, err)
    # the same kernels on the same inputs: nothing may leak through the scratch
    assert torch.equal(out, ref), name


@pytest.mark.parametrize("name", NAMES)
def test_noalloc_matches_workspace_entry_point_twice(kvc, name):
    wl = kvc_synth.make_workload(name, small=True)
    st = bench.DecodeState(wl, 1, source="cpu")
    ref = _workspace_reference(kvc, st)
    for _ in range(2):
        _check(kvc, st, ref, name)


def test_noalloc_calls_of_different_layouts_interleaved(kvc):
    """Each call finds the scratch as a call of another layout, batch and split
    count left it (partials, plan and counters at other offsets)."""
    states = {}
    for name in NAMES:
        st = bench.DecodeState(kvc_synth.make_workload(name, small=True), 1, source="cpu")
        states[name] = (st, _workspace_reference(kvc, st))
    order = ["paged_shared_prefix_bf16", "ring_bf16", "paged_shared_prefix_bf16", "sink_window_bf16",
             "long_context_pool_bf16", "ring_bf16", "long_context_pool_bf16", "paged_shared_prefix_bf16"]
    for name in order:
        st, ref = states[name]
        _check(kvc, st, ref, name)


def test_noalloc_rejects_problems_larger_than_the_scratch(kvc):
    # a workspace of more than KVC_NOALLOC_SCRATCH_BYTES: refused before any launch
    d = kvc.make_desc("ring", "baked", "bf16", 1, 4096, 64, 8, 256, window=65536, num_splits=64)
    assert kvc.workspace_bytes(d) > kvc.KVC_NOALLOC_SCRATCH_BYTES
    A = 1 << 20   # never dereferenced: the size check comes first
    rc = kvc.lib().kvc_decode_attention_noalloc(ctypes.byref(d), A, 0, A, A, None, None, A, None)
    assert rc == kvc.KVC_ERR_TOO_LARGE
    assert "scratch" in kvc.strerror(rc)
