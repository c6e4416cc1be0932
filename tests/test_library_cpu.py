"""Host-side checks that need no GPU: the library builds and loads, exports
every entry point of include/kvc.h, and validates its arguments before any
CUDA call; host logic of the binding and the benchmark."""

import ctypes
import os
import re
import subprocess

import numpy as np
import pytest
import torch

import bench
import kvc_synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvc():
    import __graft_entry__
    __graft_entry__.build()
    import sliding_window_attention_kvc_gb300 as m
    return m


def _declared():
    with open(os.path.join(ROOT, "include", "kvc.h")) as f:
        src = f.read()
    return re.findall(r"KVC_API\s+[\w\s\*]+?\b(kvc_\w+)\s*\(", src)


def test_header_declares_the_abi():
    names = _declared()
    for n in ("kvc_append", "kvc_decode_attention", "kvc_block_table_write", "kvc_get_error",
              "kvc_cache_bytes", "kvc_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(kvc):
    L = kvc.lib()
    for name in _declared():
        assert hasattr(L, name), name
    assert set(_declared()) == set(kvc.ABI_FUNCTIONS)
    nm = subprocess.run(["nm", "-D", "--defined-only", kvc.LIB_PATH], capture_output=True, text=True)
    if nm.returncode == 0:
        exported = {ln.split()[-1] for ln in nm.stdout.splitlines() if " T " in ln}
        assert set(_declared()) <= exported
        assert not [s for s in exported if s.startswith("cuda")], "CUDA runtime symbols leak out"


def _header_without_comments():
    with open(os.path.join(ROOT, "include", "kvc.h")) as f:
        src = f.read()
    return re.sub(r"//[^\n]*", "", re.sub(r"/\*.*?\*/", "", src, flags=re.S))


def test_binding_types_match_the_header(kvc):
    """Every ctypes signature of the binding has the header's parameter count,
    widths and pointer-ness, and the descriptor mirrors `kvc_desc` field by
    field: a mismatch would pass the wrong bits through the ABI silently."""
    src = _header_without_comments()
    L = kvc.lib()
    scalar = {"int32_t": ctypes.c_int32, "size_t": ctypes.c_size_t, "int": ctypes.c_int, "float": ctypes.c_float}
    decls = re.findall(r"KVC_API\s+([\w\s\*]+?)\b(kvc_\w+)\s*\(([^)]*)\)\s*;", src)
    assert {name for _, name, _ in decls} == set(kvc.ABI_FUNCTIONS)
    for ret, name, params in decls:
        fn = getattr(L, name)
        ps = [" ".join(p.split()) for p in params.split(",") if p.strip()]
        assert fn.argtypes is not None and len(fn.argtypes) == len(ps), (name, ps, fn.argtypes)
        for p, t in zip(ps, fn.argtypes):
            ctype = p.rsplit(" ", 1)[0].replace("const ", "").strip()
            if "*" in p:
                if ctype.startswith("kvc_desc"):
                    assert t is ctypes.POINTER(kvc.KvcDesc), (name, p)
                else:
                    assert t is ctypes.c_void_p, (name, p, t)
            else:
                assert ctypes.sizeof(t) == ctypes.sizeof(scalar[ctype]) and t is not ctypes.c_void_p, (name, p, t)
        ret = " ".join(ret.split())
        want = {"int": ctypes.c_int, "size_t": ctypes.c_size_t, "const char*": ctypes.c_char_p,
                "void": None, "kvc_pager*": ctypes.c_void_p}[ret]
        assert fn.restype is want, (name, ret, fn.restype)
    body = re.search(r"typedef struct\s*(?:\w+\s*)?\{(.*?)\}\s*kvc_desc\s*;", src, re.S).group(1)
    fields = re.findall(r"(int32_t|float)\s+(\w+)\s*;", body)
    assert [(n, scalar[t]) for t, n in fields] == list(kvc.KvcDesc._fields_)


def test_sizes_above_2gib_come_back_whole(kvc):
    """size_t results (cache, workspace and prefill workspace bytes) pass
    through the binding without truncation to 32 bits."""
    d = kvc.make_desc("paged", "baked", "bf16", 1, 4096, 32, 8, 128, block_size=16, num_blocks=1 << 20,
                      max_blocks_per_seq=4096)
    assert kvc.cache_bytes(d) == 2 * (1 << 20) * 8 * 16 * 128 * 2 > 2 ** 32
    assert kvc.workspace_bytes(d) > 0
    assert kvc.prefill_workspace_bytes(d, 256) > 2 ** 32


def test_missing_library_fails_loudly(kvc, monkeypatch):
    """Without libkvc.so every call raises: there is no CPU fallback."""
    monkeypatch.setattr(kvc, "_lib", None)
    monkeypatch.setattr(kvc, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libkvc.so"))
    with pytest.raises(RuntimeError, match="not built"):
        kvc.lib()
    with pytest.raises(RuntimeError, match="not built"):
        kvc.cache_bytes(_desc(kvc))


def _desc(kvc, **kw):
    base = dict(layout="ring", rope="baked", dtype="bf16", layers=2, batch=3, q_heads=8, kv_heads=2,
                head_dim=128, window=100)
    base.update(kw)
    return kvc.make_desc(**base)


def test_cache_and_workspace_sizes(kvc):
    for name in kvc_synth.WORKLOAD_NAMES:
        wl = kvc_synth.make_workload(name)
        d = bench.workload_desc(wl, layers=2)
        n = int(np.prod(wl.cache_shape(2)))
        if wl.dtype == "i8":      # codes, then one fp32 scale per row
            assert kvc.cache_bytes(d) == n + 4 * (n // wl.head_dim)
        else:
            assert kvc.cache_bytes(d) == n * (4 if wl.dtype == "f32" else 2)
        assert kvc.workspace_bytes(d) > 0
        assert tuple(kvc.cache_shape(d)) == wl.cache_shape(2)


def test_invalid_descriptors_are_rejected(kvc):
    bad = [
        dict(head_dim=96),                    # unsupported head_dim
        dict(q_heads=6, kv_heads=4),          # not a multiple
        dict(window=0),
        dict(layout="sink_ring", sinks=0),
        dict(layout="ring", sinks=2),
        dict(layout="paged", block_size=0, num_blocks=4, max_blocks_per_seq=4),
        dict(layers=0),
        dict(dtype="i8", head_dim=64),                       # INT8: whole 128-byte column blocks
        dict(dtype="i8", layout="paged", rope="read_time", block_size=16, num_blocks=4,
             max_blocks_per_seq=4),                          # paged: no read-time RoPE
        dict(dtype="i8", batch=1, kv_heads=1, window=98),    # INT8: rows of a half not a multiple of 4
    ]
    for kw in bad:
        assert kvc.cache_bytes(_desc(kvc, **kw)) == 0, kw
        assert kvc.workspace_bytes(_desc(kvc, **kw)) == 0, kw
    L = kvc.lib()
    assert L.kvc_cache_bytes(None) == 0


def _documented_cache_bytes(f):
    """The cache size include/kvc.h documents for descriptor fields f, or 0
    where the documented constraints reject it."""
    layout, rope, dtype = f["layout"], f["rope"], f["dtype"]
    if min(f["layers"], f["batch"], f["q_heads"], f["kv_heads"]) < 1 or f["q_heads"] % f["kv_heads"]:
        return 0
    if f["head_dim"] not in (64, 128, 256) or f["num_splits"] < 0 or f["softmax_scale"] < 0:
        return 0
    g = f["q_heads"] // f["kv_heads"]
    pairs = f["q_heads"] // (4 if g % 4 == 0 else 2 if g % 2 == 0 else 1)
    if f["batch"] > 65535 or pairs > 65535 or f["batch"] * pairs >= 2 ** 31:
        return 0
    if rope != 0 and not f["rope_base"] > 0:
        return 0
    if layout == 2:                                   # PAGED
        if min(f["block_size"], f["num_blocks"], f["max_blocks_per_seq"]) < 1 or rope == 2:
            return 0
        rows = f["num_blocks"] * f["kv_heads"] * f["block_size"]
    else:
        if f["window"] < 1 or (layout == 0 and f["sinks"] != 0) or (layout == 1 and f["sinks"] < 1):
            return 0
        rows = f["batch"] * f["kv_heads"] * (f["sinks"] + f["window"])
    if dtype == 2 and (f["head_dim"] < 128 or rows % 4):
        return 0
    elems = f["layers"] * 2 * rows * f["head_dim"]
    if dtype == 2:
        return elems + 4 * f["layers"] * 2 * rows     # codes, then one fp32 scale per row
    return elems * (4 if dtype == 0 else 2)


def test_launch_grid_limits(kvc):
    """Descriptors past the launch-grid limits of include/kvc.h are rejected
    up front; those at the limits are accepted."""
    L = kvc.lib()

    def size(batch, q_heads, kv_heads):
        d = kvc.make_desc("ring", "none", "bf16", 1, batch, q_heads, kv_heads, 64, window=1)
        return L.kvc_cache_bytes(ctypes.byref(d))

    assert size(1, 4 * 65535, 1) > 0                  # 65535 groups of 4 q heads
    assert size(1, 4 * 65536, 1) == 0
    assert size(1, 65535, 65535) > 0                  # one q head per kv head
    assert size(1, 2 * 65536, 65536) == 0
    assert size(65535, 8, 2) > 0 and size(65536, 8, 2) == 0
    assert size(32768, 4 * 65535, 1) > 0              # 2^31 - 32768 units
    assert size(32769, 4 * 65535, 1) == 0             # past 2^31


def test_random_descriptors_follow_the_documented_rules(kvc):
    # seeded random descriptors around the boundaries of every documented rule
    rng = np.random.default_rng(2024)
    L = kvc.lib()
    pick = lambda *v: v[int(rng.integers(len(v)))]

    def field(good, bad):                             # a valid value 85% of the time
        return pick(*good) if rng.random() < 0.85 else pick(*bad)

    accepted = 0
    for _ in range(3000):
        f = dict(layout=pick(0, 1, 2), rope=pick(0, 1, 2), dtype=pick(0, 1, 2), layers=field((1, 2, 3), (0,)),
                 batch=field((1, 2, 5), (0,)), kv_heads=field((1, 2, 3), (0,)),
                 head_dim=field((64, 128, 256), (32, 96)), window=field((1, 7, 64, 100), (-1, 0)),
                 sinks=pick(-1, 0, 0, 1, 4), block_size=field((1, 16, 64), (0,)), num_blocks=field((1, 3, 8), (0,)),
                 max_blocks_per_seq=field((1, 4), (0,)), num_splits=field((0, 3), (-1,)),
                 rope_base=field((10000.0, 500.0), (-1.0, 0.0)), softmax_scale=field((0.0, 0.125), (-0.5,)))
        f["q_heads"] = max(f["kv_heads"], 1) * pick(1, 2, 4) + (1 if rng.random() < 0.1 else 0)
        d = kvc.KvcDesc(f["layout"], f["rope"], f["dtype"], f["layers"], f["batch"], f["q_heads"], f["kv_heads"],
                        f["head_dim"], f["window"], f["sinks"], f["block_size"], f["num_blocks"],
                        f["max_blocks_per_seq"], f["num_splits"], f["rope_base"], f["softmax_scale"])
        want = _documented_cache_bytes(f)
        assert L.kvc_cache_bytes(ctypes.byref(d)) == want, f
        assert (L.kvc_workspace_bytes(ctypes.byref(d)) > 0) == (want > 0), f
        accepted += want > 0
    assert 100 < accepted < 2900                      # both sides of the rules were exercised


def test_argument_errors_return_codes_without_launching(kvc):
    L = kvc.lib()
    d = _desc(kvc)
    ws_n = kvc.workspace_bytes(d)
    A = 1 << 20   # fake, 16-byte aligned "device" addresses: never dereferenced on these paths
    dp = ctypes.byref(d)
    assert L.kvc_append(dp, None, 0, A, A, 1, A, None, A, ws_n, None) == kvc.KVC_ERR_NULL
    assert L.kvc_append(dp, A + 8, 0, A, A, 1, A, None, A, ws_n, None) == kvc.KVC_ERR_ALIGN
    assert L.kvc_append(dp, A, 5, A, A, 1, A, None, A, ws_n, None) == kvc.KVC_ERR_ARG
    assert L.kvc_append(dp, A, 0, A, A, 0, A, None, A, ws_n, None) == kvc.KVC_ERR_ARG
    assert L.kvc_append(dp, A, 0, A, A, 1, A, None, A, ws_n - 1, None) == kvc.KVC_ERR_WORKSPACE
    assert L.kvc_decode_attention(dp, A, 0, A, A, None, None, A + 4, A, ws_n, None) == kvc.KVC_ERR_ALIGN
    assert L.kvc_decode_attention(dp, A, -1, A, A, None, None, A, A, ws_n, None) == kvc.KVC_ERR_ARG
    assert L.kvc_decode_attention(dp, A, 0, None, A, None, None, A, A, ws_n, None) == kvc.KVC_ERR_NULL
    dpg = _desc(kvc, layout="paged", rope="baked", block_size=16, num_blocks=10, max_blocks_per_seq=4)
    nws = kvc.workspace_bytes(dpg)
    assert L.kvc_decode_attention(ctypes.byref(dpg), A, 0, A, A, None, None, A, A, nws, None) == kvc.KVC_ERR_NULL
    dpr = _desc(kvc, layout="paged", rope="read_time", block_size=16, num_blocks=10, max_blocks_per_seq=4)
    assert L.kvc_decode_attention(ctypes.byref(dpr), A, 0, A, A, A, None, A, A, 1 << 30, None) == \
        kvc.KVC_ERR_UNSUPPORTED
    assert L.kvc_block_table_write(dp, A, None, 1, A, A, A, A, ws_n, None) == kvc.KVC_ERR_DESC
    assert L.kvc_block_table_write(ctypes.byref(dpg), A, None, 0, None, None, None, None, 0, None) == kvc.KVC_OK
    assert L.kvc_get_error(None, None) == kvc.KVC_ERR_NULL
    assert kvc.strerror(kvc.KVC_ERR_ALIGN).startswith("pointer")
    # block manager: paged descriptors only, pointers checked, nothing launched
    dg = ctypes.byref(dpg)
    assert L.kvc_block_prepare(dp, A, A, A, None, A, A, A, A, ws_n, None) == kvc.KVC_ERR_DESC
    assert L.kvc_block_prepare(dg, A, A, None, None, A, A, A, A, nws, None) == kvc.KVC_ERR_NULL
    assert L.kvc_block_prepare(dg, A + 8, A, A, None, A, A, A, A, nws, None) == kvc.KVC_ERR_ALIGN
    assert L.kvc_block_prepare(dg, A, A, A, None, A, A, A, A, nws - 1, None) == kvc.KVC_ERR_WORKSPACE
    deep = _desc(kvc, layout="paged", rope="baked", layers=128, q_heads=256, kv_heads=256, block_size=16,
                 num_blocks=10, max_blocks_per_seq=4)   # 128 * 2 * 256 copy rows: past the launch grid
    assert L.kvc_block_prepare(ctypes.byref(deep), A, A, A, None, A, A, A, A, 1 << 40, None) == \
        kvc.KVC_ERR_UNSUPPORTED
    assert L.kvc_block_share(dg, A, A, -1, A, A, A, A, nws, None) == kvc.KVC_ERR_ARG
    assert L.kvc_block_share(dg, A, A, 0, None, None, None, None, 0, None) == kvc.KVC_OK
    assert L.kvc_block_share(dg, A, A, 1, A, None, A, A, nws, None) == kvc.KVC_ERR_NULL
    assert L.kvc_block_release(dg, A, None, A, A, A, -1, A, A, nws, None) == kvc.KVC_ERR_ARG
    assert L.kvc_block_release(dg, A, None, A, A, None, 1, A, A, nws, None) == kvc.KVC_ERR_NULL
    assert "free" in kvc.strerror(kvc.KVC_DEV_NO_FREE_BLOCK)
    # chunked prefill: bf16 and INT8 caches (fp32 refused), head_dim 64 / 128 / 256; a
    # head_dim 256 paged cache needs blocks that pack a 64-key tile, an INT8 cache
    # a chunk no longer than its window; sizes checked first
    pw = kvc.prefill_workspace_bytes(d, 16)
    assert pw > ws_n and kvc.prefill_workspace_bytes(d, 0) == 0
    assert L.kvc_prefill(dp, A, 0, A, A, A, 0, A, None, None, A, A, pw, None) == kvc.KVC_ERR_ARG
    assert L.kvc_prefill(dp, A, 0, A, A, A, 16, A, None, None, A, A, pw - 1, None) == kvc.KVC_ERR_WORKSPACE
    assert L.kvc_prefill(dp, A, 0, None, A, A, 16, A, None, None, A, A, pw, None) == kvc.KVC_ERR_NULL
    df = _desc(kvc, dtype="f32")
    assert L.kvc_prefill(ctypes.byref(df), A, 0, A, A, A, 16, A, None, None, A, A, 1 << 30, None) == \
        kvc.KVC_ERR_UNSUPPORTED
    d8 = _desc(kvc, dtype="i8", window=8)             # 3 * 2 * 8 rows per half: a multiple of 4
    assert L.kvc_prefill(ctypes.byref(d8), A, 0, A, A, A, 16, A, None, None, A, A, 1 << 30, None) == \
        kvc.KVC_ERR_UNSUPPORTED
    d256p = _desc(kvc, head_dim=256, layout="paged", rope="baked", block_size=12, num_blocks=10,
                  max_blocks_per_seq=4)
    assert L.kvc_prefill(ctypes.byref(d256p), A, 0, A, A, A, 16, A, A, None, A, A, 1 << 30, None) == \
        kvc.KVC_ERR_UNSUPPORTED


def test_decode_arguments_are_checked_before_anything_is_issued(kvc):
    """With no GPU any launch or copy fails with KVC_ERR_CUDA, so getting the
    argument's own error code shows nothing was issued before the check: the
    fp32 step's append, the no-allocation call's scratch clear."""
    L = kvc.lib()
    A = 1 << 20   # fake, 16-byte aligned "device" addresses: never dereferenced on these paths
    for dtype in ("f32", "bf16"):
        d = _desc(kvc, dtype=dtype)
        dp, n = ctypes.byref(d), kvc.workspace_bytes(d)
        step = lambda cache=A, layer=0, q=A, pos=A, out=A, ws=A, ws_n=n: L.kvc_decode_step(
            dp, cache, layer, q, A, A, pos, None, None, out, ws, ws_n, None)
        assert step(q=None) == kvc.KVC_ERR_NULL
        assert step(out=None) == kvc.KVC_ERR_NULL
        assert step(ws=None) == kvc.KVC_ERR_NULL
        assert step(out=A + 4) == kvc.KVC_ERR_ALIGN
        assert step(ws=A + 8) == kvc.KVC_ERR_ALIGN
        assert step(layer=2) == kvc.KVC_ERR_ARG
        assert step(ws_n=n - 1) == kvc.KVC_ERR_WORKSPACE
        noalloc = lambda q=A, out=A, layer=0: L.kvc_decode_attention_noalloc(dp, A, layer, q, A, None, None, out,
                                                                             None)
        assert noalloc(q=None) == kvc.KVC_ERR_NULL
        assert noalloc(out=A + 2) == kvc.KVC_ERR_ALIGN
        assert noalloc(layer=-1) == kvc.KVC_ERR_ARG
    dpg = _desc(kvc, layout="paged", rope="baked", block_size=16, num_blocks=10, max_blocks_per_seq=4)
    assert L.kvc_decode_attention_noalloc(ctypes.byref(dpg), A, 0, A, A, None, None, A, None) == kvc.KVC_ERR_NULL


def test_int8_views_cover_the_buffer(kvc):
    d = _desc(kvc, dtype="i8", window=100)
    buf = torch.zeros(kvc.cache_bytes(d), dtype=torch.uint8)
    codes, scales = kvc.int8_views(d, buf)
    assert codes.dtype == torch.int8 and tuple(codes.shape) == tuple(kvc.cache_shape(d))
    assert scales.dtype == torch.float32 and tuple(scales.shape) == tuple(kvc.cache_shape(d))[:-1]
    assert codes.numel() + 4 * scales.numel() == buf.numel()
    scales.fill_(1.5)
    codes.fill_(-3)
    assert int(buf[:codes.numel()].view(torch.int8).min()) == -3
    assert float(buf[codes.numel():].view(torch.float32).max()) == 1.5
    assert kvc.desc_dtype(d) == torch.bfloat16 and kvc.cache_dtype(d) == torch.uint8


def test_pack_valid_bits(kvc):
    rng = np.random.default_rng(0)
    for n in (1, 31, 32, 33, 1024, 1000):
        m = rng.random(n) < 0.5
        w = kvc.pack_valid_bits(torch.from_numpy(m)).numpy().view(np.uint32)
        for k in range(n):
            assert bool((w[k // 32] >> (k % 32)) & 1) == bool(m[k])


def test_step_bytes_formula():
    # KV bytes per token: 2 (K and V) x layers x kv_heads x head_dim x element bytes;
    # the pages' example (32 layers, 32 heads, D 128, FP16) is 524288 bytes.
    import json
    with open(os.path.join(ROOT, "tests", "golden", "window_examples.json")) as f:
        ex = json.load(f)["kv_bytes_per_token"]
    wl = kvc_synth.Workload(name="x", layout="window", dtype="bf16", rope="none", batch=1,
                            q_heads=ex["kv_heads"], kv_heads=ex["kv_heads"], head_dim=ex["head_dim"],
                            window=10, positions=[0])
    per_layer = bench.step_bytes(wl)["kv_logical"]      # t = 0: one attended token, one layer
    assert per_layer * ex["layers"] == ex["bytes"]
    wl = kvc_synth.make_workload("ring_bf16")
    assert bench.step_bytes(wl)["kv_logical"] == 8 * 8 * 4096 * 2 * 128 * 2      # 128 MiB
    wl = kvc_synth.make_workload("paged_shared_prefix_bf16")
    nb = bench.step_bytes(wl)
    assert nb["kv_unique"] < nb["kv_logical"]


@pytest.mark.parametrize("name", ["tiny_ring_sink_f32", "ring_bf16", "sink_window_bf16", "paged_shared_prefix_bf16",
                                  "long_context_pool_bf16", "ring_int8"])
def test_step_bytes_match_the_oracle_attended_sets(name):
    # the roofline's algorithmic bytes, recounted from the oracle's attended
    # sets: logical = every (sequence, attended position); unique (paged) =
    # the distinct (physical block, row) pairs those positions read
    import oracle
    wl = kvc_synth.make_workload(name)
    row = wl.kv_heads * 2 * (wl.head_dim * wl.elt_bytes + wl.row_scale_bytes)
    logical, cells = 0, set()
    for b in range(wl.batch):
        t = int(wl.positions[b])
        if wl.layout == "window":
            ps = oracle.window_attended(t, wl.sinks, wl.window)
        else:
            ps = oracle.paged_attended(t, wl.block_table[b], wl.valid, wl.block_size)
            phys = wl.block_table[b][ps // wl.block_size]
            cells.update(zip(phys.tolist(), (ps % wl.block_size).tolist()))
        logical += len(ps)
    nb = bench.step_bytes(wl)
    assert nb["kv_logical"] == logical * row
    assert nb["kv_unique"] == (logical if wl.layout == "window" else len(cells)) * row


def test_binding_refuses_buffers_smaller_than_the_descriptor(kvc):
    """The library sees only addresses, so the binding checks sizes: a cache
    tensor below kvc_cache_bytes, or a host page-in buffer too short for the
    listed blocks, raises before anything is passed on."""
    z = lambda n, dt=torch.bfloat16: torch.zeros(n, dtype=dt)
    for dtype in ("f32", "bf16", "i8"):
        d = _desc(kvc, dtype=dtype, window=104)
        short = z(kvc.cache_bytes(d) - 1, torch.uint8).view(torch.uint8)
        with pytest.raises(ValueError, match="cache holds"):
            kvc.decode_step(d, short, 0, z(1), z(1), z(1), z(1, torch.int32), z(1, torch.uint8))
        with pytest.raises(ValueError, match="cache holds"):
            kvc.decode_attention(d, short, 0, z(1), z(1, torch.int32), z(1, torch.uint8))
        with pytest.raises(ValueError, match="cache holds"):
            kvc.append(d, short, 0, z(1), z(1), z(1, torch.int32), z(1, torch.uint8))
        with pytest.raises(ValueError, match="cache holds"):
            kvc.prefill(d, short, 0, z(1), z(1), z(1), z(1, torch.int32), z(1, torch.uint8))
    dp = _desc(kvc, layout="paged", rope="baked", layers=2, block_size=16, num_blocks=8, max_blocks_per_seq=32)
    with pytest.raises(ValueError, match="cache holds"):
        kvc.block_prepare(dp, z(10), z(1, torch.int32), None, z(1, torch.uint8))
    pg = kvc.Pager(8)
    per_block = 2 * 2 * 2 * 16 * 128 * 2                # layers, K|V, kv heads, rows, D, bf16
    with pytest.raises(ValueError, match="host_kv holds"):
        pg.issue(dp, z(1), z(4 * per_block // 2 - 1), [(0, 1), (3, 2)], None)
    pg.close()
