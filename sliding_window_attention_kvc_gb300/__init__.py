"""Decode-step KV-cache attention on GB300: Python binding of libkvc.so.

Thin ctypes wrappers with the names of the C ABI in include/kvc.h.  They only
marshal arguments (torch tensors -> device pointers, the current CUDA stream)
and raise `KvcError` on a non-zero status; every step of the computation runs
in the library's CUDA kernels.  There is no CPU fallback: if libkvc.so is
missing or cannot be loaded, every call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvc.so")

LAYOUTS = {"ring": 0, "sink_ring": 1, "paged": 2}
ROPES = {"none": 0, "baked": 1, "read_time": 2}
DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.int8: 2}
DTYPE_NAMES = {"f32": torch.float32, "bf16": torch.bfloat16, "i8": torch.int8}
KVC_I8 = 2

KVC_OK = 0
KVC_ERR_NULL, KVC_ERR_DESC, KVC_ERR_UNSUPPORTED = -1, -2, -3
KVC_ERR_ALIGN, KVC_ERR_WORKSPACE, KVC_ERR_ARG, KVC_ERR_CUDA = -4, -5, -6, -7
KVC_ERR_TOO_LARGE = -8
KVC_NOALLOC_SCRATCH_BYTES = 8 << 20
KVC_DEV_BAD_BLOCK, KVC_DEV_UNMAPPED_APPEND, KVC_DEV_BAD_POSITION = 0x1, 0x2, 0x4
KVC_DEV_TIMEOUT, KVC_DEV_BAD_ENTRY = 0x8, 0x10
KVC_DEV_INTERNAL, KVC_DEV_NO_FREE_BLOCK = 0x20, 0x40

ABI_FUNCTIONS = (
    "kvc_cache_bytes", "kvc_workspace_bytes", "kvc_workspace_init", "kvc_append",
    "kvc_decode_attention", "kvc_block_table_write", "kvc_valid_write", "kvc_get_error",
    "kvc_strerror", "kvc_decode_attention_noalloc", "kvc_decode_step",
    "kvc_block_prepare", "kvc_block_share", "kvc_block_release",
    "kvc_pager_create", "kvc_pager_destroy", "kvc_pager_plan", "kvc_pager_evict", "kvc_pagein_issue",
    "kvc_pagein_commit", "kvc_prefill_workspace_bytes", "kvc_prefill",
)


class KvcDesc(ctypes.Structure):
    """Mirror of `kvc_desc` in include/kvc.h."""
    _fields_ = [
        ("layout", ctypes.c_int32), ("rope", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("layers", ctypes.c_int32), ("batch", ctypes.c_int32), ("q_heads", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("window", ctypes.c_int32),
        ("sinks", ctypes.c_int32), ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32), ("num_splits", ctypes.c_int32),
        ("rope_base", ctypes.c_float), ("softmax_scale", ctypes.c_float),
    ]


class KvcError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: kvc status {code} ({strerror(code)})")


_lib = None


def lib() -> ctypes.CDLL:
    """Load libkvc.so (built in-tree by build.py); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} not built: run sliding_window_attention_kvc_gb300/build.py "
                               "(or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        dp = ctypes.POINTER(KvcDesc)
        L.kvc_cache_bytes.argtypes = [dp]
        L.kvc_cache_bytes.restype = sz
        L.kvc_workspace_bytes.argtypes = [dp]
        L.kvc_workspace_bytes.restype = sz
        L.kvc_workspace_init.argtypes = [dp, vp, sz, vp]
        L.kvc_append.argtypes = [dp, vp, i32, vp, vp, i32, vp, vp, vp, sz, vp]
        L.kvc_decode_attention.argtypes = [dp, vp, i32, vp, vp, vp, vp, vp, vp, sz, vp]
        L.kvc_block_table_write.argtypes = [dp, vp, vp, i32, vp, vp, vp, vp, sz, vp]
        L.kvc_valid_write.argtypes = [dp, vp, i32, vp, vp, vp, sz, vp]
        L.kvc_get_error.argtypes = [vp, vp]
        L.kvc_decode_attention_noalloc.argtypes = [dp, vp, i32, vp, vp, vp, vp, vp, vp]
        L.kvc_decode_step.argtypes = [dp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.kvc_prefill_workspace_bytes.argtypes = [dp, i32]
        L.kvc_prefill_workspace_bytes.restype = sz
        L.kvc_prefill.argtypes = [dp, vp, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp, sz, vp]
        L.kvc_block_prepare.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.kvc_block_share.argtypes = [dp, vp, vp, i32, vp, vp, vp, vp, sz, vp]
        L.kvc_block_release.argtypes = [dp, vp, vp, vp, vp, vp, i32, vp, vp, sz, vp]
        L.kvc_pager_create.argtypes = [i32]
        L.kvc_pager_create.restype = vp
        L.kvc_pager_destroy.argtypes = [vp]
        L.kvc_pager_destroy.restype = None
        L.kvc_pager_plan.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        L.kvc_pager_evict.argtypes = [dp, i32, i32, vp, vp, vp, vp, vp]
        L.kvc_pagein_issue.argtypes = [vp, dp, vp, vp, i32, vp, vp, vp, vp]
        L.kvc_pagein_commit.argtypes = [vp, dp, i32, i32, vp, vp, vp, vp, vp]
        L.kvc_strerror.argtypes = [ctypes.c_int]
        L.kvc_strerror.restype = ctypes.c_char_p
        for name in ABI_FUNCTIONS:
            if name not in ("kvc_cache_bytes", "kvc_workspace_bytes", "kvc_prefill_workspace_bytes", "kvc_strerror",
                            "kvc_pager_create", "kvc_pager_destroy"):
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def strerror(code: int) -> str:
    try:
        return lib().kvc_strerror(int(code)).decode()
    except Exception:  # the library itself is unavailable
        return "unknown"


def make_desc(layout: str, rope: str, dtype, layers: int, batch: int, q_heads: int, kv_heads: int,
              head_dim: int, window: int = 0, sinks: int = 0, block_size: int = 0, num_blocks: int = 0,
              max_blocks_per_seq: int = 0, num_splits: int = 0, rope_base: float = 10000.0,
              softmax_scale: float = 0.0) -> KvcDesc:
    if isinstance(dtype, str):
        dtype = DTYPE_NAMES[dtype]
    return KvcDesc(LAYOUTS[layout], ROPES[rope], DTYPES[dtype], layers, batch, q_heads, kv_heads, head_dim,
                   window, sinks, block_size, num_blocks, max_blocks_per_seq, num_splits,
                   float(rope_base), float(softmax_scale))


def desc_dtype(d: KvcDesc) -> torch.dtype:
    """Element type of q, out, k_new and v_new (bf16 for an INT8 cache)."""
    return torch.float32 if d.dtype == 0 else torch.bfloat16


def cache_dtype(d: KvcDesc) -> torch.dtype:
    """Element type of the cache tensor: fp32, bf16, or bytes (uint8) for an
    INT8 cache, whose buffer holds the codes followed by the fp32 row scales."""
    return {0: torch.float32, 1: torch.bfloat16}.get(d.dtype, torch.uint8)


def cache_shape(d: KvcDesc) -> tuple:
    """[layers, 2, batch, kv_heads, sinks + window, D] or [layers, 2, num_blocks, kv_heads, block_size, D]."""
    if d.layout == LAYOUTS["paged"]:
        return (d.layers, 2, d.num_blocks, d.kv_heads, d.block_size, d.head_dim)
    return (d.layers, 2, d.batch, d.kv_heads, d.window + d.sinks, d.head_dim)


def cache_bytes(d: KvcDesc) -> int:
    return int(lib().kvc_cache_bytes(ctypes.byref(d)))


def workspace_bytes(d: KvcDesc) -> int:
    return int(lib().kvc_workspace_bytes(ctypes.byref(d)))


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, what: str):
    if rc != 0:
        raise KvcError(rc, what)


def _need(t: torch.Tensor, name: str, dtype=None, numel=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")


def _need_cache(d: KvcDesc, cache: torch.Tensor):
    """The cache tensor: the descriptor's element type and at least
    kvc_cache_bytes(d) bytes (the library sees only its address)."""
    need = cache_bytes(d)
    if isinstance(cache, torch.Tensor) and cache.numel() * cache.element_size() < need:
        raise ValueError(f"cache holds {cache.numel() * cache.element_size()} bytes, the descriptor needs {need}")
    _need(cache, "cache", cache_dtype(d))


def alloc_cache(d: KvcDesc, device="cuda", fill=None) -> torch.Tensor:
    """Caller-owned cache tensor of the layout's shape (uninitialised unless `fill`).

    INT8 cache: a flat uint8 tensor of kvc_cache_bytes(d) bytes (`int8_views`
    gives its codes and scales); `fill` sets every code and scale to
    rint(fill) and fill, or NaN scales when fill is NaN."""
    shape = cache_shape(d)
    if d.dtype == KVC_I8:
        buf = torch.empty(cache_bytes(d), dtype=torch.uint8, device=device)
        if fill is not None:
            codes, scales = int8_views(d, buf)
            codes.fill_(0 if fill != fill else int(round(fill)))
            scales.fill_(fill)
        return buf
    if fill is None:
        return torch.empty(shape, dtype=desc_dtype(d), device=device)
    return torch.full(shape, fill, dtype=desc_dtype(d), device=device)


def int8_views(d: KvcDesc, cache: torch.Tensor):
    """(codes int8 [cache_shape], scales fp32 [cache_shape[:-1]]) views of an INT8 cache buffer."""
    shape = cache_shape(d)
    n = 1
    for x in shape:
        n *= x
    codes = cache[:n].view(torch.int8).view(shape)
    scales = cache[n:n + 4 * (n // shape[-1])].view(torch.float32).view(shape[:-1])
    return codes, scales


def alloc_workspace(d: KvcDesc, device="cuda") -> torch.Tensor:
    """Zero-filled workspace of kvc_workspace_bytes(d) bytes."""
    n = workspace_bytes(d)
    if n == 0:
        raise KvcError(KVC_ERR_DESC, "kvc_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def workspace_init(d: KvcDesc, workspace: torch.Tensor, stream=None):
    _need(workspace, "workspace", torch.uint8)
    _check(lib().kvc_workspace_init(ctypes.byref(d), _ptr(workspace), workspace.numel(), _stream(stream)),
           "kvc_workspace_init")


def append(d: KvcDesc, cache: torch.Tensor, layer: int, k_new: torch.Tensor, v_new: torch.Tensor,
           pos: torch.Tensor, workspace: torch.Tensor, block_table: torch.Tensor | None = None, stream=None):
    """kvc_append: k_new / v_new [batch, n_new, kv_heads, D] (or [batch, kv_heads, D] for one token)."""
    dt = desc_dtype(d)
    _need_cache(d, cache)
    _need(k_new, "k_new", dt)
    _need(v_new, "v_new", dt)
    _need(pos, "pos", torch.int32, d.batch)
    _need(workspace, "workspace", torch.uint8)
    per_tok = d.kv_heads * d.head_dim
    if k_new.numel() % (d.batch * per_tok) or v_new.numel() != k_new.numel():
        raise ValueError("k_new / v_new must be [batch, n_new, kv_heads, head_dim]")
    n_new = k_new.numel() // (d.batch * per_tok)
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, d.batch * d.max_blocks_per_seq)
    _check(lib().kvc_append(ctypes.byref(d), _ptr(cache), int(layer), _ptr(k_new), _ptr(v_new), int(n_new),
                            _ptr(pos), _ptr(block_table), _ptr(workspace), workspace.numel(), _stream(stream)),
           "kvc_append")


def decode_attention(d: KvcDesc, cache: torch.Tensor, layer: int, q: torch.Tensor, pos: torch.Tensor,
                     workspace: torch.Tensor, block_table: torch.Tensor | None = None,
                     valid_bits: torch.Tensor | None = None, out: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """kvc_decode_attention: q [batch, q_heads, D] -> out [batch, q_heads, D]."""
    dt = desc_dtype(d)
    _need_cache(d, cache)
    _need(q, "q", dt, d.batch * d.q_heads * d.head_dim)
    _need(pos, "pos", torch.int32, d.batch)
    _need(workspace, "workspace", torch.uint8)
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, d.batch * d.max_blocks_per_seq)
    if valid_bits is not None:
        _need(valid_bits, "valid_bits", torch.int32, (d.num_blocks + 31) // 32)
    if out is None:
        out = torch.empty((d.batch, d.q_heads, d.head_dim), dtype=dt, device=q.device)
    _need(out, "out", dt, d.batch * d.q_heads * d.head_dim)
    _check(lib().kvc_decode_attention(ctypes.byref(d), _ptr(cache), int(layer), _ptr(q), _ptr(pos),
                                      _ptr(block_table), _ptr(valid_bits), _ptr(out), _ptr(workspace),
                                      workspace.numel(), _stream(stream)),
           "kvc_decode_attention")
    return out


def decode_step(d: KvcDesc, cache: torch.Tensor, layer: int, q: torch.Tensor, k_new: torch.Tensor,
                v_new: torch.Tensor, pos: torch.Tensor, workspace: torch.Tensor,
                block_table: torch.Tensor | None = None, valid_bits: torch.Tensor | None = None,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """kvc_decode_step: append the token at pos (k_new / v_new [batch, kv_heads, D]) and attend."""
    dt = desc_dtype(d)
    _need_cache(d, cache)
    _need(q, "q", dt, d.batch * d.q_heads * d.head_dim)
    _need(k_new, "k_new", dt, d.batch * d.kv_heads * d.head_dim)
    _need(v_new, "v_new", dt, d.batch * d.kv_heads * d.head_dim)
    _need(pos, "pos", torch.int32, d.batch)
    _need(workspace, "workspace", torch.uint8)
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, d.batch * d.max_blocks_per_seq)
    if valid_bits is not None:
        _need(valid_bits, "valid_bits", torch.int32, (d.num_blocks + 31) // 32)
    if out is None:
        out = torch.empty((d.batch, d.q_heads, d.head_dim), dtype=dt, device=q.device)
    _need(out, "out", dt, d.batch * d.q_heads * d.head_dim)
    _check(lib().kvc_decode_step(ctypes.byref(d), _ptr(cache), int(layer), _ptr(q), _ptr(k_new), _ptr(v_new),
                                 _ptr(pos), _ptr(block_table), _ptr(valid_bits), _ptr(out), _ptr(workspace),
                                 workspace.numel(), _stream(stream)),
           "kvc_decode_step")
    return out


def prefill_workspace_bytes(d: KvcDesc, T: int) -> int:
    return int(lib().kvc_prefill_workspace_bytes(ctypes.byref(d), int(T)))


def alloc_prefill_workspace(d: KvcDesc, T: int, device="cuda") -> torch.Tensor:
    """Zero-filled workspace for kvc_prefill with chunks of up to T tokens (also a decode workspace)."""
    n = prefill_workspace_bytes(d, T)
    if n == 0:
        raise KvcError(KVC_ERR_DESC, "kvc_prefill_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def prefill(d: KvcDesc, cache: torch.Tensor, layer: int, q: torch.Tensor, k_new: torch.Tensor,
            v_new: torch.Tensor, pos0: torch.Tensor, workspace: torch.Tensor,
            block_table: torch.Tensor | None = None, valid_bits: torch.Tensor | None = None,
            out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """kvc_prefill: q [batch, T, q_heads, D], k_new / v_new [batch, T, kv_heads, D] -> out [batch, T, q_heads, D]."""
    dt = desc_dtype(d)
    _need_cache(d, cache)
    _need(q, "q", dt)
    if q.numel() % (d.batch * d.q_heads * d.head_dim):
        raise ValueError("q must be [batch, T, q_heads, head_dim]")
    T = q.numel() // (d.batch * d.q_heads * d.head_dim)
    _need(k_new, "k_new", dt, d.batch * T * d.kv_heads * d.head_dim)
    _need(v_new, "v_new", dt, d.batch * T * d.kv_heads * d.head_dim)
    _need(pos0, "pos0", torch.int32, d.batch)
    _need(workspace, "workspace", torch.uint8)
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, d.batch * d.max_blocks_per_seq)
    if valid_bits is not None:
        _need(valid_bits, "valid_bits", torch.int32, (d.num_blocks + 31) // 32)
    if out is None:
        out = torch.empty((d.batch, T, d.q_heads, d.head_dim), dtype=dt, device=q.device)
    _need(out, "out", dt, d.batch * T * d.q_heads * d.head_dim)
    _check(lib().kvc_prefill(ctypes.byref(d), _ptr(cache), int(layer), _ptr(q), _ptr(k_new), _ptr(v_new), int(T),
                             _ptr(pos0), _ptr(block_table), _ptr(valid_bits), _ptr(out), _ptr(workspace),
                             workspace.numel(), _stream(stream)),
           "kvc_prefill")
    return out


def block_table_write(d: KvcDesc, block_table: torch.Tensor, seq: torch.Tensor, logical_block: torch.Tensor,
                      physical_block: torch.Tensor, workspace: torch.Tensor,
                      valid_bits: torch.Tensor | None = None, stream=None):
    n = seq.numel()
    _need(block_table, "block_table", torch.int32, d.batch * d.max_blocks_per_seq)
    for name, t in (("seq", seq), ("logical_block", logical_block), ("physical_block", physical_block)):
        _need(t, name, torch.int32, n)
    if valid_bits is not None:
        _need(valid_bits, "valid_bits", torch.int32, (d.num_blocks + 31) // 32)
    _need(workspace, "workspace", torch.uint8)
    _check(lib().kvc_block_table_write(ctypes.byref(d), _ptr(block_table), _ptr(valid_bits), int(n), _ptr(seq),
                                       _ptr(logical_block), _ptr(physical_block), _ptr(workspace),
                                       workspace.numel(), _stream(stream)),
           "kvc_block_table_write")


def valid_write(d: KvcDesc, valid_bits: torch.Tensor, slot: torch.Tensor, value: torch.Tensor,
                workspace: torch.Tensor, stream=None):
    n = slot.numel()
    _need(valid_bits, "valid_bits", torch.int32, (d.num_blocks + 31) // 32)
    _need(slot, "slot", torch.int32, n)
    _need(value, "value", torch.int32, n)
    _need(workspace, "workspace", torch.uint8)
    _check(lib().kvc_valid_write(ctypes.byref(d), _ptr(valid_bits), int(n), _ptr(slot), _ptr(value),
                                 _ptr(workspace), workspace.numel(), _stream(stream)),
           "kvc_valid_write")


class BlockState:
    """Device state of the paged cache's block manager (include/kvc.h): the
    block table and valid bits, a reference count per block, and the free
    list (a stack of block ids, `free_count` entries)."""

    def __init__(self, d: KvcDesc, device="cuda", free_order=None):
        self.table = torch.full((d.batch, d.max_blocks_per_seq), -1, dtype=torch.int32, device=device)
        self.valid_bits = torch.zeros((d.num_blocks + 31) // 32, dtype=torch.int32, device=device)
        self.refcount = torch.zeros(d.num_blocks, dtype=torch.int32, device=device)
        order = list(range(d.num_blocks)) if free_order is None else list(free_order)
        self.free_list = torch.tensor(order, dtype=torch.int32, device=device)
        self.free_count = torch.tensor([len(order)], dtype=torch.int32, device=device)


def block_prepare(d: KvcDesc, cache: torch.Tensor, pos: torch.Tensor, state: BlockState,
                  workspace: torch.Tensor, stream=None):
    _need_cache(d, cache)
    _need(pos, "pos", torch.int32, d.batch)
    _need(workspace, "workspace", torch.uint8)
    _check(lib().kvc_block_prepare(ctypes.byref(d), _ptr(cache), _ptr(pos), _ptr(state.table),
                                   _ptr(state.valid_bits), _ptr(state.refcount), _ptr(state.free_list),
                                   _ptr(state.free_count), _ptr(workspace), workspace.numel(), _stream(stream)),
           "kvc_block_prepare")


def block_share(d: KvcDesc, state: BlockState, src_seq: torch.Tensor, dst_seq: torch.Tensor,
                nblocks: torch.Tensor, workspace: torch.Tensor, stream=None):
    n = src_seq.numel()
    for t, name in ((src_seq, "src_seq"), (dst_seq, "dst_seq"), (nblocks, "nblocks")):
        _need(t, name, torch.int32, n)
    _check(lib().kvc_block_share(ctypes.byref(d), _ptr(state.table), _ptr(state.refcount), int(n), _ptr(src_seq),
                                 _ptr(dst_seq), _ptr(nblocks), _ptr(workspace), workspace.numel(),
                                 _stream(stream)),
           "kvc_block_share")


def block_release(d: KvcDesc, state: BlockState, seq: torch.Tensor, workspace: torch.Tensor, stream=None):
    n = seq.numel()
    _need(seq, "seq", torch.int32, n)
    _check(lib().kvc_block_release(ctypes.byref(d), _ptr(state.table), _ptr(state.valid_bits),
                                   _ptr(state.refcount), _ptr(state.free_list), _ptr(state.free_count), int(n),
                                   _ptr(seq), _ptr(workspace), workspace.numel(), _stream(stream)),
           "kvc_block_release")


class Pager:
    """kvc_pager: LRU residency of a fixed pool of slots (host object), with
    page-in of blocks from pinned host memory on a copy stream."""

    def __init__(self, num_slots: int):
        self.num_slots = num_slots
        self._p = lib().kvc_pager_create(int(num_slots))
        if not self._p:
            raise KvcError(KVC_ERR_ARG, "kvc_pager_create")

    def close(self):
        if self._p:
            lib().kvc_pager_destroy(self._p)
            self._p = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def plan(self, need, pinned=None):
        """need: logical block ids of this step -> (page-ins [(block, slot)], victims [(block, slot)])."""
        n = len(need)
        arr = (ctypes.c_int32 * max(1, n))
        nd = arr(*need)
        pn = (ctypes.c_uint8 * max(1, n))(*[1 if x else 0 for x in pinned]) if pinned is not None else None
        ib, isl, ob, osl = arr(), arr(), arr(), arr()
        ni, no = ctypes.c_int32(0), ctypes.c_int32(0)
        _check(lib().kvc_pager_plan(self._p, n, nd, pn, ctypes.byref(ni), ib, isl, ctypes.byref(no), ob, osl),
               "kvc_pager_plan")
        return ([(ib[i], isl[i]) for i in range(ni.value)], [(ob[i], osl[i]) for i in range(no.value)])

    def evict(self, d: KvcDesc, seq: int, victims, block_table, valid_bits, stream=None):
        n = len(victims)
        arr = ctypes.c_int32 * max(1, n)
        _check(lib().kvc_pager_evict(ctypes.byref(d), int(seq), n, arr(*[b for b, _ in victims]),
                                     arr(*[s for _, s in victims]), _ptr(block_table),
                                     _ptr(valid_bits) if valid_bits is not None else None, _stream(stream)),
               "kvc_pager_evict")

    def issue(self, d: KvcDesc, cache, host_kv, pageins, copy_stream, compute_stream=None):
        """Copy each (logical block, slot) of `pageins` from host_kv, pinned host memory laid out
        [logical block][layer][K|V][kv head][row][D], into its slot of the cache."""
        n = len(pageins)
        if n:
            elt = 4 if d.dtype == 0 else 2
            need = (max(b for b, _ in pageins) + 1) * d.layers * 2 * d.kv_heads * d.block_size * d.head_dim * elt
            if host_kv.numel() * host_kv.element_size() < need:
                raise ValueError(f"host_kv holds {host_kv.numel() * host_kv.element_size()} bytes, "
                                 f"the listed blocks need {need}")
        _need_cache(d, cache)
        arr = ctypes.c_int32 * max(1, n)
        _check(lib().kvc_pagein_issue(self._p, ctypes.byref(d), _ptr(cache), ctypes.c_void_p(host_kv.data_ptr()), n,
                                      arr(*[b for b, _ in pageins]), arr(*[s for _, s in pageins]),
                                      _stream(copy_stream), _stream(compute_stream)),
               "kvc_pagein_issue")

    def commit(self, d: KvcDesc, seq: int, pageins, block_table, valid_bits, stream=None):
        n = len(pageins)
        arr = ctypes.c_int32 * max(1, n)
        _check(lib().kvc_pagein_commit(self._p, ctypes.byref(d), int(seq), n, arr(*[b for b, _ in pageins]),
                                       arr(*[s for _, s in pageins]), _ptr(block_table),
                                       _ptr(valid_bits) if valid_bits is not None else None, _stream(stream)),
               "kvc_pagein_commit")


def get_error(workspace: torch.Tensor, stream=None) -> int:
    """Device error bits (KVC_DEV_*) since the last call; synchronises the stream and clears them."""
    _need(workspace, "workspace", torch.uint8)
    rc = lib().kvc_get_error(_ptr(workspace), _stream(stream))
    if rc < 0:
        raise KvcError(rc, "kvc_get_error")
    return rc


def pack_valid_bits(mask: torch.Tensor) -> torch.Tensor:
    """bool [num_blocks] -> int32 words, bit (k & 31) of word k // 32 = mask[k] (the layout valid_bits uses)."""
    m = mask.to(torch.int64).flatten()
    n = m.numel()
    words = (n + 31) // 32
    pad = torch.zeros(words * 32, dtype=torch.int64, device=m.device)
    pad[:n] = m
    w = (pad.view(words, 32) << torch.arange(32, device=m.device, dtype=torch.int64)).sum(dim=1)
    w = torch.where(w >= 2 ** 31, w - 2 ** 32, w)
    return w.to(torch.int32)
