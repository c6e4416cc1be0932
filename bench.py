#!/usr/bin/env python
"""Benchmark of decode-step KV-cache attention on GB300.

One step = one decode step of one attention layer for the whole batch:
kvc_decode_step: the new token's K/V appended (RoPE fused; fused into the
attention kernel for bf16 ring caches), then split-K attention.  Steps cycle
over `layers` cache layers so the working set (>= 1 GiB) is far larger than
the 126 MiB L2: every step reads its KV from HBM.

Prints one JSON line.  `value` = algorithmic bytes per step (attended K/V
rows + q + out + the appended row) / device time per step, in GB/s, from the
median of five timed loops of exactly K steps (CUDA graphs, replayed once
untimed first); `roofline` relates the step's time to the measured HBM copy
peak; `per_workload` times the other workloads the same way in the same
process; `e2e` repeats the metric with host-resident inputs copied in (one
packed copy) and the output copied out every step; `cpu_baseline` times the
CPU oracle on a bounded sample.  `--impl reference` times the CPU oracle as
the reference arm, with the same metric and config.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import kvc_synth  # noqa: E402

DEFAULT_WORKLOAD = "paged_shared_prefix_bf16"
DEFAULT_LAYERS = {"tiny_ring_sink_f32": 1, "ring_bf16": 8, "sink_window_bf16": 2,
                  "paged_shared_prefix_bf16": 2, "long_context_pool_bf16": 4,
                  "ring_int8": 8, "sink_window_int8": 2, "paged_shared_prefix_int8": 2}


def _kvc():
    import sliding_window_attention_kvc_gb300 as kvc
    return kvc


# ---------------------------------------------------------------------------
# workload -> library descriptor, algorithmic bytes
# ---------------------------------------------------------------------------

def workload_desc(wl, layers=None, num_splits=0, batch=None):
    kvc = _kvc()
    L = wl.layers if layers is None else layers
    B = wl.batch if batch is None else batch
    if wl.layout == "window":
        layout = "sink_ring" if wl.sinks > 0 else "ring"
        return kvc.make_desc(layout, wl.rope, wl.dtype, L, B, wl.q_heads, wl.kv_heads, wl.head_dim,
                             window=wl.window, sinks=wl.sinks, num_splits=num_splits, rope_base=wl.rope_base)
    return kvc.make_desc("paged", wl.rope, wl.dtype, L, B, wl.q_heads, wl.kv_heads, wl.head_dim,
                         block_size=wl.block_size, num_blocks=wl.num_blocks,
                         max_blocks_per_seq=wl.max_blocks_per_seq, num_splits=num_splits,
                         rope_base=wl.rope_base)


def attended_rows(wl):
    """Per sequence: number of cached rows the step at t_b attends, and for the
    paged layout the (physical block -> rows read) map (for unique bytes)."""
    t = wl.positions
    if wl.layout == "window":
        return np.minimum(t + 1, wl.capacity), None
    rows = np.zeros(wl.batch, dtype=np.int64)
    touched = {}
    for b in range(wl.batch):
        tb = int(t[b])
        for lb in range(tb // wl.block_size + 1):
            phys = int(wl.block_table[b, lb])
            if phys < 0 or (wl.valid is not None and not wl.valid[phys]):
                continue
            n = wl.block_size if lb < tb // wl.block_size else tb - lb * wl.block_size + 1
            rows[b] += n
            touched[phys] = max(touched.get(phys, 0), n)
    return rows, touched


def attended_count(wl, b, t):
    """Keys the token at position t of sequence b attends: the sinks below S
    and the window's last W positions (window layouts), or the rows up to t of
    mapped and valid blocks (paged)."""
    if t < 0:
        return 0
    if wl.layout == "window":
        sinks = min(wl.sinks, t + 1)
        lo = max(wl.sinks, t - wl.window + 1)
        return sinks + max(0, t - lo + 1)
    bs = wl.block_size
    n = 0
    for lb in range(t // bs + 1):
        phys = int(wl.block_table[b, lb])
        if phys < 0 or (wl.valid is not None and not wl.valid[phys]):
            continue
        n += bs if lb < t // bs else t - lb * bs + 1
    return n


def step_bytes(wl):
    """Algorithmic bytes of one decode step (whole batch, one layer)."""
    rows, touched = attended_rows(wl)
    # K and V of one token (INT8: codes and row scales)
    row_bytes = wl.kv_heads * 2 * (wl.head_dim * wl.elt_bytes + wl.row_scale_bytes)
    logical_kv = int(rows.sum()) * row_bytes
    unique_kv = logical_kv if touched is None else sum(touched.values()) * row_bytes
    qo = 2 * wl.batch * wl.q_heads * wl.head_dim * wl.value_bytes   # q in, out
    # new K/V read, and written to the cache
    appended = wl.batch * wl.kv_heads * 2 * (wl.head_dim * (wl.value_bytes + wl.elt_bytes) + wl.row_scale_bytes)
    return {"kv_logical": logical_kv, "kv_unique": unique_kv, "qo": qo, "append": appended,
            "decode_algorithmic": unique_kv + qo, "step_algorithmic": unique_kv + qo + appended}


# ---------------------------------------------------------------------------
# cache set-up through kvc_append
# ---------------------------------------------------------------------------

def _raw_rows_device(shape, dtype, seed_key):
    g = torch.Generator(device="cuda")
    g.manual_seed(kvc_synth.derive_seed(*seed_key))
    return torch.randn(shape, generator=g, device="cuda", dtype=torch.float32).to(kvc_synth.to_dtype(dtype))


def _window_fill_inputs(wl, layer, source):
    """K/V rows for positions before t_b that the cache holds at step t_b:
    sinks [0, min(S, t_b)) and the last W positions [t_b - W, t_b), both
    left-padded to fixed lengths (negative positions are skipped by kvc_append)."""
    calls = []
    t = wl.positions
    parts = [("sinks", wl.sinks, np.minimum(wl.sinks, t) - wl.sinks)] if wl.sinks > 0 else []
    parts.append(("window", wl.window, t - wl.window))
    for name, n, start in parts:
        if source == "cpu":
            k = torch.zeros((wl.batch, n, wl.kv_heads, wl.head_dim), dtype=kvc_synth.to_dtype(wl.value_dtype))
            v = torch.zeros_like(k)
            for b in range(wl.batch):
                p = np.arange(start[b], start[b] + n)
                keep = p >= 0
                kb, vb = wl.kv_history(layer, b, p[keep])
                k[b, keep] = kb
                v[b, keep] = vb
            k, v = k.cuda(), v.cuda()
        else:
            k = _raw_rows_device((wl.batch, n, wl.kv_heads, wl.head_dim), wl.value_dtype,
                                 (wl.seed, layer, 101 if name == "sinks" else 102))
            v = _raw_rows_device((wl.batch, n, wl.kv_heads, wl.head_dim), wl.value_dtype,
                                 (wl.seed, layer, 103 if name == "sinks" else 104))
        calls.append((k, v, torch.from_numpy(start.astype(np.int32)).cuda()))
    return calls


def _paged_runs(wl, b):
    """Runs [p0, p1) of positions before t_b whose logical blocks are mapped."""
    bs, tb = wl.block_size, int(wl.positions[b])
    mapped = wl.block_table[b] >= 0
    runs, lb, nlb = [], 0, tb // bs + 1
    while lb < nlb:
        if not mapped[lb]:
            lb += 1
            continue
        lb1 = lb
        while lb1 < nlb and mapped[lb1]:
            lb1 += 1
        p0, p1 = lb * bs, min(lb1 * bs, tb)
        if p1 > p0:
            runs.append((p0, p1))
        lb = lb1
    return runs


class DecodeState:
    """Device state of one workload: cache, workspace, per-layer step inputs."""

    def __init__(self, wl, layers, source="device", num_splits=0, poison=True):
        kvc = _kvc()
        self.wl = wl
        self.layers = layers
        self.desc = workload_desc(wl, layers, num_splits)
        self.cache = kvc.alloc_cache(self.desc, fill=float("nan") if poison else 0.0)
        self.ws = kvc.alloc_workspace(self.desc)
        self.pos = torch.from_numpy(wl.positions.astype(np.int32)).cuda()
        self.table = None
        self.valid_bits = None
        if wl.layout == "paged":
            self.table = torch.from_numpy(wl.block_table.astype(np.int32)).contiguous().cuda()
            if wl.valid is not None:
                self.valid_bits = kvc.pack_valid_bits(torch.from_numpy(wl.valid)).cuda()
        self.q, self.k_new, self.v_new = [], [], []
        for layer in range(layers):
            self._fill_layer(layer, source)
            if source == "cpu":
                q = wl.queries(layer)
                kn, vn = wl.new_kv(layer)
            else:
                q = _raw_rows_device((wl.batch, wl.q_heads, wl.head_dim), wl.value_dtype, (wl.seed, layer, 105))
                kn = _raw_rows_device((wl.batch, wl.kv_heads, wl.head_dim), wl.value_dtype, (wl.seed, layer, 106))
                vn = _raw_rows_device((wl.batch, wl.kv_heads, wl.head_dim), wl.value_dtype, (wl.seed, layer, 107))
            self.q.append(q.contiguous().cuda())
            self.k_new.append(kn.contiguous().cuda())
            self.v_new.append(vn.contiguous().cuda())
        if wl.layout == "paged" and wl.valid is not None and poison:
            # non-resident slots hold no data: poison them, they must never be read
            bad = torch.from_numpy(~wl.valid).cuda()
            if wl.dtype == "i8":
                kvc.int8_views(self.desc, self.cache)[1][:, :, bad] = float("nan")
            else:
                self.cache[:, :, bad] = float("nan")
        self.out = torch.empty((wl.batch, wl.q_heads, wl.head_dim), dtype=kvc.desc_dtype(self.desc),
                               device="cuda")
        torch.cuda.synchronize()
        err = kvc.get_error(self.ws)
        if err:
            raise RuntimeError(f"device error bits {err:#x} while filling the cache")

    def _fill_layer(self, layer, source):
        kvc = _kvc()
        wl = self.wl
        if wl.layout == "window":
            for k, v, start in _window_fill_inputs(wl, layer, source):
                kvc.append(self.desc, self.cache, layer, k, v, start, self.ws)
            return
        d1 = workload_desc(wl, self.layers, batch=1)
        ws1 = kvc.alloc_workspace(d1)
        elt = self.table.element_size()
        for b in range(wl.batch):
            row_ptr = self.table.data_ptr() + b * wl.max_blocks_per_seq * elt
            for p0, p1 in _paged_runs(wl, b):
                n = p1 - p0
                if source == "cpu":
                    k, v = wl.kv_history(layer, b, np.arange(p0, p1))
                    k, v = k[None].cuda(), v[None].cuda()
                else:
                    k = _raw_rows_device((1, n, wl.kv_heads, wl.head_dim), wl.value_dtype, (wl.seed, layer, b, p0, 108))
                    v = _raw_rows_device((1, n, wl.kv_heads, wl.head_dim), wl.value_dtype, (wl.seed, layer, b, p0, 109))
                start = torch.tensor([p0], dtype=torch.int32, device="cuda")
                rc = kvc.lib().kvc_append(ctypes.byref(d1), self.cache.data_ptr(), layer, k.data_ptr(),
                                          v.data_ptr(), n, start.data_ptr(), row_ptr, ws1.data_ptr(),
                                          ws1.numel(), torch.cuda.current_stream().cuda_stream)
                if rc != 0:
                    raise kvc.KvcError(rc, "kvc_append (fill)")
        torch.cuda.synchronize()
        if kvc.get_error(ws1):
            raise RuntimeError("device error while filling the paged cache")

    # one decode step on `layer` (append the token at pos, attend), through the
    # C ABI with device buffers
    def step(self, layer, out=None):
        kvc = _kvc()
        return kvc.decode_step(self.desc, self.cache, layer, self.q[layer], self.k_new[layer], self.v_new[layer],
                               self.pos, self.ws, block_table=self.table, valid_bits=self.valid_bits,
                               out=self.out if out is None else out)

    def launches_per_step(self):
        """Kernels one kvc_decode_step launches.  bf16 / INT8 caches: the
        decode kernel (which writes the new token of window layouts) and its
        combine kernel, plus a paged batch's plan kernel (which writes the new
        tokens; a one-sequence paged cache whose table and valid words fit the
        decode's shared memory, 5120 and 4096 words, is planned inside the
        decode kernel).  fp32 caches: the decode kernel (its last CTA combines)
        plus a separate append (window layouts) or the plan kernels (paged: one
        for a single sequence of at most 4096 blocks, else two)."""
        wl = self.wl
        paged = wl.layout == "paged"
        if wl.dtype in ("bf16", "i8"):
            self_plan = (paged and wl.batch == 1 and wl.max_blocks_per_seq <= 5120
                         and (wl.num_blocks + 31) // 32 <= 4096)
            return 2 + (1 if paged and not self_plan else 0)
        if paged:
            return 1 + (1 if wl.batch == 1 and wl.max_blocks_per_seq <= 4096 else 2)
        return 2


class FastCalls:
    """Pre-marshalled ctypes calls of kvc_append / kvc_decode_attention for the
    timed loop (same C entry points as the binding, minus per-call checks)."""

    def __init__(self, st: DecodeState):
        kvc = _kvc()
        L = kvc.lib()
        self.L = L
        s = torch.cuda.current_stream().cuda_stream
        d = ctypes.byref(st.desc)
        tb = st.table.data_ptr() if st.table is not None else None
        vb = st.valid_bits.data_ptr() if st.valid_bits is not None else None
        ws, wsn = st.ws.data_ptr(), st.ws.numel()
        self.app = [(d, st.cache.data_ptr(), l, st.k_new[l].data_ptr(), st.v_new[l].data_ptr(), 1,
                     st.pos.data_ptr(), tb, ws, wsn, s) for l in range(st.layers)]
        self.dec = [(d, st.cache.data_ptr(), l, st.q[l].data_ptr(), st.pos.data_ptr(), tb, vb,
                     st.out.data_ptr(), ws, wsn, s) for l in range(st.layers)]
        self.stp = [(d, st.cache.data_ptr(), l, st.q[l].data_ptr(), st.k_new[l].data_ptr(), st.v_new[l].data_ptr(),
                     st.pos.data_ptr(), tb, vb, st.out.data_ptr(), ws, wsn, s) for l in range(st.layers)]

    def append(self, layer):
        rc = self.L.kvc_append(*self.app[layer])
        if rc:
            raise RuntimeError(f"kvc_append: {rc}")

    def decode(self, layer):
        rc = self.L.kvc_decode_attention(*self.dec[layer])
        if rc:
            raise RuntimeError(f"kvc_decode_attention: {rc}")

    def step(self, layer):
        rc = self.L.kvc_decode_step(*self.stp[layer])
        if rc:
            raise RuntimeError(f"kvc_decode_step: {rc}")


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0, period_ms=50):
        self.proc = None
        self.lines = []
        self.device_index = device_index
        self.period_ms = period_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.device_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


# DRAM bytes (read + write) per launch of decode_mma_kernel, from one ncu
# capture per workload, and the digest of the kernel's sources
# (KERNEL_TRAFFIC_FILES) they were taken on: reported only while those
# sources are unchanged.
KERNEL_TRAFFIC = {"ring_bf16": 137679616, "sink_window_bf16": 543395584,
                  "paged_shared_prefix_bf16": 842048256, "long_context_pool_bf16": 156166144,
                  "ring_int8": 70007552}
KERNEL_TRAFFIC_SOURCES = "24d6eacb67dbe03dc8e15f6823c3bd723a1a13f551c9d31eef08d159a6fe4904"


# the sources decode_mma_kernel and its launch are built from
KERNEL_TRAFFIC_FILES = ("decode_inst.cuh", "decode_paged_bf16.cu", "decode_paged_i8.cu", "decode_window_bf16.cu",
                        "decode_window_i8.cu", "kvc_api.cu", "kvc_decode.cuh", "kvc_decode_mma.cuh",
                        "kvc_device.cuh", "kvc_params.h")


def _kernel_sources_digest():
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_TRAFFIC_FILES:
        h.update(name.encode())
        with open(os.path.join(ROOT, "sliding_window_attention_kvc_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _traffic(wl_name, override):
    if override is not None:
        return override
    if wl_name in KERNEL_TRAFFIC and _kernel_sources_digest() == KERNEL_TRAFFIC_SOURCES:
        return KERNEL_TRAFFIC[wl_name]
    return None


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# the CPU oracle as a timed baseline
# ---------------------------------------------------------------------------

def oracle_sample(wl, budget_s, max_rows=None, part=(0, 1)):
    """Run the CPU oracle on (sequence, kv head) units of layer 0 until
    `budget_s` seconds of oracle time are spent; returns (bytes, seconds,
    units).  part = (k, n): only the units u = b * kv_heads + h with u mod n == k."""
    import oracle
    spec = dict(rope=wl.rope, base=wl.rope_base, storage=wl.dtype, sinks=wl.sinks, window=wl.window)
    row_bytes = 2 * (wl.head_dim * wl.elt_bytes + wl.row_scale_bytes)
    g = wl.group_size
    done_bytes, spent, units = 0, 0.0, 0
    for b in range(wl.batch):
        mine = [h for h in range(wl.kv_heads) if (b * wl.kv_heads + h) % part[1] == part[0]]
        if not mine:
            continue
        t = int(wl.positions[b])
        if wl.layout == "window":
            pos = oracle.window_attended(t, wl.sinks, wl.window)
        else:
            pos = oracle.paged_attended(t, wl.block_table[b], wl.valid, wl.block_size)
        if max_rows is not None:
            pos = pos[-max_rows:]
        k, v = wl.kv_history(0, b, pos)
        q = wl.query(0, b)
        for h in mine:
            qf = q[h * g:(h + 1) * g].double().numpy()
            kf, vf = k[:, h].double().numpy(), v[:, h].double().numpy()
            t0 = time.perf_counter()
            if wl.dtype == "i8":        # rows as an INT8 cache stores them (baked keys: after rotation)
                vf = oracle.quant.store_i8(vf)
                if wl.rope != "baked":
                    kf = oracle.quant.store_i8(kf)
            oracle.decode_reference(qf, kf, vf, pos, t, **spec)
            spent += time.perf_counter() - t0
            done_bytes += len(pos) * row_bytes
            units += 1
            if spent >= budget_s:
                return done_bytes, spent, units
    return done_bytes, spent, units


def _oracle_worker(name, kw, budget_s, k, n):
    """One process of the all-core oracle timing (spawned: one BLAS thread)."""
    wl = kvc_synth.make_workload(name, **kw)
    return oracle_sample(wl, budget_s, part=(k, n))


def _workload_kw(args):
    """Generator options taken from the command line (the pool's valid density)."""
    if getattr(args, "density", None) is None:
        return {}
    if not args.workload.startswith("long_context_pool"):
        raise SystemExit("--density applies to long_context_pool_bf16 only")
    if not 0.0 <= args.density <= 1.0:
        raise SystemExit("--density must be in [0, 1]")
    return {"density": args.density}


def cpu_baseline(wl, budget_s=10.0, cores=None, kw=None):
    """The fp64 oracle on the host cores: all cores (a spawn-started process
    per core over disjoint sequences, for the same budget of wall time), and
    one core, over bounded samples of the workload's units."""
    nbytes1, secs1, units1 = oracle_sample(wl, budget_s)
    single = nbytes1 / secs1 / 1e9
    cores = cores or min(os.cpu_count() or 1, max(1, wl.batch * wl.kv_heads))
    line = {"value": single, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{units1} (sequence, kv head) units of one layer-step of {wl.name}, "
                      f"{nbytes1 / 1e6:.1f} MB of attended K/V, {secs1:.1f} s single-threaded fp64"}
    if cores > 1:
        import multiprocessing as mpr
        env = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in env:
            os.environ[k] = "1"
        try:
            with mpr.get_context("spawn").Pool(cores) as pool:
                t0 = time.perf_counter()
                res = pool.starmap(_oracle_worker, [(wl.name, kw or {}, budget_s, k, cores) for k in range(cores)])
                wall = time.perf_counter() - t0
        finally:
            for k, v in env.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        nbytes = sum(r[0] for r in res)
        busy = max(r[1] for r in res)
        units = sum(r[2] for r in res)
        line.update(value=nbytes / busy / 1e9, cores=cores,
                    sample=f"{units} (sequence, kv head) units of one layer-step of {wl.name} over {cores} "
                           f"processes (disjoint units), {nbytes / 1e6:.1f} MB of attended K/V, "
                           f"{busy:.1f} s of oracle time per process (wall {wall:.1f} s incl. start-up)",
                    single_core_value=single)
    return line


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ---------------------------------------------------------------------------
# replicas (N > 1): one process per GPU, no collective on the data path; the
# ranks only meet for the barriers around the timed region and the max of
# their times
# ---------------------------------------------------------------------------

def replica_init(world, backend="nccl", device=None):
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            dist.init_process_group("nccl", device_id=device)
        else:
            dist.init_process_group(backend)


def replica_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def replica_max(value, world, device="cuda"):
    """Largest `value` over the ranks (the slowest replica sets the job time)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_done(world):
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def job_throughput(bytes_per_step, world, ms_per_step):
    """Whole-job GB/s: every rank streams bytes_per_step per step (weak scaling)."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


METRIC = "decode-attention KV HBM GB/s"
TIMED_LOOPS = 5           # timed loops of K steps; the median loop sets ms_per_step
PER_WORKLOAD_STEPS = 200  # steps per timed loop of each per_workload entry
# configurations timed beside the headline in the same process: the other
# workloads of the statement, the pool's valid-density sweep, the INT8 caches
PER_WORKLOAD = [("tiny_ring_sink_f32", {}), ("ring_bf16", {}), ("sink_window_bf16", {}),
                ("paged_shared_prefix_bf16", {}), ("long_context_pool_bf16", {}),
                ("long_context_pool_bf16", {"density": 0.25}), ("long_context_pool_bf16", {"density": 1.0}),
                ("ring_int8", {}), ("sink_window_int8", {}), ("paged_shared_prefix_int8", {})]


def workload_config(wl, layers, world, kw):
    """The `config` object of both arms' JSON lines: the workload by name and shape."""
    nb = step_bytes(wl)
    return {"workload": wl.name, "batch": wl.batch, "q_heads": wl.q_heads, "kv_heads": wl.kv_heads,
            "head_dim": wl.head_dim, "window": wl.window, "sinks": wl.sinks,
            "block_size": wl.block_size, "layers_cycled": layers, "rope": wl.rope, "cache_dtype": wl.dtype,
            "l2": f"inputs larger than L2: {layers} layers cycled, "
                  f"{layers * nb['kv_unique'] / 2**20:.0f} MiB of attended K/V",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU", **kw}


def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return None
    kw = _workload_kw(args)
    wl = kvc_synth.make_workload(args.workload, **kw)
    layers = getattr(args, "layers", 0) or DEFAULT_LAYERS[args.workload]
    per_step = max(0.002, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    # rows per step sized to the per-step budget (about 25k rows/s for D=128)
    rows = max(64, int(per_step * 25000 * 128 / wl.head_dim))
    for _ in range(args.warmup):
        oracle_sample(wl, per_step, max_rows=rows)
    tot_b, tot_s, tot_u = 0, 0.0, 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        b, s, u = oracle_sample(wl, per_step, max_rows=rows)
        tot_b, tot_s, tot_u = tot_b + b, tot_s + s, tot_u + u
    wall = time.perf_counter() - t0
    val = tot_b / tot_s / 1e9
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_s / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, layers, world, kw),
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: up to {rows} attended rows of (sequence, kv head) units, "
                                       f"~{per_step:.3f} s of fp64 oracle time; {tot_u} units, wall {wall:.1f} s"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def capture_graphs(st, K):
    """CUDA graphs of K consecutive steps (layers cycled): graph A holds n steps
    (a whole number of layer cycles) and is replayed K // n times, graph B the
    remaining K mod n steps.  Returns [(graph, replays)], or [] if capture fails."""
    layers = st.layers
    n = min(K, max(layers, (512 // layers) * layers))
    reps, rest = divmod(K, n)
    graphs = []
    for count in (n, rest):
        if count == 0 or (count == n and reps == 0):
            continue
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fcg = FastCalls(st)           # binds the capture stream
            for i in range(count):
                fcg.step(i % layers)
        graphs.append((g, reps if count == n else 1))
    return graphs


def timed_loops(st, fc, K, loops, graphs, barrier=lambda: None):
    """`loops` timed loops of exactly K steps each, every loop bracketed by a
    barrier and a device synchronize on both sides and timed with CUDA events
    on the launching stream.  Graphs are replayed once, untimed, first (their
    upload and first launch stay out of the timed region); before each loop
    the GPU is held ~10 ms so that the host's launches queue ahead of it.
    Returns the loop times in ms."""
    layers = st.layers
    if graphs:
        for g, _ in graphs:
            g.replay()
    else:
        for i in range(min(K, 3 * layers)):
            fc.step(i % layers)
    torch.cuda.synchronize()
    out = []
    for _ in range(loops):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        torch.cuda._sleep(20_000_000)
        start.record()
        if graphs:
            for g, r in graphs:
                for _ in range(r):
                    g.replay()
        else:
            for i in range(K):
                fc.step(i % layers)
        end.record()
        torch.cuda.synchronize()
        barrier()
        out.append(start.elapsed_time(end))
    return out


def _roofline(wl, nb, ms_per_step, kw, traffic_override):
    peak, peak_kind = _peaks()
    achieved = nb["step_algorithmic"] / (ms_per_step * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_kind": peak_kind,
            "traffic": _traffic(wl.name, traffic_override) if not kw else traffic_override,
            "traffic_kernel": "decode_mma_kernel, dram__bytes_read.sum + dram__bytes_write.sum per launch",
            "kernel": "kvc_decode_step: " + ("decode_mma_kernel + combine_streamk_kernel"
                                             if wl.dtype in ("bf16", "i8") else "append + decode"),
            "timer": "CUDA events around each timed loop of K kvc_decode_step calls; median loop, per step",
            "algorithmic_bytes_per_launch": nb["step_algorithmic"]}


def measure_workload(name, kw, steps, loops):
    """One per_workload entry: the workload's own state, graph-replayed loops
    of `steps` steps, median loop."""
    wl = kvc_synth.make_workload(name, **kw)
    layers = DEFAULT_LAYERS[name]
    st = DecodeState(wl, layers, source="device")
    fc = FastCalls(st)
    for i in range(3 * layers):
        fc.step(i % layers)
    torch.cuda.synchronize()
    graphs = capture_graphs(st, steps)
    times = timed_loops(st, fc, steps, loops, graphs)
    kvc = _kvc()
    err = kvc.get_error(st.ws)
    ms = statistics.median(times) / steps
    nb = step_bytes(wl)
    entry = {"workload": name, **kw, "ms_per_step": ms, "us_per_step": ms * 1e3, "steps_per_s": 1e3 / ms,
             "value": nb["step_algorithmic"] / (ms * 1e-3) / 1e9, "unit": "GB/s",
             "bytes_per_step": nb, "loop_ms": times, "steps_per_loop": steps, "layers_cycled": layers,
             "gpu_launches_per_step": st.launches_per_step(), "device_errors": err}
    if wl.dtype != "f32":
        entry["roofline_frac"] = entry["value"] / _peaks()[0]
        entry["frac_of_8tbs"] = entry["value"] / 8000.0
    else:
        entry["note"] = "latency-bound (32 KiB of K/V per step): steps/s is the figure"
    del st, fc, graphs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def run_ours(args):
    kvc = _kvc()
    rank, world, local = _dist()
    torch.cuda.set_device(local)
    replica_init(world, "nccl", torch.device("cuda", local))
    kw = _workload_kw(args)
    wl = kvc_synth.make_workload(args.workload, **kw)
    layers = args.layers or DEFAULT_LAYERS[args.workload]
    st = DecodeState(wl, layers, source="device", num_splits=args.num_splits)
    fc = FastCalls(st)
    nb = step_bytes(wl)

    def barrier():
        replica_barrier(world)

    # warm-up
    for i in range(args.warmup):
        fc.step(i % layers)
    torch.cuda.synchronize()

    K = args.steps
    # The timed loops replay CUDA graphs of the K steps (the launches keep
    # their programmatic-dependency edges); without --eager the host's launch
    # cost stays out of the device timeline.
    graphs, timing = [], "eager"
    if not args.eager:
        try:
            graphs = capture_graphs(st, K)
            timing = "cuda_graph (one untimed replay first)"
        except Exception as exc:                  # capture unsupported: time eagerly
            graphs = []
            timing = f"eager (graph capture failed: {type(exc).__name__})"
        torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    loops = timed_loops(st, fc, K, args.loops, graphs, barrier)
    med = statistics.median(loops)
    total_ms = replica_max(med, world)
    ms_per_step = total_ms / K
    value = job_throughput(nb["step_algorithmic"], world, ms_per_step)
    err = kvc.get_error(st.ws)
    if err:
        raise RuntimeError(f"device error bits {err:#x} during the timed region")

    # the same steps launched one by one: what a caller without graphs sees
    eager_ms = None
    if graphs:
        ne = min(max(K, 200), 2000)
        eager_ms = statistics.median(timed_loops(st, fc, ne, 3, [])) / ne

    per_workload = None
    prefill = None
    if rank == 0 and world == 1 and not args.no_per_workload:
        per_workload = []
        for name, pkw in PER_WORKLOAD:
            if name == wl.name and pkw == kw:
                continue
            per_workload.append(measure_workload(name, pkw, PER_WORKLOAD_STEPS, args.loops))
        # chunked prefill (kvc_prefill), 128-token chunks ending at each
        # sequence's position, on the three bf16 layouts and the INT8 paged batch
        prefill = []
        for name in ("ring_bf16", "paged_shared_prefix_bf16", "sink_window_bf16", "paged_shared_prefix_int8"):
            pa = argparse.Namespace(workload=name, chunk=128, steps=20, warmup=3)
            r = measure_prefill(pa)
            prefill.append({"workload": name, "chunk_tokens": 128, "ms_per_call": r["ms_per_call"],
                            "tokens_per_s": r["tokens_per_s"], "tflops": r["value"],
                            "roofline_frac": r["roofline"]["frac"], "peak_kind": r["roofline"]["peak_kind"],
                            "rope": "read_time" if name.startswith("sink_window") else "baked",
                            "cache_dtype": "i8" if name.endswith("int8") else "bf16",
                            "device_errors": r["device_errors"]})
            torch.cuda.empty_cache()
    clk = clocks.stop()

    # end to end: host inputs copied in, host output copied out, every step
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(st, args, nb)

    line = {
        "metric": METRIC,
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": workload_config(wl, layers, world, kw),
        "steps_per_s": 1e3 / ms_per_step,
        "bytes_per_step": nb,
        "timing": timing,
        "timed_loops": len(loops),
        "loop_ms": loops,
        "eager_ms_per_step": eager_ms,
        "roofline": _roofline(wl, nb, ms_per_step, kw, args.traffic),
        "frac_of_8tbs": value / 8000.0,
        "clocks": clk,
        "gpu_launches": st.launches_per_step() * K,
        "gpu_launches_note": "kernels launched in one timed loop of K steps",
        "e2e": e2e,
        "per_workload": per_workload,
        "prefill": prefill,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_budget, kw=kw)
    replica_done(world)
    return line if rank == 0 else None


class PackedInputs:
    """A step's inputs packed into one buffer, q | k_new | v_new | pos, each
    part at a 256-byte offset: one pinned host buffer per layer and one device
    staging buffer whose views the step reads, so that a step copies its
    inputs in with one host-to-device copy."""

    def __init__(self, st):
        parts0 = [st.q[0], st.k_new[0], st.v_new[0], st.pos]
        self.offs, off = [], 0
        for t in parts0:
            self.offs.append(off)
            off = (off + t.numel() * t.element_size() + 255) // 256 * 256
        self.nbytes = off
        self.dev = torch.zeros(off, dtype=torch.uint8, device="cuda")
        self.host = []
        for layer in range(st.layers):
            h = torch.zeros(off, dtype=torch.uint8)
            for t, o in zip([st.q[layer], st.k_new[layer], st.v_new[layer], st.pos], self.offs):
                raw = t.contiguous().view(-1).view(torch.uint8).cpu()
                h[o:o + raw.numel()] = raw
            self.host.append(h.pin_memory())

    def ptr(self, i):
        return self.dev.data_ptr() + self.offs[i]


def run_e2e(st, args, nb):
    """The metric end to end through the C ABI: every step copies its packed
    inputs from pinned host memory (one copy), runs kvc_decode_step on the
    staged views, copies the output back to pinned host memory and waits."""
    kvc = _kvc()
    L = kvc.lib()
    layers = st.layers
    K = max(10, min(args.steps, 2000))
    pk = PackedInputs(st)
    hout = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
    s = torch.cuda.current_stream()
    d = ctypes.byref(st.desc)
    tb = st.table.data_ptr() if st.table is not None else None
    vb = st.valid_bits.data_ptr() if st.valid_bits is not None else None
    args_of = [(d, st.cache.data_ptr(), l, pk.ptr(0), pk.ptr(1), pk.ptr(2), pk.ptr(3), tb, vb,
                st.out.data_ptr(), st.ws.data_ptr(), st.ws.numel(), s.cuda_stream) for l in range(layers)]

    def step(i):
        layer = i % layers
        pk.dev.copy_(pk.host[layer], non_blocking=True)
        rc = L.kvc_decode_step(*args_of[layer])
        if rc:
            raise RuntimeError(f"kvc_decode_step: {rc}")
        hout.copy_(st.out, non_blocking=True)
        s.synchronize()

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    times = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(K):
            step(i)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = statistics.median(times) / K
    return {"value": nb["step_algorithmic"] / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": pk.nbytes, "d2h_bytes_per_step": hout.numel() * hout.element_size(),
            "steps": K, "loops": len(times),
            "note": "per step: one copy of the packed inputs (q, k_new, v_new, pos) from pinned host memory, "
                    "kvc_decode_step on the staged views, out -> pinned host, host waits for the result; "
                    "median of 3 loops"}


def measure_block_prepare(args):
    """One kvc_block_prepare call on a shared-prefix batch shaped like the
    paged workload: 64 sequences in groups of 8 share a 2050-token prefix
    (129 blocks of 16, the last holding 2 rows); every sequence then writes
    token 2050, so in each group 7 copy the shared tail block and the last
    writes in place.  The state is restored before each timed call; device
    time per call from CUDA events, median over the repeats."""
    kvc = _kvc()
    B, G, prefix, bs, Hq, Hkv, D = 64, 8, 2050, 16, 32, 8, 128
    layers = args.layers or 1
    nb_seq = (prefix + bs - 1) // bs
    num_blocks = (B // G) * nb_seq + B + 16
    d = kvc.make_desc("paged", "baked", "bf16", layers, B, Hq, Hkv, D, block_size=bs, num_blocks=num_blocks,
                      max_blocks_per_seq=nb_seq + 4)
    cache = kvc.alloc_cache(d, fill=0.0)
    ws = kvc.alloc_workspace(d)
    st = kvc.BlockState(d)
    leaders = list(range(0, B, G))
    for t in range(0, prefix, bs):                 # leaders take their prefix blocks
        pos = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        pos[leaders] = t
        kvc.block_prepare(d, cache, pos, st, ws)
    src = torch.tensor([l for l in leaders for m in range(1, G)], dtype=torch.int32, device="cuda")
    dst = torch.tensor([l + m for l in leaders for m in range(1, G)], dtype=torch.int32, device="cuda")
    kvc.block_share(d, st, src, dst, torch.full_like(src, nb_seq), ws)
    torch.cuda.synchronize()
    snap = [x.clone() for x in (st.table, st.valid_bits, st.refcount, st.free_list, st.free_count)]
    pos = torch.full((B,), prefix, dtype=torch.int32, device="cuda")
    times = []
    for i in range(args.warmup + args.steps):
        for x, y in zip((st.table, st.valid_bits, st.refcount, st.free_list, st.free_count), snap):
            x.copy_(y)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        kvc.block_prepare(d, cache, pos, st, ws)
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1) * 1e3)
    err = kvc.get_error(ws)
    copies = int((st.table[:, nb_seq - 1] != snap[0][:, nb_seq - 1]).sum().item())
    return {"measure": "kvc_block_prepare", "value": statistics.median(times), "unit": "us per call",
            "higher_is_better": False, "steps": args.steps, "warmup": args.warmup,
            "config": {"sequences": B, "group": G, "prefix_tokens": prefix, "block_size": bs, "layers": layers,
                       "kv_heads": Hkv, "head_dim": D, "copies": copies, "copied_bytes":
                       copies * layers * 2 * Hkv * (prefix % bs) * D * 2},
            "device_errors": err}


def measure_pagein(args):
    """Page-in overlapped with decode on the long-context pool's shape (one
    sequence, 1024 slots of 64 tokens, 16 q / 4 kv heads, D 256): each step
    brings `k` new blocks from pinned host memory into slots freed by the LRU
    pager while the step's decode runs over the resident blocks.  Reports the
    decode alone, the copies alone (copy stream), and the overlapped step,
    each the median of device times from CUDA events."""
    kvc = _kvc()
    Hq, Hkv, D, bs, slots, nlog, k = 16, 4, 256, 64, 1024, 2048, 64
    layers = args.layers or 1
    d = kvc.make_desc("paged", "baked", "bf16", layers, 1, Hq, Hkv, D, block_size=bs, num_blocks=slots,
                      max_blocks_per_seq=nlog)
    g = torch.Generator().manual_seed(9)
    host = torch.randn((nlog, layers, 2, Hkv, bs, D), generator=g).to(torch.bfloat16).pin_memory()
    cache = kvc.alloc_cache(d, fill=0.0)
    ws = kvc.alloc_workspace(d)
    table = torch.full((1, nlog), -1, dtype=torch.int32, device="cuda")
    valid = torch.zeros((slots + 31) // 32, dtype=torch.int32, device="cuda")
    pager = kvc.Pager(slots)
    cs = torch.cuda.Stream()
    t = nlog * bs - 1
    pos = torch.tensor([t], dtype=torch.int32, device="cuda")
    q = torch.randn((1, Hq, D), device="cuda").to(torch.bfloat16)
    window = list(range(nlog - 64, nlog))
    rng = np.random.default_rng(9)
    resident = list(rng.choice(nlog - 64, size=slots - 64, replace=False))
    ins, outs = pager.plan(window + resident, [1] * 64 + [0] * (slots - 64))
    pager.issue(d, cache, host, ins, cs)
    pager.commit(d, 0, ins, table, valid)
    torch.cuda.synchronize()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    dec, cop, both = [], [], []
    for i in range(args.warmup + args.steps):
        keep = [b for b in resident if rng.random() > k / len(resident)][: len(resident) - k]
        new = [b for b in rng.permutation(nlog - 64).tolist() if b not in keep][:len(resident) - len(keep)]
        resident = keep + new
        ins, outs = pager.plan(window + resident, [1] * 64 + [0] * len(resident))
        pager.evict(d, 0, outs, table, valid)
        # decode alone
        a0, a1 = ev(), ev()
        a0.record()
        kvc.decode_attention(d, cache, 0, q, pos, ws, block_table=table, valid_bits=valid)
        a1.record()
        # copies alone, then overlapped with a decode
        c0, c1 = ev(), ev()
        torch.cuda.synchronize()
        c0.record(cs)
        pager.issue(d, cache, host, ins, cs)
        c1.record(cs)
        torch.cuda.synchronize()
        b0, b1 = ev(), ev()
        b0.record()
        pager.issue(d, cache, host, ins, cs)
        kvc.decode_attention(d, cache, 0, q, pos, ws, block_table=table, valid_bits=valid)
        pager.commit(d, 0, ins, table, valid)
        b1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            dec.append(a0.elapsed_time(a1))
            cop.append(c0.elapsed_time(c1))
            both.append(b0.elapsed_time(b1))
    nbytes = len(ins) * layers * 2 * Hkv * bs * D * 2
    med = statistics.median
    return {"measure": "page-in overlapped with decode", "unit": "ms",
            "decode_ms": med(dec), "copy_ms": med(cop), "overlapped_step_ms": med(both),
            "copy_GBps": nbytes / (med(cop) * 1e-3) / 1e9, "blocks_per_step": len(ins), "bytes_per_step": nbytes,
            "steps": args.steps, "warmup": args.warmup,
            "config": {"slots": slots, "logical_blocks": nlog, "block_size": bs, "q_heads": Hq, "kv_heads": Hkv,
                       "head_dim": D, "layers": layers, "pinned_window_blocks": 64},
            "device_errors": kvc.get_error(ws)}


def measure_prefill(args):
    """Chunked prefill (kvc_prefill) of T = --chunk tokens per sequence on a
    bf16 or INT8 workload (default ring_bf16: 8 sequences, 32 q / 8 kv heads,
    D 128, a full 4096-slot ring; also sink_window_bf16, whose RoPE is applied
    at read time, paged_shared_prefix_bf16, and their INT8 forms ring_int8,
    sink_window_int8, paged_shared_prefix_int8), each chunk ending at the workload's position t_b,
    the cache holding every earlier position.  One call stages the chunk,
    runs the attention and appends the chunk.  L2 is flushed (a 256 MiB write)
    between timed calls; each call is timed with CUDA events.  Reports tokens/s
    and the attention's algorithmic TFLOP/s (4 D flops per (token, q head,
    attended key): q.k and p.v) against the measured bf16 tensor peak."""
    kvc = _kvc()
    name = args.workload if args.workload in ("ring_bf16", "paged_shared_prefix_bf16", "sink_window_bf16",
                                              "ring_int8", "paged_shared_prefix_int8", "sink_window_int8") \
        else "ring_bf16"
    wl = kvc_synth.make_workload(name)
    T = args.chunk
    pos0 = np.maximum(wl.positions - T + 1, 0)
    import dataclasses
    wl0 = dataclasses.replace(wl, positions=pos0)
    st = DecodeState(wl0, 1, source="device")
    B, Hq, Hkv, D = wl.batch, wl.q_heads, wl.kv_heads, wl.head_dim
    q = _raw_rows_device((B, T, Hq, D), "bf16", (wl.seed, 0, 201))
    k = _raw_rows_device((B, T, Hkv, D), "bf16", (wl.seed, 0, 202))
    v = _raw_rows_device((B, T, Hkv, D), "bf16", (wl.seed, 0, 203))
    ws = kvc.alloc_prefill_workspace(st.desc, T)
    out = torch.empty((B, T, Hq, D), dtype=torch.bfloat16, device="cuda")
    pos_t = torch.from_numpy(pos0.astype(np.int32)).cuda()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    # algorithmic work: attended keys of every chunk token
    keys = sum(attended_count(wl, b, int(pos0[b]) + i) for b in range(B) for i in range(T))
    flops = 4.0 * D * Hq * keys
    times = []
    for i in range(args.warmup + args.steps):
        flush.fill_(i & 255)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        kvc.prefill(st.desc, st.cache, 0, q, k, v, pos_t, ws, block_table=st.table, valid_bits=st.valid_bits,
                    out=out)
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        with open(peaks_path) as f:
            peak, peak_kind = float(json.load(f)["bf16_tflops"]), "measured (cuBLAS bf16, burst)"
    else:
        peak, peak_kind = 1900.0, "fallback (one earlier GB300 measurement, burst)"
    achieved = flops / (ms * 1e-3) / 1e12
    return {"measure": "chunked prefill", "metric": "prefill attention TFLOP/s", "value": achieved,
            "unit": "TFLOP/s", "ms_per_call": ms, "tokens_per_s": B * T / (ms * 1e-3),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "algorithmic_flops_per_call": flops,
                         "kernel": "kvc_prefill: prefill_stage_kernel + prefill_ws_kernel (tcgen05, warp-specialised) + append_kernel",
                         "timer": "CUDA events around each call, median, L2 flushed between calls"},
            "steps": args.steps, "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "chunk_tokens": T, "batch": B, "q_heads": Hq, "kv_heads": Hkv,
                       "head_dim": D, "attended_keys": keys},
            "device_errors": kvc.get_error(ws)}


def build_parser():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(kvc_synth.WORKLOAD_NAMES), default=DEFAULT_WORKLOAD)
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--density", type=float, default=None,
                    help="long_context_pool_bf16: valid-bit density of the pool's slots (default 0.5)")
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="time only the headline workload (no per_workload entries)")
    ap.add_argument("--loops", type=int, default=TIMED_LOOPS, help="timed loops of K steps (median reported)")
    ap.add_argument("--eager", action="store_true", help="launch the timed steps one by one (no CUDA graph)")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--chunk", type=int, default=128, help="--measure prefill: tokens per chunk")
    ap.add_argument("--measure", choices=["block_prepare", "pagein", "prefill"], default=None,
                    help="time a block-manager call instead of the decode step (separate JSON line)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per decode launch from an ncu capture of the current kernel")
    return ap


def main(argv=None):
    args = build_parser().parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.measure == "block_prepare":
        line = measure_block_prepare(args)
    elif args.measure == "pagein":
        line = measure_pagein(args)
    elif args.measure == "prefill":
        line = measure_prefill(args)
    else:
        line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
