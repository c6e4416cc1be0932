"""Helpers shared by the GPU parity tests and smoke(): oracle outputs for a
workload (CPU, fp64), and a step-by-step decode loop through the C ABI."""

from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {"f32": 2e-3, "bf16": 2e-2, "i8": 2e-2}   # max abs error of the outputs (INT8 cache: bf16 outputs)


def attended(wl, b, t=None):
    t = int(wl.positions[b]) if t is None else int(t)
    if wl.layout == "window":
        return oracle.window_attended(t, wl.sinks, wl.window)
    return oracle.paged_attended(t, wl.block_table[b], wl.valid, wl.block_size)


def oracle_outputs(wl, layer, seqs=None, positions=None):
    """Oracle decode output [len(seqs), Hq, D] (fp64) for sequences `seqs` of `wl`."""
    seqs = range(wl.batch) if seqs is None else seqs
    pos_all = wl.positions if positions is None else np.asarray(positions)
    spec = dict(rope=wl.rope, base=wl.rope_base, storage=wl.dtype, sinks=wl.sinks, window=wl.window)
    outs = []
    for b in seqs:
        t = int(pos_all[b])
        p = attended(wl, b, t)
        k, v = wl.kv_history(layer, b, p)
        kd, vd = k.double().numpy(), v.double().numpy()
        if wl.dtype == "i8":
            # rows as an INT8 cache stores them; baked keys are quantised after
            # rotation, inside the oracle
            vd = oracle.quant.store_i8(vd)
            if wl.rope != "baked":
                kd = oracle.quant.store_i8(kd)
        q = wl.query(layer, b, t)
        outs.append(oracle.decode_sequence(q.double().numpy(), kd, vd, p, t, **spec))
    return np.stack(outs)


def run_stepwise(wl, steps, num_splits=0, layer=0):
    """Decode steps t in `steps` (ascending, from an empty cache) of a window
    workload with batch 1: append token t, then attend.  Returns {t: out [Hq, D]}."""
    import bench
    import sliding_window_attention_kvc_gb300 as kvc

    assert wl.layout == "window" and wl.batch == 1
    d = bench.workload_desc(wl, layers=1, num_splits=num_splits)
    cache = kvc.alloc_cache(d, fill=float("nan"))
    ws = kvc.alloc_workspace(d)
    outs = {}
    steps = sorted(steps)
    t_prev = -1
    for t in steps:
        # append every token up to t (the ones before t in one bulk call)
        if t - 1 > t_prev:
            n = t - 1 - t_prev
            k, v = wl.kv_history(layer, 0, np.arange(t_prev + 1, t))
            kvc.append(d, cache, 0, k[None].contiguous().cuda(), v[None].contiguous().cuda(),
                       torch.tensor([t_prev + 1], dtype=torch.int32, device="cuda"), ws)
            del n
        k, v = wl.kv_history(layer, 0, [t])
        pos = torch.tensor([t], dtype=torch.int32, device="cuda")
        kvc.append(d, cache, 0, k[None].contiguous().cuda(), v[None].contiguous().cuda(), pos, ws)
        q = wl.query(layer, 0, t)[None].contiguous().cuda()
        out = kvc.decode_attention(d, cache, 0, q, pos, ws)
        outs[t] = out[0].float().cpu().numpy()
        t_prev = t
    assert kvc.get_error(ws) == 0
    return outs
