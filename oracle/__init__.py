"""CPU oracle for decode-step KV-cache attention.

TEST INFRASTRUCTURE ONLY.  Only `tests/`, `__graft_entry__.smoke()` and the
CPU-baseline leg of `bench.py` may import or run anything in this package; the
library under `sliding_window_attention_kvc_gb300/` never does, and shares no
code with it.  Inputs come from `kvc_synth` (seeded draws, no arithmetic of the
method).

What it computes, in fp64 numpy, slowly and plainly:

* `storage`   – rounding of a value to the cache's storage type (bf16 / fp32).
* `quant`     – per-row INT8 storage: fp32 scale max|x| / 127, codes rounded
                to nearest-even ([primer] 5.1, quantised cache).
* `rope`      – rotary position embedding, rotate-half pairing (i, i + D/2).
* `layouts`   – slot maps, attended sets and in-cache positions of the three
                cache layouts, plus step-by-step layout models (a ring with a
                head pointer, a compacting StreamingLLM cache, a physical
                sink+ring, a block pool with a block table and valid bits).
* `blocks`    – the paged cache's block manager: free list, prefix sharing
                with reference counts, copy-on-write, release ([share] §3.2,
                §5.1, §6.1).
* `prefill`   – a chunk of T tokens: each token's output equals the decode
                step at its position after the chunk's earlier tokens are
                appended ([pool] chunked prefill, [ring] window as a mask).
* `attention` – one decode step: scores q.k / sqrt(D), max-subtracted softmax,
                weighted sum of V.  Every sum is exactly rounded (math.fsum),
                so a result never depends on the order in which the attended
                tokens are visited.

Pages cited (by title and section):
  [ring]   "Why sliding-window attention decodes with a ring KV cache"
           (2kiu.com/news/4318096), numbered sections 1.1-8.
  [share]  "Shared state, isolated problems: KV cache and batching"
           (pwwt.cn/news/6215824), numbered sections 1-7.
  [sink]   "Attention sinks and StreamingLLM" (openeuler.csdn.net), the
           softmax equations, the cache-set equation, the cache manager
           class and the "RoPE cache position shifting" section.
  [primer] "KV cache primer" (pwwt.cn/news/5010196), numbered sections 1-6.
  [pool]   "KV cache paging" (cloudlnk.cn/blog/kv-cache-paging), sections
           "kernel forgets absent blocks" and "self-contained shards: RoPE
           baked into K rows".

Pin status: every function here is pinned by `tests/test_oracle_pins.py`
(the block manager by `tests/test_oracle_blocks.py`)
against values the pages print, closed forms, a library routine
(torch scaled_dot_product_attention in fp64) or brute force on tiny inputs.
The numeric attention outputs of the full workloads have no worked example
on the pages; they are pinned through those checks of the definition.
"""

from . import attention, blocks, layouts, prefill, quant, rope, storage
from .attention import attend, decode_masked_history, decode_reference, decode_sequence
from .layouts import (
    PagedKV,
    RingKV,
    SinkRingKV,
    StreamingKV,
    incache_position,
    paged_attended,
    window_attended,
    window_slot,
)
from .rope import inv_freq, rotate
from .storage import round_bf16, round_storage

__all__ = [
    "attention", "blocks", "layouts", "prefill", "quant", "rope", "storage",
    "attend", "decode_reference", "decode_masked_history", "decode_sequence",
    "PagedKV", "RingKV", "SinkRingKV", "StreamingKV",
    "incache_position", "paged_attended", "window_attended", "window_slot",
    "inv_freq", "rotate", "round_bf16", "round_storage",
]
