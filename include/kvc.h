/*
 * kvc.h - C ABI of the decode-step KV-cache attention library (libkvc.so).
 *
 * One new query per sequence attends over a fixed-capacity KV cache kept in
 * one of three layouts, and the new token's K/V is appended to that cache;
 * a chunk of new tokens can be prefilled the same way (kvc_prefill), and the
 * cache can hold bf16, fp32 or per-row INT8 rows.
 * The operations follow these pages (cited by title and section):
 *
 *   [ring]   "Why sliding-window attention decodes with a ring KV cache"
 *            (2kiu.com/news/4318096)
 *   [share]  "Shared state, isolated problems: KV cache and batching"
 *            (pwwt.cn/news/6215824)
 *   [sink]   "Attention sinks and StreamingLLM" (openeuler.csdn.net)
 *   [primer] "KV cache primer" (pwwt.cn/news/5010196)
 *   [pool]   "KV cache paging" (cloudlnk.cn/blog/kv-cache-paging)
 *
 * Conventions shared by every entry point
 *   - Every buffer argument is a DEVICE pointer owned by the caller (cache,
 *     queries, outputs, tables, workspace); the library allocates no device
 *     memory.  `stream` is a cudaStream_t (NULL = the legacy default stream);
 *     every call except kvc_get_error only enqueues work on it and returns.
 *   - State the library keeps across calls (host side, thread-safe):
 *     (1) the TMA tensor maps of the last 8 bf16 / INT8 caches it decoded,
 *     keyed by (cache address, layers, rows per K half, head_dim, dtype,
 *     device): a cache freed and a different one allocated at the same
 *     address with the same shape reuses the maps, which are still correct,
 *     since they depend on nothing else;  (2) kvc_pager objects, which the
 *     caller creates and destroys;  (3) the fixed device scratch of
 *     kvc_decode_attention_noalloc (see there).  Everything else a call
 *     needs lives in the caller's workspace.
 *   - Return value: KVC_OK (0) or a negative KVC_ERR_* code.  On a negative
 *     code nothing was launched.  Errors that only the device can see (a
 *     block id out of range, an append into an unmapped block, a bad
 *     position) set bits in the workspace's error word; the kernel skips the
 *     offending access and carries on.  kvc_get_error() reads and clears them.
 *   - Element types: the cache, q, out, k_new and v_new share one element
 *     type (kvc_desc.dtype), except that an INT8 cache (KVC_I8) takes and
 *     returns bf16 q, out, k_new and v_new.  All arithmetic is fp32.
 *   - Alignment: cache, q, out, k_new, v_new and workspace must be 16-byte
 *     aligned (KVC_ERR_ALIGN otherwise).
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KVC_API __attribute__((visibility("default")))
#else
#define KVC_API
#endif

/* Cache layouts.
 *  RING       [ring] 3.2-3.3, 5.1: W slots per (sequence, kv head); token p
 *             goes to slot p mod W.  Token t attends t-W+1 .. t ([ring] 2.2,
 *             6), itself included.
 *  SINK_RING  [sink] cache-set equation: S pinned sink slots, then a W-slot
 *             ring.  Token p goes to slot p (p < S) or S + ((p - S) mod W).
 *             Token t attends {0 .. S-1} U {t-W+1 .. t}.
 *  PAGED      [share] 3.1-3.2, [pool] "kernel forgets absent blocks": a pool
 *             of fixed-size blocks; block_table[b][p / block_size] names the
 *             physical block of token p (-1 = not mapped); a per-block valid
 *             bit drops non-resident blocks.  Token t attends every p <= t
 *             whose block is mapped and valid. */
typedef enum { KVC_LAYOUT_RING = 0, KVC_LAYOUT_SINK_RING = 1, KVC_LAYOUT_PAGED = 2 } kvc_layout;

/* RoPE handling (rotate-half pairs (i, i + D/2), theta_i = base^(-2i/D)).
 *  NONE          no rotation.
 *  BAKED         [primer] 4.5, [pool] "RoPE baked into K rows": K is rotated
 *                at its absolute position when appended; q is rotated at t.
 *  READ_INCACHE  [sink] "RoPE cache position shifting": K is stored raw and
 *                rotated when read, at its index in the compacted cache
 *                (sinks 0..S-1; window token p at p - max(0, t - C + 1),
 *                C = S + W); q at min(t, C - 1).  RING and SINK_RING only. */
typedef enum { KVC_ROPE_NONE = 0, KVC_ROPE_BAKED = 1, KVC_ROPE_READ_INCACHE = 2 } kvc_rope;

/* Cache element types.
 *  KVC_F32, KVC_BF16  rows stored as fp32 / bf16 (round to nearest even).
 *  KVC_I8             [primer] 5.1 (quantised cache: INT8 halves the bytes):
 *                     each stored row (one token's K or V of one kv head)
 *                     keeps int8 codes and one fp32 scale s = max|x| / 127,
 *                     codes rint(x / s) clamped to +-127 (IEEE fp32 quotient,
 *                     ties to even), read back as code * s; a zero row has
 *                     s = 0.  With baked RoPE the rotated key is quantised;
 *                     with READ_INCACHE the raw key is, and the decode
 *                     rotates code * s at the in-cache position.  q, out,
 *                     k_new and v_new are bf16.  Requires head_dim 128 or
 *                     256, and rows per K (or V) half of a layer (batch *
 *                     kv_heads * capacity, or num_blocks * kv_heads *
 *                     block_size) a multiple of 4.
 *                     Not accepted by the pool pager (kvc_pagein_issue). */
typedef enum { KVC_F32 = 0, KVC_BF16 = 1, KVC_I8 = 2 } kvc_dtype;

/* Cache geometry.  Cache memory layout ([primer] 3.1, K at index 0, V at 1):
 *   RING / SINK_RING: [layers, 2, batch, kv_heads, capacity, head_dim],
 *                     capacity = sinks + window;
 *   PAGED:            [layers, 2, num_blocks, kv_heads, block_size, head_dim].
 * KVC_I8: that array holds the int8 codes and is followed directly by the
 * fp32 row scales, [layers, 2, batch, kv_heads, capacity] (or [layers, 2,
 * num_blocks, kv_heads, block_size]); kvc_cache_bytes counts both.
 * q_heads must be a multiple of kv_heads; q head h reads kv head
 * h / (q_heads / kv_heads) ([share] 2.2 and 4.1, grouped-query attention).
 * Launch-grid limits (else KVC_ERR_DESC): batch <= 65535, P = q_heads / g4
 * <= 65535 and batch * P < 2^31, where g4 is the largest of 4, 2, 1 that
 * divides q_heads / kv_heads (q heads are processed in groups of g4). */
typedef struct kvc_desc {
    int32_t layout;             /* kvc_layout */
    int32_t rope;               /* kvc_rope */
    int32_t dtype;              /* kvc_dtype (cache element type) */
    int32_t layers;
    int32_t batch;              /* sequences (rows of block_table for PAGED) */
    int32_t q_heads;
    int32_t kv_heads;
    int32_t head_dim;           /* 64, 128 or 256 */
    int32_t window;             /* RING / SINK_RING: W */
    int32_t sinks;              /* SINK_RING: S >= 1; RING: 0 */
    int32_t block_size;         /* PAGED */
    int32_t num_blocks;         /* PAGED: physical blocks in the pool */
    int32_t max_blocks_per_seq; /* PAGED: columns of block_table */
    int32_t num_splits;         /* 0 = library choice; else KV splits per (sequence, kv head)
                                   for RING / SINK_RING, work items for PAGED */
    float rope_base;            /* e.g. 10000 */
    float softmax_scale;        /* 0 => 1 / sqrt(head_dim) */
} kvc_desc;

/* Host-detected status codes (nothing launched). */
#define KVC_OK 0
#define KVC_ERR_NULL (-1)        /* a required pointer is NULL */
#define KVC_ERR_DESC (-2)        /* inconsistent descriptor */
#define KVC_ERR_UNSUPPORTED (-3) /* combination not built (e.g. PAGED + READ_INCACHE) */
#define KVC_ERR_ALIGN (-4)       /* pointer not 16-byte aligned */
#define KVC_ERR_WORKSPACE (-5)   /* workspace smaller than kvc_workspace_bytes() */
#define KVC_ERR_ARG (-6)         /* argument out of range (layer, n_new, n) */
#define KVC_ERR_CUDA (-7)        /* a CUDA runtime call or launch failed */
#define KVC_ERR_TOO_LARGE (-8)   /* kvc_decode_attention_noalloc: the call needs more than
                                    KVC_NOALLOC_SCRATCH_BYTES of scratch */

/* Device-detected error bits, returned by kvc_get_error(). */
#define KVC_DEV_BAD_BLOCK 0x1u       /* block_table entry >= num_blocks (access skipped) */
#define KVC_DEV_UNMAPPED_APPEND 0x2u /* append into a logical block whose entry is -1 */
#define KVC_DEV_BAD_POSITION 0x4u    /* decode position < 0, or beyond the block table */
#define KVC_DEV_TIMEOUT 0x8u         /* a bounded wait inside a kernel gave up */
#define KVC_DEV_BAD_ENTRY 0x10u      /* kvc_block_table_write / kvc_valid_write entry out of range */
#define KVC_DEV_INTERNAL 0x20u       /* an index computed inside a kernel failed its bounds check
                                        (access skipped); a library bug, please report */
#define KVC_DEV_NO_FREE_BLOCK 0x40u  /* kvc_block_prepare: the free list ran out (that sequence skipped) */

/* Bytes of the cache tensor described by `d` (0 if `d` is invalid). */
KVC_API size_t kvc_cache_bytes(const kvc_desc* d);

/* Bytes of workspace that kvc_append / kvc_decode_attention /
 * kvc_block_table_write / kvc_valid_write need for `d` (0 if `d` is invalid).
 * The workspace holds the device error word, split-K partial results and
 * per-(sequence, kv head) completion counters, and for PAGED caches the
 * step's plan (attended rows and an attended-block directory per sequence,
 * the number of sequences reading each physical block) and the block
 * manager's scratch.  It must be zero-filled once before first use
 * (kvc_workspace_init); every call leaves it ready for the next one.  Calls
 * that share a workspace must not overlap on the GPU. */
KVC_API size_t kvc_workspace_bytes(const kvc_desc* d);

/* Zero-fill `workspace` (cudaMemsetAsync on `stream`). */
KVC_API int kvc_workspace_init(const kvc_desc* d, void* workspace, size_t workspace_bytes, void* stream);

/* Append n_new tokens per sequence to layer `layer` of the cache
 * ([ring] 3.3 and 5.1, [primer] 4.4: write in place, no allocation).
 *   k_new, v_new  [batch, n_new, kv_heads, head_dim], pre-RoPE.
 *   pos           [batch] int32: position of token 0 of each sequence; token
 *                 i is at pos[b] + i.  Tokens at negative positions are
 *                 skipped (left padding).
 *   block_table   PAGED: [batch, max_blocks_per_seq] int32; else NULL.
 * BAKED rotates K at its absolute position (the angle p * theta_i reduced
 * exactly as a 64-bit fixed-point fraction of a turn, its sine and cosine
 * and the rotation in fp32, stored rounded to nearest-even); V is never
 * rotated ([pool]).  For
 * RING / SINK_RING the cache ends as if the tokens were appended one at a
 * time in order: a token that a later token of the same call overwrites is
 * not written.  Ring appends must come in position order, one call per step,
 * before the attention call that reads them.  PAGED: an unmapped target
 * block sets KVC_DEV_UNMAPPED_APPEND; a block shared by several sequences
 * must be copied first by the caller (copy-on-write, [share] 3.2). */
KVC_API int kvc_append(const kvc_desc* d, void* cache, int32_t layer,
                       const void* k_new, const void* v_new, int32_t n_new,
                       const int32_t* pos, const int32_t* block_table,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Decode attention for one layer ([primer] 2.2 and 4.2, [sink] softmax
 * equations): out = softmax(q . K^T * scale) . V over the attended set of
 * each sequence, fp32 online softmax, split over the KV length into partial
 * results (m, l, o) in the workspace.  fp32 caches combine the partials in
 * the same kernel (the last CTA of a sequence); bf16 and INT8 caches launch
 * a separate combine kernel right behind the attention kernel (programmatic
 * dependent launch).  PAGED batches run a planning kernel before the
 * attention kernel (per sequence: attended rows, attended-block directory,
 * the readers of each block); a single paged sequence on a bf16 or INT8
 * cache is planned inside the attention kernel.
 *   q       [batch, q_heads, head_dim], pre-RoPE.
 *   pos     [batch] int32: position t of the token being decoded (already
 *           appended, so t attends to itself; [ring] 4.3).
 *   block_table, valid_bits  PAGED only (else NULL): block_table as in
 *           kvc_append; valid_bits [ceil(num_blocks / 32)] uint32, bit
 *           (k & 31) of word k / 32 set when physical block k is resident.
 *           valid_bits NULL = every block resident.
 *   out     [batch, q_heads, head_dim], same element type as q.
 * An empty attended set (a fully masked PAGED sequence) gives zeros. */
KVC_API int kvc_decode_attention(const kvc_desc* d, const void* cache, int32_t layer,
                                 const void* q, const int32_t* pos,
                                 const int32_t* block_table, const uint32_t* valid_bits,
                                 void* out, void* workspace, size_t workspace_bytes, void* stream);

/* One decode step: kvc_append of the token at pos[b] (n_new = 1), then
 * kvc_decode_attention at pos[b], with the same arguments and results as
 * that pair of calls.  For bf16 and INT8 caches, RING / SINK_RING and PAGED
 * with one sequence (planned inside the attention kernel), the append is
 * fused into the attention kernel (the CTA that reads the token's row writes
 * it, with RoPE baked when BAKED, to the cache and to its own copy of the
 * tile); on other PAGED caches the planning kernel writes the tokens before
 * the attention kernel reads; fp32 RING / SINK_RING caches make the two calls
 * in turn.
 *   k_new, v_new  [batch, kv_heads, head_dim], pre-RoPE, 16-byte aligned. */
KVC_API int kvc_decode_step(const kvc_desc* d, void* cache, int32_t layer, const void* q,
                            const void* k_new, const void* v_new, const int32_t* pos,
                            const int32_t* block_table, const uint32_t* valid_bits,
                            void* out, void* workspace, size_t workspace_bytes, void* stream);

/* Chunked prefill ([pool] "the real cost of long context": prefill in chunks
 * of 128-256 tokens; [ring] 3.1 and 5.2: the window as a mask on the score
 * matrix).  For each sequence b, T consecutive tokens at positions
 * pos0[b] + i (i < T): token i gets the output the decode step at that
 * position would give after the chunk's earlier tokens were appended --
 * attention of its q over its attended set A(pos0[b] + i), keys before
 * pos0[b] read from the cache as it stands (the state after position
 * pos0[b] - 1), the chunk's keys from k_new / v_new -- and then the chunk is
 * appended to the cache as kvc_append(n_new = T) would.  Positions below 0
 * are left padding: zero output, nothing appended.
 *   q          [batch, T, q_heads, head_dim] bf16, pre-RoPE.
 *   k_new, v_new [batch, T, kv_heads, head_dim] bf16, pre-RoPE.
 *   pos0       [batch] int32.
 *   block_table, valid_bits  PAGED as in kvc_decode_attention; the chunk's
 *              blocks must be mapped (the append reports unmapped ones).
 *   out        [batch, T, q_heads, head_dim] bf16.
 *   workspace  kvc_prefill_workspace_bytes(d, T) bytes: the decode workspace
 *              followed by the chunk's staged rows.
 * READ_INCACHE: each token's window keys at distance t - p and its sinks at
 * min(t, C - 1) - p, as the decode step at t rotates them.
 * bf16 caches (head_dim 64, 128 or 256) and INT8 caches (128 or 256: cached
 * rows are read back as code * scale, the chunk's own rows as the cache will
 * read them back).  KVC_ERR_UNSUPPORTED: an fp32 cache; at head_dim 256 or on
 * an INT8 cache, a ring or sink+ring chunk longer than the window, paged
 * blocks whose size is not a multiple of 8 dividing 64, or a GQA group that
 * does not divide 128.  Calls on one workspace must not overlap on the
 * GPU.  The attention runs on the tcgen05 tensor cores: a CTA of the
 * warp-specialised kernel (one per SM) holds all 512 tensor-memory columns
 * of its SM while it runs (the kernel for chunks longer than the window: 256
 * columns, two CTAs per SM), so a kernel of another library that holds an
 * SM's tensor memory at the same time delays it.  A wait that does not end
 * within its bound sets KVC_DEV_TIMEOUT in the device error word and the
 * CTA returns, leaving that chunk's output undefined. */
KVC_API size_t kvc_prefill_workspace_bytes(const kvc_desc* d, int32_t T);
KVC_API int kvc_prefill(const kvc_desc* d, void* cache, int32_t layer, const void* q,
                        const void* k_new, const void* v_new, int32_t T, const int32_t* pos0,
                        const int32_t* block_table, const uint32_t* valid_bits,
                        void* out, void* workspace, size_t workspace_bytes, void* stream);

/* Batched block-table update ([share] 3.1 block table, 5.1 block manager):
 * for each i < n, block_table[seq[i]][logical_block[i]] = physical_block[i];
 * -1 unmaps.  When valid_bits is not NULL, each mapped physical block gets its
 * valid bit set (the data is in place); unmapping does not touch valid bits,
 * since other sequences may still map that block.  Entries out of range set
 * KVC_DEV_BAD_ENTRY and are skipped.  Two entries naming the same
 * (seq, logical_block) in one call: which one lands is unspecified. */
KVC_API int kvc_block_table_write(const kvc_desc* d, int32_t* block_table, uint32_t* valid_bits,
                                  int32_t n, const int32_t* seq, const int32_t* logical_block,
                                  const int32_t* physical_block,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* Batched residency update ([pool] "kernel forgets absent blocks"): for each
 * i < n, set (value[i] != 0) or clear the valid bit of physical block slot[i]. */
KVC_API int kvc_valid_write(const kvc_desc* d, uint32_t* valid_bits, int32_t n,
                            const int32_t* slot, const int32_t* value,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Block manager of a paged cache ([share] 3.1-3.2 block table and prefix
 * sharing, 5.1 block manager, 6.1 reclaim on sequence end).  State, all
 * caller-owned device memory: the block table and valid bits as above,
 * refcount int32 [num_blocks] (table references of each block), free_list
 * int32 [num_blocks] used as a stack (entries 0 .. *free_count - 1, top last)
 * and free_count (one int32).  Start: table -1, refcount 0, free_list any
 * permutation of the blocks, *free_count = num_blocks, valid bits 0.
 * Within one call sequences are served in ascending order, exactly as one
 * after the other, so the results are deterministic. */

/* Before appending each sequence's next token (pos[b]; < 0: none), once per
 * token for all layers: a token at a block's first row whose logical block
 * is unmapped gets a new block from the top of the free list; a block
 * referenced by more than one sequence (count > 1) is copied first: a new
 * block receives its rows 0 .. pos mod block_size - 1 of every layer, K and
 * V, every kv head, the sequence's entry points at it, the shared block's
 * count drops by one (copy-on-write, [share] 3.2).  New blocks get count 1
 * and their valid bit (valid_bits may be NULL).  Errors (device bits): an
 * unmapped block entered mid-block (KVC_DEV_UNMAPPED_APPEND), a position past
 * the table (KVC_DEV_BAD_POSITION), an exhausted free list
 * (KVC_DEV_NO_FREE_BLOCK); the sequence is skipped.  Requires layers * 2 *
 * kv_heads <= 65535 (the copy's launch grid), else KVC_ERR_UNSUPPORTED. */
KVC_API int kvc_block_prepare(const kvc_desc* d, void* cache, const int32_t* pos, int32_t* block_table,
                              uint32_t* valid_bits, int32_t* refcount, int32_t* free_list, int32_t* free_count,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Prefix sharing ([share] 3.2, 5.1 share_prefix): for each i < n, logical
 * blocks 0 .. nblocks[i] - 1 of sequence dst_seq[i] point at those of
 * src_seq[i]; each shared block's count rises by one.  The destination's
 * entries must be unmapped, else KVC_DEV_BAD_ENTRY and the entry is skipped. */
KVC_API int kvc_block_share(const kvc_desc* d, int32_t* block_table, int32_t* refcount, int32_t n,
                            const int32_t* src_seq, const int32_t* dst_seq, const int32_t* nblocks,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Sequences end ([share] 6.1): for each listed sequence every mapped block's
 * count drops by one and its entry is unmapped; blocks whose count reaches
 * zero return to the free list in ascending block id and lose their valid
 * bit.  A sequence listed twice is released twice (caller error). */
KVC_API int kvc_block_release(const kvc_desc* d, int32_t* block_table, uint32_t* valid_bits, int32_t* refcount,
                              int32_t* free_list, int32_t* free_count, int32_t n, const int32_t* seq,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Paging of a fixed pool of block slots between host memory and the device
 * ([pool] "KV cache paging": a fixed pool of resident slots; blocks move on
 * demand; the copy engine moves them while attention runs; LRU residency;
 * blocks inside a sliding window stay resident).  A paged cache whose
 * num_blocks slots hold logical blocks of sequence `seq`; the block table maps
 * resident logical blocks to their slot, absent ones to -1 (valid bit off).
 * The host copy of the K/V is pinned memory laid out
 * [logical block][layer][K|V][kv head][row][head_dim] in the cache dtype. */
typedef struct kvc_pager kvc_pager;

/* Host object tracking num_slots slots; NULL if num_slots < 1. */
KVC_API kvc_pager* kvc_pager_create(int32_t num_slots);
KVC_API void kvc_pager_destroy(kvc_pager* pager);

/* Host only.  The blocks one step needs (need[0 .. n-1], logical block ids;
 * pinned[i] != 0 keeps block need[i] resident in later steps until a later
 * call lists it with pinned 0; pinned may be NULL).  Missing blocks take, in
 * list order, the lowest free slot, else the least recently used slot whose
 * block is neither needed now nor pinned (ties: lowest slot).  Outputs (host
 * arrays of n entries): the page-ins (in_block, in_slot; *n_in) and the
 * victims (out_block, out_slot; *n_out).  KVC_ERR_ARG, nothing changed, if the
 * needed and pinned blocks do not fit. */
KVC_API int kvc_pager_plan(kvc_pager* pager, int32_t n, const int32_t* need, const uint8_t* pinned,
                           int32_t* n_in, int32_t* in_block, int32_t* in_slot,
                           int32_t* n_out, int32_t* out_block, int32_t* out_slot);

/* Compute stream: the victims' table entries (sequence seq) become -1 and
 * their slots' valid bits clear.  Host arrays; asynchronous. */
KVC_API int kvc_pager_evict(const kvc_desc* d, int32_t seq, int32_t n, const int32_t* out_block,
                            const int32_t* out_slot, int32_t* block_table, uint32_t* valid_bits, void* stream);

/* Copy stream, after the compute stream's work enqueued so far: one 2-D copy
 * per block (every layer, K and V) from host_kv into its slot, then an event
 * kept by the pager.  Work enqueued on the compute stream after this call
 * overlaps the copies. */
KVC_API int kvc_pagein_issue(kvc_pager* pager, const kvc_desc* d, void* cache, const void* host_kv, int32_t n,
                             const int32_t* in_block, const int32_t* in_slot, void* copy_stream,
                             void* compute_stream);

/* Compute stream waits for the last issue's copies, then the blocks' table
 * entries point at their slots and the slots' valid bits are set. */
KVC_API int kvc_pagein_commit(kvc_pager* pager, const kvc_desc* d, int32_t seq, int32_t n, const int32_t* in_block,
                              const int32_t* in_slot, int32_t* block_table, uint32_t* valid_bits,
                              void* compute_stream);

/* Size of the library's own fixed scratch array used by
 * kvc_decode_attention_noalloc: 8 MiB of device memory, reserved on every GPU
 * that loads the library, from the first use until the process exits. */
#define KVC_NOALLOC_SCRATCH_BYTES (8u << 20)

/* kvc_decode_attention for callers that cannot allocate device memory.
 *
 * Same operation, arguments and results as kvc_decode_attention, except that
 * the caller passes no workspace: the split-K partial results, completion
 * counters and (PAGED) work plan live in a fixed scratch array inside the
 * library (KVC_NOALLOC_SCRATCH_BYTES).  It is meant for code that must not
 * call cudaMalloc once it is running - a serving loop whose device memory is
 * fixed when it starts, or a plugin inside a host framework that owns all
 * device memory and offers no way to allocate - and so has nowhere to put a
 * workspace.  The pages have no counterpart of this entry point.
 *
 *   - It allocates nothing: no cudaMalloc / cudaFree, no allocating library
 *     call.  Inputs and outputs are still the caller's device buffers.
 *   - The first call on a device (with that device current) looks up the
 *     scratch array's device address; make that first call before any stream
 *     capture.  The address is kept per device and context: after the
 *     device's context was destroyed and created again (cudaDeviceReset),
 *     the next call looks it up again, so make that call outside capture
 *     too.  Later calls only enqueue work on `stream`.
 *   - Every call on a device shares the one scratch array and finds it as the
 *     previous call left it; the call clears the parts that must start at
 *     zero (error word, completion counters) on `stream` before its kernels.
 *     Calls that overlap on the GPU (different streams, no ordering between
 *     them) race on the scratch and give wrong results: order them.
 *   - A problem whose workspace (kvc_workspace_bytes) exceeds
 *     KVC_NOALLOC_SCRATCH_BYTES is rejected with KVC_ERR_TOO_LARGE before
 *     anything is launched.
 *   - Device-detected errors are not reported: the kernels still skip bad
 *     accesses, but there is no workspace for kvc_get_error to read. */
KVC_API int kvc_decode_attention_noalloc(const kvc_desc* d, const void* cache, int32_t layer,
                                         const void* q, const int32_t* pos,
                                         const int32_t* block_table, const uint32_t* valid_bits,
                                         void* out, void* stream);

/* Wait for `stream`, then return the workspace's device error bits
 * (KVC_DEV_*, 0 = none) and clear them.  Negative KVC_ERR_* on failure. */
KVC_API int kvc_get_error(void* workspace, void* stream);

/* Static description of a status code or device error bit. */
KVC_API const char* kvc_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
