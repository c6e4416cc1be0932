// Kernel parameter blocks and launch entry points shared by the host-side
// ABI (kvc_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvc {

constexpr int kMaxHalfDim = 128;                 // head_dim <= 256
constexpr long long kWaitCycles = 2000000000LL;  // bounded mbarrier wait (~1 s)
constexpr int kConsumerWarps = 4;                // decode kernel: 4 compute warps
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;  // + 1 copy-issuing warp
constexpr int kStages = 4;                       // bulk-copy pipeline depth
constexpr int kTargetCtas = 608;                 // 152 SMs x 2 CTAs x 2 waves
constexpr int kStreamCtas = 304;                 // stream-K grid: 152 SMs x 2 CTAs
// bf16 stream-K shares per persistent CTA (default).  Claiming several
// shares in turn would even out CTAs that stream at different speeds, but
// every share costs a segment (a q load, a partial, a block walk): on the
// 64-sequence shared-prefix batch one share per CTA measured 153.0 us, 2
// 156.7, 3 160.6, 4 166.6, 6 172.2 -- so paged batches keep one, as the
// other layouts do.
constexpr int kPagedShareFactor = 1;             // paged caches with >= kPagedShareBatch sequences
constexpr int kPagedShareBatch = 8;
// bf16 ring / sink+ring stream-K partition: units charged to each sequence
// for the start of its segment (a second segment costs a CTA a q load and a
// partial write), besides one unit per 16 rows.
constexpr int kSeqUnits = 4;
constexpr int kRunMaps = 4;                      // bf16 kernel: copies of runs of 16, 32, 48, 64 rows
// bf16 caches: K/V rows of its first share that a decode CTA prefetches into
// L2 while it waits for the previous kernel in the stream (window caches:
// rows; paged batches: whole blocks, at most kSpecRows rows of them).
constexpr int kSpecRows = 128;
// Paged caches of one sequence: the decode CTAs plan their own stream-K share
// from the block table and valid bits, staged in their (still empty) pipeline
// stages, without a plan kernel, when the table has at most kSelfPlanMax
// entries and the valid bits at most kSelfPlanValidWords words.
constexpr int kSelfPlanMax = 5120;
constexpr int kSelfPlanValidWords = 4096;
// Resident CTAs per SM of the decode kernel.  INT8 stages are half the
// bytes of bf16 ones; paged INT8 batches at head_dim <= 128 run three CTAs
// per SM (the compute warps are the bound there; measured 164 -> 151 us on
// the shared-prefix batch, while the ring lost 2% and head_dim 256 spills).
constexpr int decode_ctas_per_sm(bool q8, bool paged, bool read, int D) {
    return (read && D >= 256) ? 1 : ((q8 && paged && D <= 128) ? 3 : 2);
}

enum Layout : int { kRing = 0, kSinkRing = 1, kPaged = 2 };
enum Rope : int { kRopeNone = 0, kRopeBaked = 1, kRopeRead = 2 };

// Workspace carve-up (byte offsets from the workspace base).
struct WorkspaceLayout {
    size_t err;          // uint32 error word
    size_t counters;     // uint32 [batch * kv_heads * nsub + 1]: completion tickets (last: paged plan)
    size_t part_ml;      // float2 [items * q_heads]: running max (log2 units), sum of weights
    size_t part_o;       // float  [items * q_heads * head_dim]: unnormalised output
    size_t plan_acc;     // PAGED: int64 [batch] rows before each sequence, then int32 [batch] its rows
    size_t plan_seq;     // PAGED: int2  [batch]: first item, item count
    size_t plan_items;   // PAGED: int4  [items]: (seq, first block, first row, rows)
    size_t plan_info;    // PAGED: int4  [items]: (t of the sequence, its first slot, its slot count, first physical block)
    size_t plan_total;   // PAGED: int32 items used, int32 shares G, int64 attended rows R
    size_t plan_cta;     // PAGED: int2 [ctas]: first item, item count
    size_t plan_dir;     // PAGED: int2 [batch][ceil(maxb / 32)]: attended-block directory (mask, blocks before)
    size_t plan_refs;    // PAGED: uint32 [num_blocks]: sequences attending each block this step (zero between calls)
    size_t blocks;       // PAGED: block manager scratch: int32 [6 * batch], int4 [batch], int32 count,
                         // int32 [num_blocks] reclaim flags
    size_t total;
    int items;           // partial slots per (q head): batch * nsplit, or shares + batch
    int nsplit;          // RING / SINK_RING fp32: splits per (sequence, kv head)
    int shares;          // stream-K shares per (kv head, q-head group) (bf16, paged)
    int ctas;            // persistent CTAs per (kv head, q-head group) that claim the shares
};

struct DecodeParams {
    const void* cache;          // whole cache tensor
    const void* q;              // [B, Hq, D]
    const int32_t* pos;         // [B]
    const int32_t* table;       // PAGED [B, maxb]
    const uint32_t* valid;      // PAGED, may be null
    void* out;                  // [B, Hq, D]
    const void* k_new;          // fused append (kvc_decode_step): [B, Hkv, D] pre-RoPE; null = none
    const void* v_new;
    uint32_t* err;
    uint32_t* counters;         // bf16: [Hkv * nsub] share counters, zero between calls
    float2* part_ml;
    float* part_o;
    const int4* items;          // PAGED plan
    const int4* item_info;      // PAGED plan: (t, first slot, slot count, first physical block) per item
    const int2* seq_items;      // PAGED plan
    const int32_t* n_items;     // PAGED plan
    const int2* cta_items;      // PAGED plan: first item, item count of each CTA (stream-K kernel)
    const int32_t* seq_rows;    // PAGED batch on the tensor-core kernel: attended rows of each sequence
    const int2* dir;            // ... and each sequence's attended-block directory (plan_rows_kernel)
    int dir_groups;             // directory entries per sequence: ceil(maxb / 32)
    uint32_t* refs;             // ... and the sequences attending each physical block (the combine
                                // kernel zeroes it for the next call)
    long long layer_off;        // elements from cache base to this layer's K half
    long long kv_off;           // elements from the K half to the V half
    float* scales;              // INT8 cache: row scales [layers][K|V][rows of a half]; else null
    long long sc_layer_off;     // INT8: scales from `scales` to this layer's K half
    long long sc_kv_off;        // INT8: scales from the K half to the V half (rows of a half)
    int layer;
    int B, Hq, Hkv, G, nsub;
    int window, sinks, capacity;
    int bs, num_blocks, maxb;
    int nsplit;                 // fp32 window: splits per (sequence, kv head); bf16: stream-K shares
    int max_items;              // partial slots per q head (bound for every slot index)
    int rope;                   // kRopeNone / kRopeBaked / kRopeRead
    int tma_whole;              // bf16: 1 = one tensor copy per run covers every column block
    int self_plan;              // PAGED, one sequence: the decode CTAs plan their shares (no plan kernel)
    float q_scale;              // softmax scale * log2(e)
    float theta_f[kMaxHalfDim];     // RoPE frequencies, fp32 (small in-tile angles)
    unsigned long long theta[kMaxHalfDim];   // RoPE frequencies as turns, fixed point: theta_i / (2 pi) * 2^64
};

struct PlanParams {
    const int32_t* pos;
    const int32_t* table;
    const uint32_t* valid;
    uint32_t* err;
    int32_t* seq_rows;    // [B]: attended rows of each sequence
    long long* seq_off;   // [B]: attended rows of the sequences before it
    uint32_t* ticket;     // zero between plans
    int2* seq_items;      // [B]: first item, item count
    int4* items;          // [max_items]: (seq, first block, first row, rows); seq -1 = unused
    int4* item_info;      // [max_items]: (t_b, first slot, slot count of b, physical block of the first block)
    int2* cta_items;      // [ctas]: first item, item count
    int32_t* n_items;     // [0] one past the last item used, [1] G, [2..3] R (int64)
    int2* dir;            // plan_rows_kernel: [B][dir_groups] (mask of attended blocks 32 g .. 32 g + 31,
                          // attended blocks of the sequence before block 32 g)
    int dir_groups;
    uint32_t* refs;       // plan_rows_kernel: [num_blocks] += 1 per sequence attending the block
    int B, bs, num_blocks, maxb, max_items, ctas;
    // the step's new token (kvc_decode_step); k_new == null: none
    void* cache;
    const void* k_new;    // [B, Hkv, D] pre-RoPE
    const void* v_new;
    long long layer_off, kv_off;
    float* scales;        // INT8 cache (elt 1): row scales; sc_layer_off / sc_kv_off as in DecodeParams
    long long sc_layer_off, sc_kv_off;
    int Hkv, D, rope, elt;
    unsigned long long theta[kMaxHalfDim];   // theta_i / (2 pi) * 2^64 (see rope_cos_sin)
};

struct AppendParams {
    void* cache;
    const void* k_new;    // [B, n_new, Hkv, D]
    const void* v_new;
    const int32_t* pos;
    const int32_t* table;
    uint32_t* err;
    long long layer_off;
    long long kv_off;
    float* scales;        // INT8 cache: row scales; sc_layer_off / sc_kv_off as in DecodeParams
    long long sc_layer_off, sc_kv_off;
    int B, Hkv, D, n_new;
    int layout, window, sinks, capacity;
    int bs, num_blocks, maxb;
    int rope;
    unsigned long long theta[kMaxHalfDim];   // theta_i / (2 pi) * 2^64 (see rope_cos_sin)
};

// Chunked prefill (kvc_prefill): T tokens per sequence at pos0[b] + i.
struct PrefillParams {
    const void* cache;
    const void* q;              // [B, T, Hq, D] pre-RoPE
    const void* kst;            // staged chunk rows [B, T, Hkv, D], K as the cache stores it
    const void* vst;
    const int32_t* pos0;        // [B]
    const int32_t* table;       // PAGED [B, maxb]
    const uint32_t* valid;      // PAGED, may be null
    void* out;                  // [B, T, Hq, D]
    uint32_t* err;
    long long layer_off, kv_off;
    int B, T, Hq, Hkv, G;
    int layout, window, sinks, capacity, bs, num_blocks, maxb;
    int rope;
    int layer;
    float q_scale;              // softmax scale * log2(e)
    const float* scales;        // INT8 cache: row scales [layers][K|V][rows of a half]; else null
    long long sc_layer_off;     // INT8: scales from `scales` to this layer's K half
    long long sc_kv_off;        // INT8: from the K half's scales to the V half's (rows of a half)
    long long half_rows;        // rows of a K (or V) half of a layer
    unsigned long long theta[kMaxHalfDim];   // theta_i / (2 pi) * 2^64 (see rope_cos_sin)
};

// Tensor maps of the warp-specialised prefill (kvc_prefill_ws.cu), bf16 rows,
// 64-column boxes, 128-byte swizzle:
//   slot   window caches: 64 consecutive rows of a K half with their V rows,
//          5-D {64 columns, row, K|V, layer, column block} (slot_whole) or
//          4-D {column, row, K|V, layer} one column block at a time;
//   block  paged caches: {column, row, K|V, layer}, boxes of one block (bs
//          rows) of K or of V, one column block;
//   stage  the chunk's staged rows [batch][T][kv head][D] (K, then V):
//          {64 columns, kv head, batch * T, K|V, column block}, 64 tokens.
// INT8 caches: slot and block are code maps {D bytes, row, K|V, layer} with
// boxes of 128 codes of 64 rows (slot) or one block (block), no swizzle.
struct PrefillMaps {
    CUtensorMap slot, block, stage;
    int slot_whole;
};

struct TableParams {
    int32_t* table;
    uint32_t* valid;
    const int32_t* seq;
    const int32_t* lb;
    const int32_t* phys;
    const int32_t* value;
    uint32_t* err;
    int n, B, maxb, num_blocks;
};

// Block manager of a paged cache (kvc_block_prepare / _share / _release).
struct BlockParams {
    void* cache;
    const int32_t* pos;        // [B]
    int32_t* table;            // [B, maxb]
    uint32_t* valid;           // may be null
    int32_t* refcount;         // [num_blocks]
    int32_t* free_list;        // [num_blocks]: stack, entries 0 .. *free_count - 1
    int32_t* free_count;
    uint32_t* err;
    // workspace
    int32_t* tgt;              // [B]: block of the next token, -2 new, -1 none
    int32_t* rcnt;             // [B]: count of that block before the call
    int32_t* need;             // [B]: takes a block
    int32_t* aidx;             // [B]: allocation index
    int32_t* prev;             // [B]: last earlier sequence writing the same block, or -1
    int4* copies;              // [B]: (source, destination, rows, sequence)
    int32_t* ncopies;
    int32_t* flags;            // [num_blocks]: reclaimed by a release (zero between calls)
    // share / release entries
    const int32_t* src_seq;    // share: source; release: the sequences
    const int32_t* dst_seq;
    const int32_t* nblocks;
    float* scales;             // INT8 cache: row scales [layers][K|V][num_blocks * Hkv * bs]; else null
    int B, bs, num_blocks, maxb, layers, Hkv, D;
};

// bf16 and INT8 caches: tensor maps over the cache for copies of a run of
// 16 r rows (r = 1..kRunMaps), K and V of every column at once.  A column
// block is 128 bytes of a row (64 bf16 or 128 INT8 columns).  With tma_whole
// the map is 5-D {block columns, row, K|V, layer, column block} and one copy
// lands as [column block][K|V][rows][128 bytes]; otherwise it is 4-D
// {column, row, K|V, layer} and each column block is its own copy, landing
// at the same place.  INT8 caches add 3-D maps {row, K|V, layer} over the row
// scales: boxes of kScRunRows (runs) and kScSubRows (single sub-tiles) rows
// from a row index rounded down to a multiple of 4 (16-byte TMA alignment).
constexpr int kScRunRows = 68;                   // 64 + up to 3 rows of alignment, x 4 bytes = 272
constexpr int kScSubRows = 20;                   // 16 + 3, rounded to 16 bytes
struct KvTensorMaps {
    CUtensorMap run[kRunMaps];
    CUtensorMap sc_run, sc_sub;
};

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_decode(int dtype, int head_dim, int gh, bool paged, bool read_rope,
                          const DecodeParams& p, dim3 grid, cudaStream_t stream);
// bf16 and INT8 (q8) caches: tensor-core kernel fed by TMA tensor copies through `maps`.
cudaError_t launch_decode_mma(int head_dim, int gh, bool paged, bool read_rope, bool q8, const DecodeParams& p,
                              const KvTensorMaps& maps, dim3 grid, cudaStream_t stream);
cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream);
cudaError_t launch_plan_rows(const PlanParams& p, cudaStream_t stream);
cudaError_t launch_append(int dtype, const AppendParams& p, cudaStream_t stream);
cudaError_t launch_table_write(const TableParams& p, cudaStream_t stream);
// kvc_prefill: the chunk's rows staged (K rotated as stored), then attention.
cudaError_t launch_prefill_stage(const AppendParams& p, void* kst, void* vst, cudaStream_t stream);
cudaError_t launch_prefill(int head_dim, int g, const PrefillParams& p, cudaStream_t stream);
cudaError_t launch_prefill_tc(const PrefillParams& p, cudaStream_t stream);   // head_dim 128, tcgen05
// head_dim 64 / 128 / 256, warp-specialised tcgen05 with TMA tiles
cudaError_t launch_prefill_ws(int head_dim, bool q8, const PrefillParams& p, const PrefillMaps& maps,
                              cudaStream_t stream);
cudaError_t launch_valid_write(const TableParams& p, cudaStream_t stream);
cudaError_t launch_block_prepare(int elt, const BlockParams& p, cudaStream_t stream);
cudaError_t launch_block_share(const BlockParams& p, int n, cudaStream_t stream);
cudaError_t launch_block_release(const BlockParams& p, int n, cudaStream_t stream);

}  // namespace kvc
