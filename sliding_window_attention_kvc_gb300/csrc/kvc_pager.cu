// Paging of a fixed pool of block slots ([pool] "KV cache paging": a pool of
// resident slots whose size does not grow with the context; blocks move
// between host memory and the slots on demand; the copy engine moves them
// while the attention kernel runs; an LRU residency policy; blocks inside a
// sliding window stay resident and only the others page).
//
//   kvc_pager_plan    host: which needed blocks are missing, the slots they
//                     take (free slots first, then the least recently used
//                     unpinned block not needed by this step), the victims;
//   kvc_pager_evict   device, compute stream: victims' table entries -1 and
//                     valid bits cleared (before the step that no longer
//                     reads them);
//   kvc_pagein_issue  copy stream, after the compute stream's work so far:
//                     one 2-D copy per block (every layer, K and V) from
//                     pinned host memory into its slot, then an event;
//   kvc_pagein_commit compute stream waits for that event, then sets the
//                     blocks' table entries and valid bits.
#include <algorithm>
#include <cstring>
#include <vector>

#include <cuda_runtime.h>

#include "kvc.h"
#include "kvc_device.cuh"

struct kvc_pager {
    int slots = 0;
    long long step = 0;
    std::vector<int> block_of_slot;    // -1: free
    std::vector<long long> last_use;
    std::vector<char> pinned;
    cudaEvent_t after_compute = nullptr, after_copy = nullptr;
    int device = -1;
};

namespace kvc {

constexpr int kPageListMax = 1024;     // entries per table/valid update launch

struct PageListParams {
    int32_t* table;
    uint32_t* valid;
    int seq, maxb, num_blocks, n, set;
    int32_t block[kPageListMax];
    int32_t slot[kPageListMax];
};

// set: table[seq][block] = slot and the slot's valid bit on; else table
// entry -1 and the valid bit off.
__global__ void page_list_kernel(const __grid_constant__ PageListParams p) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    const int lb = p.block[i], s = p.slot[i];
    if (lb < 0 || lb >= p.maxb || s < 0 || s >= p.num_blocks) return;
    p.table[(long long)p.seq * p.maxb + lb] = p.set ? s : -1;
    if (p.valid) {
        if (p.set) atomicOr(&p.valid[s >> 5], 1u << (s & 31));
        else atomicAnd(&p.valid[s >> 5], ~(1u << (s & 31)));
    }
}

namespace {

int page_list(const kvc_desc* d, int seq, int n, const int32_t* block, const int32_t* slot, int32_t* table,
              uint32_t* valid, int set, cudaStream_t s) {
    if (!d || d->layout != KVC_LAYOUT_PAGED) return KVC_ERR_DESC;
    if (n < 0 || seq < 0 || seq >= d->batch) return KVC_ERR_ARG;
    if (n == 0) return KVC_OK;
    if (!block || !slot || !table) return KVC_ERR_NULL;
    for (int i = 0; i < n; ++i)
        if (block[i] < 0 || block[i] >= d->max_blocks_per_seq || slot[i] < 0 || slot[i] >= d->num_blocks)
            return KVC_ERR_ARG;
    for (int base = 0; base < n; base += kPageListMax) {
        PageListParams p{};
        p.table = table;
        p.valid = valid;
        p.seq = seq;
        p.maxb = d->max_blocks_per_seq;
        p.num_blocks = d->num_blocks;
        p.set = set;
        p.n = std::min(kPageListMax, n - base);
        std::memcpy(p.block, block + base, sizeof(int32_t) * p.n);
        std::memcpy(p.slot, slot + base, sizeof(int32_t) * p.n);
        page_list_kernel<<<(p.n + 127) / 128, 128, 0, s>>>(p);
        if (cudaGetLastError() != cudaSuccess) return KVC_ERR_CUDA;
    }
    return KVC_OK;
}

}  // namespace
}  // namespace kvc

extern "C" {

KVC_API kvc_pager* kvc_pager_create(int32_t num_slots) {
    if (num_slots < 1) return nullptr;
    kvc_pager* pg = new kvc_pager;
    pg->slots = num_slots;
    pg->block_of_slot.assign(num_slots, -1);
    pg->last_use.assign(num_slots, -1);
    pg->pinned.assign(num_slots, 0);
    return pg;
}

KVC_API void kvc_pager_destroy(kvc_pager* pg) {
    if (!pg) return;
    if (pg->after_compute) cudaEventDestroy(pg->after_compute);
    if (pg->after_copy) cudaEventDestroy(pg->after_copy);
    delete pg;
}

KVC_API int kvc_pager_plan(kvc_pager* pg, int32_t n, const int32_t* need, const uint8_t* pinned, int32_t* n_in,
                           int32_t* in_block, int32_t* in_slot, int32_t* n_out, int32_t* out_block,
                           int32_t* out_slot) {
    if (!pg || !n_in || !n_out) return KVC_ERR_NULL;
    if (n < 0) return KVC_ERR_ARG;
    if (n > 0 && (!need || !in_block || !in_slot || !out_block || !out_slot)) return KVC_ERR_NULL;
    const int S = pg->slots;
    std::vector<int> slot_of(n, -1);
    std::vector<char> needed(S, 0);
    for (int i = 0; i < n; ++i) {
        if (need[i] < 0) return KVC_ERR_ARG;
        for (int s = 0; s < S; ++s)
            if (pg->block_of_slot[s] == need[i]) {
                slot_of[i] = s;
                needed[s] = 1;
            }
    }
    // capacity: the needed blocks, and the pinned ones that stay, must fit
    int missing = 0, keep = 0;
    for (int i = 0; i < n; ++i) missing += slot_of[i] < 0;
    for (int s = 0; s < S; ++s) keep += needed[s] || (pg->block_of_slot[s] >= 0 && pg->pinned[s]);
    if (keep + missing > S) return KVC_ERR_ARG;
    const long long step = ++pg->step;
    int nin = 0, nout = 0;
    for (int i = 0; i < n; ++i) {
        if (slot_of[i] >= 0) continue;
        for (int j = 0; j < i; ++j)       // a block listed twice takes one slot
            if (need[j] == need[i] && slot_of[j] >= 0) slot_of[i] = slot_of[j];
        if (slot_of[i] >= 0) continue;
        int pick = -1;
        for (int s = 0; s < S && pick < 0; ++s)
            if (pg->block_of_slot[s] < 0) pick = s;
        if (pick < 0) {
            for (int s = 0; s < S; ++s) {
                if (needed[s] || pg->pinned[s]) continue;
                if (pick < 0 || pg->last_use[s] < pg->last_use[pick]) pick = s;
            }
            out_block[nout] = pg->block_of_slot[pick];
            out_slot[nout] = pick;
            ++nout;
        }
        pg->block_of_slot[pick] = need[i];
        pg->pinned[pick] = 0;
        needed[pick] = 1;
        slot_of[i] = pick;
        in_block[nin] = need[i];
        in_slot[nin] = pick;
        ++nin;
    }
    for (int i = 0; i < n; ++i) {
        pg->last_use[slot_of[i]] = step;
        if (pinned) pg->pinned[slot_of[i]] = pinned[i] ? 1 : 0;
    }
    *n_in = nin;
    *n_out = nout;
    return KVC_OK;
}

KVC_API int kvc_pager_evict(const kvc_desc* d, int32_t seq, int32_t n, const int32_t* out_block,
                            const int32_t* out_slot, int32_t* block_table, uint32_t* valid_bits, void* stream) {
    return kvc::page_list(d, seq, n, out_block, out_slot, block_table, valid_bits, 0, (cudaStream_t)stream);
}

KVC_API int kvc_pagein_issue(kvc_pager* pg, const kvc_desc* d, void* cache, const void* host_kv, int32_t n,
                             const int32_t* in_block, const int32_t* in_slot, void* copy_stream,
                             void* compute_stream) {
    if (!pg || !d) return KVC_ERR_NULL;
    if (d->layout != KVC_LAYOUT_PAGED) return KVC_ERR_DESC;
    if (d->dtype == KVC_I8) return KVC_ERR_UNSUPPORTED;   // host blocks hold no row scales
    if (n < 0) return KVC_ERR_ARG;
    if (n > 0 && (!cache || !host_kv || !in_block || !in_slot)) return KVC_ERR_NULL;
    // every entry is checked before anything is recorded or copied
    for (int i = 0; i < n; ++i)
        if (in_block[i] < 0 || in_block[i] >= d->max_blocks_per_seq || in_slot[i] < 0 || in_slot[i] >= d->num_blocks)
            return KVC_ERR_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVC_ERR_CUDA;
    if (pg->device != dev) {
        if (pg->after_compute) cudaEventDestroy(pg->after_compute);
        if (pg->after_copy) cudaEventDestroy(pg->after_copy);
        if (cudaEventCreateWithFlags(&pg->after_compute, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&pg->after_copy, cudaEventDisableTiming) != cudaSuccess)
            return KVC_ERR_CUDA;
        pg->device = dev;
    }
    const size_t elt = d->dtype == KVC_F32 ? 4 : 2;
    const size_t block_bytes = (size_t)d->kv_heads * d->block_size * d->head_dim * elt;   // one (layer, K|V)
    const size_t plane = (size_t)d->num_blocks * block_bytes;                           // cache stride per (layer, K|V)
    cudaStream_t cs = (cudaStream_t)copy_stream, ks = (cudaStream_t)compute_stream;
    // the slots may only be written once the compute stream's work so far
    // (the victims' eviction, and whatever read them before it) is done
    if (cudaEventRecord(pg->after_compute, ks) != cudaSuccess) return KVC_ERR_CUDA;
    if (cudaStreamWaitEvent(cs, pg->after_compute, 0) != cudaSuccess) return KVC_ERR_CUDA;
    for (int i = 0; i < n; ++i) {
        // host: [logical block][layer][K|V][kv head][row][D]; device: [layer][K|V][slot][kv head][row][D]
        const char* src = static_cast<const char*>(host_kv) + (size_t)in_block[i] * d->layers * 2 * block_bytes;
        char* dst = static_cast<char*>(cache) + (size_t)in_slot[i] * block_bytes;
        if (cudaMemcpy2DAsync(dst, plane, src, block_bytes, block_bytes, (size_t)d->layers * 2,
                              cudaMemcpyHostToDevice, cs) != cudaSuccess)
            return KVC_ERR_CUDA;
    }
    if (cudaEventRecord(pg->after_copy, cs) != cudaSuccess) return KVC_ERR_CUDA;
    return KVC_OK;
}

KVC_API int kvc_pagein_commit(kvc_pager* pg, const kvc_desc* d, int32_t seq, int32_t n, const int32_t* in_block,
                              const int32_t* in_slot, int32_t* block_table, uint32_t* valid_bits,
                              void* compute_stream) {
    if (!pg) return KVC_ERR_NULL;
    cudaStream_t ks = (cudaStream_t)compute_stream;
    if (pg->after_copy && cudaStreamWaitEvent(ks, pg->after_copy, 0) != cudaSuccess) return KVC_ERR_CUDA;
    return kvc::page_list(d, seq, n, in_block, in_slot, block_table, valid_bits, 1, ks);
}

}  // extern "C"
