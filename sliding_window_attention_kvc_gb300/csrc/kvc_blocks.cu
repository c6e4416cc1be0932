// Block manager of a paged cache on the device: each sequence's next block
// made mapped, private and resident (allocation from a free list, copy-on-
// write of shared blocks), prefix sharing with reference counts, release.
// [share] "Shared state, isolated problems: KV cache and batching": §3.1 and
// §5.1 (blocks from a free list through a block table), §3.2 and §5.1
// (prefix sharing raises reference counts; a block referenced more than once
// is copied before it is written), §6.1 (reclaim only when a count reaches 0).
//
// Determinism: the free list is a stack; within one call, sequences are served
// in ascending order exactly as one after the other would be, so that the
// tables, counts and free list equal those of a sequential block manager.
#include "kvc_decode.cuh"

namespace kvc {

constexpr int kBlockThreads = 1024;
constexpr uint32_t kDevNoFreeBlock = 0x40u;   // KVC_DEV_NO_FREE_BLOCK

// Block-wide exclusive scan of one int per thread (kBlockThreads threads).
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int NW = kBlockThreads / 32;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += u;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = s_warp[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += u;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    const int excl = x - v + (warp > 0 ? s_warp[warp - 1] : 0);
    *total = s_warp[NW - 1];
    __syncthreads();
    return excl;
}

// Target of sequence b's next token: its block's physical id (>= 0), or
// kNewBlock (unmapped, token at a block's first row), or kNoTarget.
constexpr int kNewBlock = -2, kNoTarget = -1;

// One CTA, in passes over the sequences: (1) each sequence's target and the
// count of that block before the call; (2) its rank k among the earlier
// sequences writing the same block and whether it takes a block (a shared
// block copies while r - k > 1; an unmapped block at its first row is new);
// (3) allocation index = exclusive scan of "takes a block" in sequence order;
// (4) apply.  A sequence writing in place after an earlier sharer failed to
// get a block fails too (in the sequential order the count it sees is still
// above one).
__global__ void __launch_bounds__(kBlockThreads) block_prepare_kernel(const __grid_constant__ BlockParams p) {
    __shared__ int s_warp[32];
    const int tid = threadIdx.x;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int free0 = *p.free_count;
    for (int b = tid; b < p.B; b += kBlockThreads) {
        const int t = p.pos[b];
        int tgt = kNoTarget;
        if (t >= 0) {
            const long long lb = t / p.bs;
            if (lb >= p.maxb) {
                set_error(p.err, 0x4u /* KVC_DEV_BAD_POSITION */);
            } else {
                const int phys = p.table[(long long)b * p.maxb + lb];
                if (phys >= p.num_blocks) {
                    set_error(p.err, 0x1u /* KVC_DEV_BAD_BLOCK */);
                } else if (phys >= 0) {
                    tgt = phys;
                } else if (t % p.bs == 0) {
                    tgt = kNewBlock;
                } else {
                    set_error(p.err, 0x2u /* KVC_DEV_UNMAPPED_APPEND */);
                }
            }
        }
        p.tgt[b] = tgt;
        p.rcnt[b] = tgt >= 0 ? p.refcount[tgt] : 0;
    }
    __syncthreads();
    for (int b = tid; b < p.B; b += kBlockThreads) {
        const int tgt = p.tgt[b];
        int rank = 0, prev = -1, need = 0;
        if (tgt >= 0) {
            for (int q = 0; q < b; ++q)
                if (p.tgt[q] == tgt) {
                    ++rank;
                    prev = q;
                }
            need = p.rcnt[b] - rank > 1 ? 1 : 0;
        } else if (tgt == kNewBlock) {
            need = 1;
        }
        p.need[b] = need;
        p.prev[b] = rank > 0 ? prev : -1;
    }
    __syncthreads();
    int carry = 0;
    for (int base = 0; base < p.B; base += kBlockThreads) {
        const int b = base + tid;
        const int need = b < p.B ? p.need[b] : 0;
        int total = 0;
        const int idx = carry + block_exclusive_scan(need, s_warp, &total);
        if (b < p.B) p.aidx[b] = idx;
        carry += total;
    }
    __syncthreads();
    for (int b = tid; b < p.B; b += kBlockThreads) {
        const int tgt = p.tgt[b];
        if (p.need[b]) {
            const int idx = p.aidx[b];
            if (idx >= free0) {
                set_error(p.err, kDevNoFreeBlock);
                continue;
            }
            const int f = p.free_list[free0 - 1 - idx];
            if (f < 0 || f >= p.num_blocks) {
                index_fault(p.err, 30, f);
                continue;
            }
            const long long lb = p.pos[b] / p.bs;
            p.refcount[f] = 1;
            if (p.valid) atomicOr(&p.valid[f >> 5], 1u << (f & 31));
            p.table[(long long)b * p.maxb + lb] = f;
            if (tgt >= 0) {
                atomicSub(&p.refcount[tgt], 1);
                const int slot = atomicAdd(p.ncopies, 1);
                p.copies[slot] = make_int4(tgt, f, p.pos[b] % p.bs, b);
            }
        } else if (tgt >= 0 && p.prev[b] >= 0) {
            const int q = p.prev[b];
            if (p.need[q] && p.aidx[q] >= free0) set_error(p.err, kDevNoFreeBlock);
        }
    }
    if (tid == 0) *p.free_count = free0 - (carry < free0 ? carry : free0);
}

// One CTA per (copy slot, layer x K|V x kv head): the first `rows` rows of the
// shared block go to the new private one.
template <typename Elt>
__global__ void __launch_bounds__(256) block_copy_kernel(const __grid_constant__ BlockParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int i = blockIdx.x;
    if (i >= *p.ncopies) return;
    const int4 c = p.copies[i];
    const int lkh = blockIdx.y;                          // (layer * 2 + kv) * Hkv + h
    const int h = lkh % p.Hkv, lk = lkh / p.Hkv;
    const long long per_half = (long long)p.num_blocks * p.Hkv * p.bs * p.D;
    const long long blk_elems = (long long)p.bs * p.D;
    const Elt* src = static_cast<const Elt*>(p.cache) + lk * per_half + ((long long)c.x * p.Hkv + h) * blk_elems;
    Elt* dst = static_cast<Elt*>(p.cache) + lk * per_half + ((long long)c.y * p.Hkv + h) * blk_elems;
    const int n16 = c.z * p.D * (int)sizeof(Elt) / 16;   // 16-byte chunks of the rows to copy
    for (int k = threadIdx.x; k < n16; k += blockDim.x)
        reinterpret_cast<uint4*>(dst)[k] = reinterpret_cast<const uint4*>(src)[k];
    if (p.scales) {                                      // INT8 cache: the rows' scales too
        const long long rows_half = (long long)p.num_blocks * p.Hkv * p.bs;
        const float* ss = p.scales + lk * rows_half + ((long long)c.x * p.Hkv + h) * p.bs;
        float* sd = p.scales + lk * rows_half + ((long long)c.y * p.Hkv + h) * p.bs;
        for (int k = threadIdx.x; k < c.z; k += blockDim.x) sd[k] = ss[k];
    }
}

// One CTA per share entry: dst's logical blocks 0 .. nblocks-1 point at src's
// (which must all be unmapped in dst); counts rise by one.
__global__ void __launch_bounds__(256) block_share_kernel(const __grid_constant__ BlockParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int e = blockIdx.x;
    const int src = p.src_seq[e], dst = p.dst_seq[e], nb = p.nblocks[e];
    if (src < 0 || src >= p.B || dst < 0 || dst >= p.B || nb < 0 || nb > p.maxb || src == dst) {
        if (threadIdx.x == 0) set_error(p.err, 0x10u /* KVC_DEV_BAD_ENTRY */);
        return;
    }
    int mapped = 0;
    for (int lb = threadIdx.x; lb < nb; lb += blockDim.x) mapped |= p.table[(long long)dst * p.maxb + lb] >= 0;
    if (__syncthreads_or(mapped)) {
        if (threadIdx.x == 0) set_error(p.err, 0x10u);
        return;
    }
    for (int lb = threadIdx.x; lb < nb; lb += blockDim.x) {
        const int phys = p.table[(long long)src * p.maxb + lb];
        if (phys >= 0 && phys < p.num_blocks) {
            p.table[(long long)dst * p.maxb + lb] = phys;
            atomicAdd(&p.refcount[phys], 1);
        }
    }
}

// Release, pass 1: one CTA per listed sequence; every mapped block's count
// drops by one and the entry is unmapped; blocks reaching zero are flagged.
__global__ void __launch_bounds__(256) block_release_kernel(const __grid_constant__ BlockParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int b = p.src_seq[blockIdx.x];
    if (b < 0 || b >= p.B) {
        if (threadIdx.x == 0) set_error(p.err, 0x10u);
        return;
    }
    for (int lb = threadIdx.x; lb < p.maxb; lb += blockDim.x) {
        int32_t* e = p.table + (long long)b * p.maxb + lb;
        const int phys = *e;
        if (phys < 0) continue;
        *e = -1;
        if (phys >= p.num_blocks) {
            set_error(p.err, 0x1u);
            continue;
        }
        if (atomicSub(&p.refcount[phys], 1) == 1) p.flags[phys] = 1;
    }
}

// Release, pass 2 (one CTA): flagged blocks go back on the free list in
// ascending id and lose their residency bit.
__global__ void __launch_bounds__(kBlockThreads) block_reclaim_kernel(const __grid_constant__ BlockParams p) {
    __shared__ int s_warp[32];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int free0 = *p.free_count;
    int carry = 0;
    for (int base = 0; base < p.num_blocks; base += kBlockThreads) {
        const int f = base + threadIdx.x;
        const int fl = f < p.num_blocks ? p.flags[f] : 0;
        int total = 0;
        const int idx = carry + block_exclusive_scan(fl, s_warp, &total);
        if (fl) {
            if (free0 + idx < p.num_blocks) p.free_list[free0 + idx] = f;
            else index_fault(p.err, 31, f);
            if (p.valid) atomicAnd(&p.valid[f >> 5], ~(1u << (f & 31)));
            p.flags[f] = 0;
        }
        carry += total;
    }
    if (threadIdx.x == 0) *p.free_count = free0 + carry;
}

namespace {
cudaLaunchConfig_t pdl_config(dim3 grid, int threads, cudaStream_t s, cudaLaunchAttribute* attr) {
    attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr->val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}
}  // namespace

cudaError_t launch_block_prepare(int elt, const BlockParams& p, cudaStream_t s) {
    cudaLaunchAttribute attr;
    cudaError_t e = cudaMemsetAsync(p.ncopies, 0, sizeof(int), s);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = pdl_config(dim3(1), kBlockThreads, s, &attr);
    e = cudaLaunchKernelEx(&cfg, block_prepare_kernel, p);
    if (e != cudaSuccess) return e;
    cfg = pdl_config(dim3(p.B, p.layers * 2 * p.Hkv), 256, s, &attr);
    return elt == 4   ? cudaLaunchKernelEx(&cfg, block_copy_kernel<float>, p)
           : elt == 2 ? cudaLaunchKernelEx(&cfg, block_copy_kernel<__nv_bfloat16>, p)
                      : cudaLaunchKernelEx(&cfg, block_copy_kernel<int8_t>, p);
}

cudaError_t launch_block_share(const BlockParams& p, int n, cudaStream_t s) {
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = pdl_config(dim3(n), 256, s, &attr);
    return cudaLaunchKernelEx(&cfg, block_share_kernel, p);
}

cudaError_t launch_block_release(const BlockParams& p, int n, cudaStream_t s) {
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = pdl_config(dim3(n), 256, s, &attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, block_release_kernel, p);
    if (e != cudaSuccess) return e;
    cfg = pdl_config(dim3(1), kBlockThreads, s, &attr);
    return cudaLaunchKernelEx(&cfg, block_reclaim_kernel, p);
}

}  // namespace kvc
