// Split-K decode attention for bf16 and INT8 caches on the tensor cores,
// stream-K.
//
// Work decomposition.  For each (kv head, q-head group) the attended rows of
// all sequences, laid end to end, are cut into gridDim.x nearly equal
// contiguous shares, one per CTA (a persistent grid of two CTAs per SM).  A
// share covers one or more *segments* (its intersection with one sequence);
// a CTA reduces each segment to a partial (m, l, o) per q head, and
// combine_streamk_kernel, launched behind it with programmatic dependent
// launch, merges each sequence's few partials:
//     M = max m_i,  out = sum o_i 2^(m_i - M) / sum l_i 2^(m_i - M).
// With shares in sequence order, segment (CTA x, sequence b) gets partial
// slot x + b: consecutive, unique, and a sequence's slots are consecutive.
//
// Contractions of a GQA group by mma.sync m16n8k16 (bf16 in, fp32 acc):
//     S = Q K^T   A = the group's q heads (rows 0..GH-1 of 16; the rest zero),
//                 B = K rows of a 16-token sub-tile, k = head_dim;
//     O += P V    A = exp2(S - m) rounded to bf16, B = V rows, k = 16 tokens.
// On a q head group of 4 the CUDA-core formulation spent ~97 warp
// instructions per cached token (measured); these two products cost ~4.
// INT8 rows (the Q8 variant) enter as fp16: codes are exact in fp16, q is
// scaled by a power of two per head, and P V is computed as V^T P^T so that
// a lane's V bytes form A fragments (see the Q8 branches below).
//
// Data movement.  Warp 4 walks the CTA's segments and cuts them into *runs*
// of up to 64 consecutive cache rows (a paged block, or the slots of a ring
// between its boundaries).  One TMA tensor copy (cp.async.bulk.tensor) per run
// brings the run's K and V rows, every column, into a ring of shared-memory
// stages guarded by mbarriers, laid out [64-column block][K|V][rows][128 B]
// with the 128-byte swizzle, so that ldmatrix reads of 8 rows at one column
// are bank-conflict free.  Issuing copies was the bottleneck with one 2 KB
// box per (16 rows, 64 columns, K or V): ~70 cycles per copy instruction plus
// the bookkeeping around it, against a stage's worth of tensor-core work.
// Warps 0..3 compute, one 16-row sub-tile of a stage each.  Each sub-tile
// carries its row count (ragged ends, partial paged blocks), its place in the
// stage and, for READ_INCACHE, its first in-cache position.  Rows of a
// sub-tile past its row count are masked out of the softmax and their V rows
// zeroed before P V (they may hold any bits, NaN included).
#pragma once

#include <cuda.h>

#include <atomic>

#include "kvc_decode.cuh"

namespace kvc {

template <int D, bool READ, bool Q8 = false, bool PAGED = false>
struct MmaShape {
    static constexpr int kSub = 16;                           // rows per sub-tile
    static constexpr int kBoxCols = Q8 ? 128 : 64;            // columns per TMA box row (128 bytes)
    static constexpr int kBoxes = D / kBoxCols;               // boxes per row of K (or V)
    static constexpr int kBoxBytes = kSub * 128;              // one 16-row box
    static constexpr int kSubBytes = kBoxes * kBoxBytes;      // K (or V) of one sub-tile
    static constexpr int kDsplit = D == 256 ? 2 : 1;          // warps sharing one sub-tile (split over dims)
    static constexpr int kTokenGroups = kConsumerWarps / kDsplit;
    static constexpr int kNsub = kTokenGroups;                // sub-tiles per stage (one per token group)
    static constexpr int kStageBytes = 2 * kNsub * kSubBytes; // K and V of kNsub sub-tiles
    static constexpr int kCtasPerSm = decode_ctas_per_sm(Q8, PAGED, READ, D);
    static constexpr int kStages =
        Q8 ? (kCtasPerSm >= 3 ? 3 : ((READ && D < 256) ? 4 : 5)) : (D == 64 ? 6 : ((READ && D >= 256) ? 5 : 3));
    // INT8: row scales of each stage, one slot per sub-tile position (the
    // first sub-tile of a copy holds that copy's K and V scales)
    static constexpr int kScSlotBytes = Q8 ? 640 : 0;         // 2 x kScRunRows floats, 128-byte aligned
    static constexpr int kScSlotFloats = kScSlotBytes / 4;
    static constexpr int kScStageBytes = kNsub * kScSlotBytes;
    // READ_INCACHE rotation: a lane owns one 16-byte chunk pair (8 rotation
    // pairs) of kRowsPerLane rows of its warp's sub-tile
    static constexpr int kCpr = D / 16;                       // chunk pairs (i, i + D/2) per row
    static constexpr int kRowGroups = 32 / kCpr;              // rows a warp visits at once
    static constexpr int kRowsPerLane = kSub / (kDsplit * kRowGroups);
    static constexpr int kDl = D / kDsplit;                   // output columns per warp
    static constexpr int kNt = kDl / 8;                       // 8-column output tiles per warp
    static constexpr int kKsteps = D / 16;                    // k-steps of Q K^T
    static constexpr int kHalf = D / 2;
};

// Segment header, carried by the first stage of each segment.
struct MmaSegment {
    int b;           // sequence
    int t;           // its current position
    int slot;        // partial slot of this segment
    int first_slot;  // first partial slot of the sequence
    int nparts;      // partials of the sequence
    int new_row;     // self-planned paged step: K-half row that receives the new token, else -1
    int pad[2];
};

// A single paged sequence's plan, made by each decode CTA for itself.
struct SelfPlan {
    int G;           // shares of the attended rows
    int lb, row;     // share blockIdx.x: first logical block, and first row in it
    int rows;        // rows of the share
    int phys;        // physical block of lb
    int traw;        // the sequence's position
    int tphys;       // physical block of the logical block holding traw (-1: unmapped or none)
    int tattended;   // that block is attended (mapped and valid)
};

// Plan of a one-sequence paged cache, by all threads of the CTA ([pool]
// "kernel forgets absent blocks": logical blocks <= t / bs that are mapped and
// valid; the last one up to row t mod bs).  The table and the valid words are
// staged in shared memory with coalesced loads (s_tab, s_val: the pipeline
// stages, not yet in use).  Warp w looks at logical blocks [1024 w, 1024 (w + 1)),
// 32 at a time; a ballot per 32 gives the attended blocks, and a scan of the
// warps' counts their ranks.  Every attended block but the sequence's last
// holds bs rows, so row r of the attended rows lies in the attended block of
// rank r / bs, at row r mod bs.  Shares: [floor(x R / G), floor((x + 1) R / G))
// with G = min(R, shares) (1 when R = 0), as the plan kernel cuts them.
// The parameters arrive by value: read through a reference to the kernel's
// parameter block, every field access would be a generic load.
struct SelfPlanArgs {
    const int32_t* table;
    const uint32_t* valid;
    const int32_t* pos;
    uint32_t* err;
    int2* seq_items;
    int maxb, num_blocks, bs, nsplit;
};

// speculative: a plan made before the previous kernel in the stream has
// finished, from the table as it stands, for prefetch hints only: it writes
// nothing to global memory and reports no error.  `parity`: the phase of
// `bar` this call's copies complete.
static __device__ __noinline__ void self_plan_single(const SelfPlanArgs p, SelfPlan* sp, int* s_red,
                                                     int32_t* s_tab, uint32_t* s_val, uint64_t* bar,
                                                     uint32_t parity, bool speculative) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NW = kDecodeThreads / 32;
    // warp w covers table entries [1024 w, 1024 w + 1024), one 32-entry group per step
    static_assert(NW * 1024 >= kSelfPlanMax, "the warps' ranges cover the table");
    const int maxb = p.maxb, nvw = (p.num_blocks + 31) >> 5;
    // the table and the valid words land in shared memory by bulk copies of
    // their whole 16-byte multiples (the host takes this path only for 16-byte
    // aligned buffers), completing on `bar`; the last 1-3 entries of each are
    // loaded by threads
    const int tab4 = maxb & ~3, val4 = p.valid ? (nvw & ~3) : 0;
    if (tid == 0) {
        mbar_expect_tx(bar, (uint32_t)((tab4 + val4) * 4));
        if (tab4) bulk_load(s_tab, p.table, (uint32_t)(tab4 * 4), bar);
        if (val4) bulk_load(s_val, p.valid, (uint32_t)(val4 * 4), bar);
        mbar_arrive(bar);
    }
    if (tid < maxb - tab4) s_tab[tab4 + tid] = __ldcg(p.table + tab4 + tid);
    if (p.valid) {
        if (tid < nvw - val4) s_val[val4 + tid] = __ldcg(p.valid + val4 + tid);
    } else {
        for (int i = tid; i < nvw; i += kDecodeThreads) s_val[i] = 0xffffffffu;
    }
    const int traw = __ldcg(p.pos);
    if (!mbar_wait(bar, parity)) {
        // the copies never landed: plan nothing (every share empty)
        if (tid == 0 && !speculative) set_error(p.err, 0x8u /* KVC_DEV_TIMEOUT */);
        for (int i = tid; i < maxb; i += kDecodeThreads) s_tab[i] = -1;
    }
    if (tid == 0) {
        sp->tphys = -1;
        sp->tattended = 0;
        sp->lb = sp->row = sp->rows = 0;
        sp->phys = -1;
    }
    __syncthreads();
    const int t = clamp_paged_t(traw, maxb, p.bs);
    const int nb = t < 0 ? 0 : t / p.bs + 1;
    const int last_rows = t < 0 ? 0 : t - (nb - 1) * p.bs + 1;
    const bool reporter = !speculative && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
    bool bad = false;
    auto attended = [&](int e) -> bool {
        if (e >= nb) return false;
        const int q = s_tab[e];
        if (q < 0) return false;
        if (q >= p.num_blocks) {
            bad = true;
            return false;
        }
        return (s_val[q >> 5] >> (q & 31)) & 1u;
    };
    // lane k keeps the ballot of the warp's k-th group of 32 blocks (a short
    // loop: this runs once per launch, from a cold instruction cache)
    uint32_t my_m = 0;
    int cnt = 0;
    const int nbk = p.num_blocks;
#pragma unroll 4
    for (int k = 0; k < 32; ++k) {
        // branch-free: both shared-memory reads issued unconditionally
        const int e = warp * 1024 + k * 32 + lane;
        const int q = s_tab[e < nb ? e : 0];
        const bool in = e < nb && q >= 0 && q < nbk;
        const uint32_t w = s_val[in ? (q >> 5) : 0];
        bad |= e < nb && q >= nbk;
        const uint32_t mk = __ballot_sync(0xffffffffu, in && ((w >> (q & 31)) & 1u));
        if (lane == k) my_m = mk;
        cnt += __popc(mk);
    }
    if (bad && reporter) set_error(p.err, 0x1u /* KVC_DEV_BAD_BLOCK */);
    if (lane == 0) s_red[warp] = cnt;
    __syncthreads();
    int before = 0, nblk = 0;
#pragma unroll 1
    for (int k = 0; k < NW; ++k) {
        const int c = s_red[k];
        before += k < warp ? c : 0;
        nblk += c;
    }
    const bool last_att = nb > 0 && attended(nb - 1);
    const int R = nblk * p.bs - (last_att ? p.bs - last_rows : 0);
    const int G = R < p.nsplit ? (R > 0 ? R : 1) : p.nsplit;
    const int x = blockIdx.x;
    if (x < G && R > 0) {
        const int lo = (int)((long long)x * R / G), hi = (int)((long long)(x + 1) * R / G);
        const int kb = lo / p.bs;                       // rank of the share's first block
        if (kb >= before && kb < before + cnt) {        // in this warp's blocks (warp-uniform)
            const int c = __popc(my_m);
            int incl = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += u;
            }
            const int j = kb - before - (incl - c);     // its rank among this lane's 32 blocks
            if (j >= 0 && j < c) {
                uint32_t mm = my_m;
#pragma unroll 1
                for (int q = 0; q < j; ++q) mm &= mm - 1u;
                const int e = warp * 1024 + lane * 32 + (__ffs(mm) - 1);
                sp->lb = e;
                sp->row = lo - kb * p.bs;
                sp->rows = hi - lo;
                sp->phys = s_tab[e];
            }
        }
    }
    // the block that receives the step's new token (kvc_decode_step)
    if (tid == 0 && traw >= 0 && traw == t) {
        const int tlb = traw / p.bs;
        sp->tphys = s_tab[tlb];
        sp->tattended = attended(tlb);
    }
    if (tid == 0) {
        sp->G = G;
        sp->traw = traw;
        if (reporter) p.seq_items[0] = make_int2(0, G);   // the combine's view of the partials
    }
    // the staged table leaves the stages to the tensor copies
    fence_proxy_async_smem();
    __syncthreads();
}

struct alignas(16) MmaStageMeta {
    int nsub;        // sub-tiles in the stage (0 allowed); -1 = end of the stream
    int flags;       // kSegBegin | kSegEnd
    int pad[2];
    int nrows[4];    // rows of each sub-tile (1..16)
    int ip0[4];      // READ_INCACHE: in-cache position of row 0 of each sub-tile
    int newrow[4];   // fused append: row of the sub-tile that holds the new token, else -1
    int base[4];     // byte offset of each sub-tile's K rows (column block 0) in the stage
    int ld[4];       // rows of the copy the sub-tile belongs to: its K|V and column
                     // blocks lie 128 * ld bytes apart
    int sbase[4];    // INT8: float index of the K scale of row 0 in the stage's scale area
    int sld[4];      // INT8: floats from a K scale to the V scale of the same row
    MmaSegment seg;  // valid with kSegBegin
};
constexpr int kSegBegin = 1, kSegEnd = 2;

template <int D, int GH, bool READ, bool Q8 = false, bool PAGED = false>
struct MmaSmem {
    using S = MmaShape<D, READ, Q8, PAGED>;
    static constexpr size_t kStage = 0;                                        // 1024-aligned stages
    static constexpr size_t kSc = kStage + (size_t)S::kStages * S::kStageBytes;  // INT8 row scales
    static constexpr size_t kBars = kSc + (size_t)S::kStages * S::kScStageBytes;
    static constexpr size_t kMeta = kBars + 2 * S::kStages * sizeof(uint64_t);
    // READ_INCACHE: R(ip0 theta_i) of each sub-tile, [stage][sub][4][D/16][2] float2
    // (pair i = 8 cp + 2 jj + e at [jj][cp][e], so a lane's float4 loads are conflict-free)
    static constexpr size_t kRot = kMeta + S::kStages * sizeof(MmaStageMeta);
    static constexpr size_t kQcs = kRot + (READ ? (size_t)S::kStages * S::kNsub * S::kHalf * 8 : 0);  // [D/2] float2
    static constexpr size_t kMergeO = kQcs + (size_t)S::kHalf * 8;
    static constexpr size_t kMergeML = kMergeO + (size_t)S::kTokenGroups * GH * D * 4;
    static constexpr size_t kHdr = kMergeML + (size_t)S::kTokenGroups * GH * 8;   // the CTA's first segment header
    // 4 mbarriers: all compute warps, 2 warp pairs, first header published
    static constexpr size_t kCbar = kHdr + sizeof(MmaSegment);
    // INT8 with read-time RoPE: each token group's K sub-tile, dequantised and
    // rotated, in bf16 ([D/64 column blocks][16 rows][128 bytes], 16-byte
    // chunks swizzled by row as the bf16 stages are)
    static constexpr size_t kKrot = (kCbar + 32 + 127) / 128 * 128;
    static constexpr size_t kTotal =
        kKrot + ((Q8 && READ) ? (size_t)S::kTokenGroups * S::kSub * D * 2 : 0) + 1024;   // + slack to align the base
};

// Barrier among a fixed set of threads built on an mbarrier, so that waiting
// is bounded like every other wait in these kernels (a hardware named barrier
// would wait forever for a warp that gave up and left).
struct BoundedBarrier {
    uint64_t* bar;
    uint32_t phase;
    __device__ __forceinline__ bool sync(uint32_t* err) {
        mbar_arrive(bar);
        const bool ok = mbar_wait(bar, phase);
        phase ^= 1u;
        if (!ok) set_error(err, 0x8u /* KVC_DEV_TIMEOUT */);
        return ok;
    }
};

// Programmatic dependent launch: wait for the preceding kernel in the stream
// to complete (its writes visible), and let the next one start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Stream-K partition of a window layout for one (kv head, q-head group):
// sequence b contributes max(1, ceil(n_live(b) / 16)) sub-tiles.  Returns the
// grand total and b's offset and size to every lane of the calling warp.
__device__ __forceinline__ void window_partition(const DecodeParams& p, int b, long long* total, long long* Ob,
                                                 long long* Sb) {
    const int lane = threadIdx.x & 31;
    const int C = p.capacity;
    long long tot = 0, before = 0, sb = 0;
    for (int base = 0; base < p.B; base += 32) {
        const int bb = base + lane;
        long long st = 0;
        if (bb < p.B) {
            const int tb = p.pos[bb];
            const int nl = tb < 0 ? 0 : (tb + 1 < C ? tb + 1 : C);
            st = (nl > 0 ? (nl + 15) / 16 : 1) + kSeqUnits;
        }
        long long pre = bb < b ? st : 0;
        long long me = bb == b ? st : 0;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            st += __shfl_xor_sync(0xffffffffu, st, off);
            pre += __shfl_xor_sync(0xffffffffu, pre, off);
            me += __shfl_xor_sync(0xffffffffu, me, off);
        }
        tot += st;
        before += pre;
        sb += me;
    }
    *total = tot;
    *Ob = before;
    *Sb = sb;
}

// The same for a paged batch: its attended rows (plan_rows_kernel's seq_rows),
// and those of the sequences before b.
__device__ __forceinline__ void paged_partition(const DecodeParams& p, int b, long long* total, long long* Ob,
                                                long long* Rb) {
    const int lane = threadIdx.x & 31;
    long long tot = 0, before = 0, rb = 0;
    for (int base = 0; base < p.B; base += 32) {
        const int bb = base + lane;
        long long st = bb < p.B ? (long long)__ldcg(p.seq_rows + bb) : 0;
        long long pre = bb < b ? st : 0;
        long long me = bb == b ? st : 0;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            st += __shfl_xor_sync(0xffffffffu, st, off);
            pre += __shfl_xor_sync(0xffffffffu, pre, off);
            me += __shfl_xor_sync(0xffffffffu, me, off);
        }
        tot += st;
        before += pre;
        rb += me;
    }
    *total = tot;
    *Ob = before;
    *Rb = rb;
}

// ---------------------------------------------------------------------------
// Combine kernel for the stream-K decode: one CTA per (sequence, kv head,
// q-head group, COLS-column chunk).  out = sum_i o_i 2^(m_i - M) / sum_i l_i 2^(m_i - M)
// over the sequence's partials, M = max m_i; an empty attended set gives 0.
// One warp per q head finds M and L; threads then split the partials into
// groups (four loads in flight each) and reduce through shared memory.
// ---------------------------------------------------------------------------
constexpr int kCombineThreads = 256;

// COLS columns per CTA: 16 when (sequence, kv head, group) units are few (more
// CTAs per unit, shorter chains), 128 (64 at head_dim 64) when they already
// fill a wave of CTAs.
template <int D, int GH, bool PAGED, int COLS>
__global__ void __launch_bounds__(kCombineThreads) combine_streamk_kernel(const __grid_constant__ DecodeParams p) {
    constexpr int C4 = COLS / 4;                   // float4 columns per chunk
    constexpr int PAIRS = GH * C4;                 // (head, float4) outputs of the chunk
    constexpr int PG = kCombineThreads / PAIRS;    // partial groups
    constexpr int kMaxStaged = 1024;
    __shared__ float2 s_ml[kMaxStaged];
    __shared__ float s_M[GH], s_L[GH];
    __shared__ float4 s_part[kCombineThreads];

    // the next kernel in the stream may begin launching; it waits for this
    // grid to complete before it reads anything
    pdl_launch_dependents();
    const int b = blockIdx.x;
    const int kvh = blockIdx.y / p.nsub, z = blockIdx.y % p.nsub;
    const int col0 = blockIdx.z * COLS;
    const int tid = threadIdx.x;
    const int qh0 = kvh * p.G + z * GH;

    // which partial slots belong to sequence b (inputs that the decode kernel does not write)
    int first = 0, nparts = 0;
    __shared__ int s_fn[2];
    if (PAGED && !p.seq_rows) {
        pdl_wait();                                 // one self-planned sequence: the decode kernel's count
        const int2 si = p.seq_items[b];
        first = si.x;
        nparts = si.y;
    } else if (PAGED) {
        // a batch: the shares that meet b, from the plan's rows (written before
        // the decode kernel started, so before this grid launched)
        if (tid < 32) {
            long long R, Ob, Rb;
            paged_partition(p, b, &R, &Ob, &Rb);
            const int2 fl = paged_seq_shares(Ob, Rb, R, paged_share_count(R, p.nsplit));
            if (tid == 0) {
                s_fn[0] = fl.x + b;
                s_fn[1] = fl.y - fl.x + 1;
            }
        }
        __syncthreads();
        first = s_fn[0];
        nparts = s_fn[1];
        pdl_wait();                                 // the decode kernel's partials
    } else {
        if (tid < 32) {
            long long total, Ob, Sb;
            window_partition(p, b, &total, &Ob, &Sb);
            const int G = (int)(total < p.nsplit ? total : p.nsplit);
            const int fx = streamk_share_of(Ob, total, G);
            const int lx = streamk_share_of(Ob + Sb - 1, total, G);
            if (tid == 0) {
                s_fn[0] = fx + b;
                s_fn[1] = lx - fx + 1;
            }
        }
        __syncthreads();
        first = s_fn[0];
        nparts = s_fn[1];
        pdl_wait();                                 // the decode kernel's partials
    }
    // the decode grid is done: ready its share counter, and a paged batch's
    // block reader counts, for the next call
    if (blockIdx.x == 0 && blockIdx.z == 0 && tid == 0) p.counters[blockIdx.y] = 0u;
    if (PAGED && p.refs) {
        const long long ncta = (long long)gridDim.x * gridDim.y * gridDim.z;
        const long long cta = ((long long)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
        for (long long i = cta * kCombineThreads + tid; i < p.num_blocks; i += ncta * kCombineThreads) p.refs[i] = 0u;
    }
    if (first < 0 || nparts < 1 || first + nparts > p.max_items) {
        if (tid == 0) index_fault(p.err, 20, first);
        return;
    }
    // this thread's first four partial outputs, loaded now: they do not depend
    // on M, so their round trip overlaps the (m, l) staging below
    const int pair = tid % PAIRS, grp = tid / PAIRS;
    const int h = pair / C4, c4 = pair % C4;
    const int d0 = col0 + c4 * 4;
    float4 v0[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int k = grp + u * PG;
        v0[u] = k < nparts ? __ldcg(reinterpret_cast<const float4*>(
                                 p.part_o + ((long long)(first + k) * p.Hq + qh0 + h) * D + d0))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int npl = nparts * GH;
    const bool staged = npl <= kMaxStaged;
    if (staged)
        for (int i = tid; i < npl; i += kCombineThreads)
            s_ml[i] = __ldcg(&p.part_ml[(long long)(first + i / GH) * p.Hq + qh0 + i % GH]);
    __syncthreads();
    auto ml_of = [&](int k, int h) -> float2 {
        return staged ? s_ml[k * GH + h] : __ldcg(&p.part_ml[(long long)(first + k) * p.Hq + qh0 + h]);
    };
    // M and L of each q head: one warp per head
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < GH) {
        float M = -INFINITY;
        for (int k = lane; k < nparts; k += 32) M = fmaxf(M, ml_of(k, warp).x);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float L = 0.f;
        for (int k = lane; k < nparts; k += 32) {
            const float2 ml = ml_of(k, warp);
            L += (ml.x == -INFINITY) ? 0.f : ml.y * exp2f(ml.x - M);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        if (lane == 0) {
            s_M[warp] = M;
            s_L[warp] = L;
        }
    }
    __syncthreads();
    const float M = s_M[h];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // four independent partial loads in flight per thread
    for (int k0 = grp; k0 < nparts; k0 += 4 * PG) {
        float4 v[4];
        float e[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = k0 + u * PG;
            e[u] = 0.f;
            v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < nparts) {
                const float2 ml = ml_of(k, h);
                e[u] = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
                v[u] = k0 == grp ? v0[u]
                                 : __ldcg(reinterpret_cast<const float4*>(
                                       p.part_o + ((long long)(first + k) * p.Hq + qh0 + h) * D + d0));
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            acc.x += v[u].x * e[u];
            acc.y += v[u].y * e[u];
            acc.z += v[u].z * e[u];
            acc.w += v[u].w * e[u];
        }
    }
    s_part[tid] = acc;
    __syncthreads();
    if (grp == 0) {
        for (int gI = 1; gI < PG; ++gI) {
            const float4 o = s_part[gI * PAIRS + pair];
            acc.x += o.x;
            acc.y += o.y;
            acc.z += o.z;
            acc.w += o.w;
        }
        const float L = s_L[h];
        const float inv = L > 0.f ? 1.f / L : 0.f;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + ((long long)b * p.Hq + qh0 + h) * D + d0;
        *reinterpret_cast<uint2*>(dst) =
            make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    }
}

// One warp writes token t of kv head kvh of sequence 0 (k_new / v_new) to
// K-half row `row` of the layer: K rotated at t when BAKED, V as it is; an
// INT8 cache stores codes and row scales.
template <int D, bool Q8>
__device__ __noinline__ void append_token_warp(const DecodeParams& p, long long row, int kvh, int t, int lane) {
    const __nv_bfloat16* kn = static_cast<const __nv_bfloat16*>(p.k_new) + (long long)kvh * D;
    const __nv_bfloat16* vn = static_cast<const __nv_bfloat16*>(p.v_new) + (long long)kvh * D;
    if constexpr (Q8) {
        int8_t* kg = const_cast<int8_t*>(static_cast<const int8_t*>(p.cache)) + p.layer_off + row * D;
        float* ksg = p.scales + p.sc_layer_off + row;
        int8_t kq[D / 32], vq[D / 32];
        float sk, sv;
        q8_store_token_warp<D / 64>(kn, vn, kg, kg + p.kv_off, ksg, ksg + p.sc_kv_off, p.rope, t, p.theta, lane, kq,
                                    vq, &sk, &sv);
    } else {
        constexpr int HALF = D / 2;
        __nv_bfloat16* kg = const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(p.cache)) + p.layer_off +
                            row * D;
        __nv_bfloat16* vg = kg + p.kv_off;
        for (int i = lane; i < HALF; i += 32) {
            __nv_bfloat16 k1 = kn[i], k2 = kn[i + HALF];
            if (p.rope == kRopeBaked) {
                float cs, sn;
                rope_cos_sin((long long)t, p.theta[i], &cs, &sn);
                const float x1 = __bfloat162float(k1), x2 = __bfloat162float(k2);
                k1 = __float2bfloat16_rn(x1 * cs - x2 * sn);
                k2 = __float2bfloat16_rn(x1 * sn + x2 * cs);
            }
            kg[i] = k1;
            kg[i + HALF] = k2;
            vg[i] = vn[i];
            vg[i + HALF] = vn[i + HALF];
        }
    }
}

template <int D, int GH, bool PAGED, bool READ, bool Q8>
// Two CTAs (ten warps) per SM: three warps share a sub-partition's 16K
// registers, so a thread may hold at most 168.
__global__ void __launch_bounds__(kDecodeThreads, decode_ctas_per_sm(Q8, PAGED, READ, D))
    decode_mma_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ KvTensorMaps maps) {
    using S = MmaShape<D, READ, Q8, PAGED>;
    using SM = MmaSmem<D, GH, READ, Q8, PAGED>;
    static_assert(!(READ && Q8 && PAGED), "paged caches take no read-time RoPE");
    static_assert(!Q8 || D >= 128, "INT8 rows are whole 128-byte column blocks");
    constexpr int NST = S::kStages, NSUB = S::kNsub, HALF = S::kHalf;

    extern __shared__ unsigned char smem_raw[];
    // the 128-byte swizzle pattern repeats every 1024 bytes: align the stages to it
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* stage_base = smem + SM::kStage;
    float* sc_base = reinterpret_cast<float*>(smem + SM::kSc);   // INT8: [stage][kScStageBytes / 4]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kBars);
    uint64_t* empty = full + NST;
    MmaStageMeta* meta = reinterpret_cast<MmaStageMeta*>(smem + SM::kMeta);
    float2* rot = reinterpret_cast<float2*>(smem + SM::kRot);
    float2* qcs = reinterpret_cast<float2*>(smem + SM::kQcs);
    float* merge_o = reinterpret_cast<float*>(smem + SM::kMergeO);
    float2* merge_ml = reinterpret_cast<float2*>(smem + SM::kMergeML);
    uint64_t* cbar = reinterpret_cast<uint64_t*>(smem + SM::kCbar);
    MmaSegment* first_hdr = reinterpret_cast<MmaSegment*>(smem + SM::kHdr);
    unsigned char* krot = smem + SM::kKrot;           // INT8 + READ_INCACHE: rotated K sub-tiles

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int kvh = blockIdx.y, z = blockIdx.z;
    const int group = kvh * gridDim.z + z;     // this (kv head, q-head group)'s share counter

    // shared-memory barriers and the tensor maps depend on the launch only:
    // set up before waiting for the previous kernel in the stream
    __shared__ uint64_t s_plan_bar;      // one paged sequence: the staged table landed
    if (tid == 0) {
        mbar_init(&s_plan_bar, 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(&cbar[0], kConsumerWarps * 32);
        mbar_init(&cbar[1], 64);
        mbar_init(&cbar[2], 64);
        mbar_init(&cbar[3], 1);
        mbar_fence_init();
#pragma unroll
        for (int r = 0; r < kRunMaps; ++r) tma_prefetch_desc(&maps.run[r]);
        if constexpr (Q8) {
            tma_prefetch_desc(&maps.sc_run);
            tma_prefetch_desc(&maps.sc_sub);
        }
    }
    if constexpr (!PAGED && !Q8) {
        // While the previous kernel in the stream finishes, the copy warp guesses
        // its first share from the positions as they stand and prefetches its
        // first kSpecRows K and V rows into L2.  A guess may be stale (the
        // previous kernel may still write positions or rows): it only steers
        // prefetch hints, clamped inside the layer, and nothing read from it is
        // used after the wait.
        if (warp == kConsumerWarps) {
            const int C = p.capacity;
            long long total = 0;
            for (int base = 0; base < p.B; base += 32) {
                const int bb = base + lane;
                long long st = 0;
                if (bb < p.B) {
                    const int tb = *(volatile const int*)(p.pos + bb);
                    const int nl = tb < 0 ? 0 : (tb + 1 < C ? tb + 1 : C);
                    st = (nl > 0 ? (nl + 15) / 16 : 1) + kSeqUnits;
                }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) st += __shfl_xor_sync(0xffffffffu, st, off);
                total += st;
            }
            const int G = (int)(total < p.nsplit ? total : p.nsplit);
            if ((int)blockIdx.x < G && total > 0) {
                const long long lo = div_nonneg((long long)blockIdx.x * total, G);
                long long run = 0;
                for (int base = 0; base < p.B; base += 32) {
                    const int bb = base + lane;
                    int nl = 0;
                    long long st = 0;
                    if (bb < p.B) {
                        const int tb = *(volatile const int*)(p.pos + bb);
                        nl = tb < 0 ? 0 : (tb + 1 < C ? tb + 1 : C);
                        st = (nl > 0 ? (nl + 15) / 16 : 1) + kSeqUnits;
                    }
                    long long incl = st;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const long long u = __shfl_up_sync(0xffffffffu, incl, off);
                        if (lane >= off) incl += u;
                    }
                    const long long Ob = run + incl - st;
                    const unsigned hit = __ballot_sync(0xffffffffu, bb < p.B && Ob <= lo && lo < Ob + st);
                    if (hit) {
                        if (lane == __ffs(hit) - 1) {
                            const int r0 = (int)max(0LL, lo - Ob - kSeqUnits) * 16;
                            const int n = min(nl - r0, kSpecRows);
                            if (n > 0) {
                                const int elt = Q8 ? 1 : 2;
                                const long long row = ((long long)bb * p.Hkv + kvh) * C + r0;
                                const char* k0 = static_cast<const char*>(p.cache) +
                                                 (p.layer_off + row * D) * elt;
                                bulk_prefetch_l2(k0, (uint32_t)(n * D * elt));
                                bulk_prefetch_l2(k0 + p.kv_off * elt, (uint32_t)(n * D * elt));
                            }
                        }
                        break;
                    }
                    run += __shfl_sync(0xffffffffu, incl, 31);
                }
            }
        }
    }
    if constexpr (PAGED && !Q8) {
        // A paged batch: the same guess from the plan's per-sequence rows and
        // block directory as they stand (the plan kernel may be rewriting them,
        // for this call or the last), and the block table; every index is
        // clamped, and only prefetch hints depend on it.
        if (warp == kConsumerWarps && !p.self_plan && p.seq_rows) {
            long long Rt = 0;
            for (int base = 0; base < p.B; base += 32)
                Rt += base + lane < p.B ? (long long)max(0, *(volatile const int*)(p.seq_rows + base + lane)) : 0;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) Rt += __shfl_xor_sync(0xffffffffu, Rt, off);
            const int G = paged_share_count(Rt, p.nsplit);
            if ((int)blockIdx.x < G && Rt > 0) {
                const long long lo = div_nonneg((long long)blockIdx.x * Rt, G);
                long long run = 0;
                for (int base = 0; base < p.B; base += 32) {
                    const int bb = base + lane;
                    const long long r =
                        bb < p.B ? (long long)max(0, *(volatile const int*)(p.seq_rows + bb)) : 0;
                    long long incl = r;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const long long u = __shfl_up_sync(0xffffffffu, incl, off);
                        if (lane >= off) incl += u;
                    }
                    const long long Ob = run + incl - r;
                    const unsigned hit = __ballot_sync(0xffffffffu, r > 0 && Ob <= lo && lo < Ob + r);
                    if (hit) {
                        const int src = __ffs(hit) - 1;
                        const int b = base + src;
                        const long long s0 = __shfl_sync(0xffffffffu, lo - Ob, src);
                        // the block of rank s0 / bs, by the directory's group counts
                        const int kb = (int)(s0 / p.bs);
                        const int2* drow = p.dir + (long long)b * p.dir_groups;
                        const int ng = min(p.dir_groups, 32);
                        int2 e = make_int2(0, 0x7fffffff);
                        if (lane < ng) {
                            e.x = *(volatile const int*)(&drow[lane].x);
                            e.y = *(volatile const int*)(&drow[lane].y);
                        }
                        const unsigned le = __ballot_sync(0xffffffffu, lane < ng && e.y <= kb);
                        if (le) {
                            const int gs = 31 - __clz(le);
                            uint32_t mm = (uint32_t)__shfl_sync(0xffffffffu, e.x, gs);
                            const int k = kb - __shfl_sync(0xffffffffu, e.y, gs);
                            if (k >= 0 && k < __popc(mm)) {
#pragma unroll 1
                                for (int q = 0; q < k; ++q) mm &= mm - 1u;
                                const int lb0 = gs * 32 + (__ffs(mm) - 1);
                                // the next blocks of the sequence from lb0, one per lane
                                const int lbl = lb0 + lane;
                                if (lane < kSpecRows / p.bs && lbl < p.maxb) {
                                    const int phys = *(volatile const int*)(p.table + (long long)b * p.maxb + lbl);
                                    if (phys >= 0 && phys < p.num_blocks) {
                                        const long long row = ((long long)phys * p.Hkv + kvh) * p.bs;
                                        const char* k0 = static_cast<const char*>(p.cache) + (p.layer_off + row * D) * 2;
                                        bulk_prefetch_l2(k0, (uint32_t)(p.bs * D * 2));
                                        bulk_prefetch_l2(k0 + p.kv_off * 2, (uint32_t)(p.bs * D * 2));
                                    }
                                }
                            }
                        }
                        break;
                    }
                    run += __shfl_sync(0xffffffffu, incl, 31);
                }
            }
        }
    }
    // one paged sequence: this CTA's share, planned here (no plan kernel)
    __shared__ SelfPlan s_plan;
    __shared__ int s_red[kDecodeThreads / 32];
    int32_t* const s_tab = reinterpret_cast<int32_t*>(stage_base);
    uint32_t* const s_val = reinterpret_cast<uint32_t*>(stage_base + kSelfPlanMax * 4);
    if constexpr (PAGED) {
        static_assert((size_t)NST * S::kStageBytes >= (size_t)(kSelfPlanMax + kSelfPlanValidWords) * 4,
                      "the stages hold the staged table and valid words");
        if (p.self_plan) {
            // While the previous kernel finishes: the plan once on the table as
            // it stands (its code and the table come into the SM's caches),
            // and the first blocks of the share it gives prefetched into L2.
            // Nothing of it is used after the wait, where the plan is made again.
            __syncthreads();                     // the barriers above are set up
            const SelfPlanArgs a{p.table, p.valid, p.pos, p.err, const_cast<int2*>(p.seq_items),
                                 p.maxb, p.num_blocks, p.bs, p.nsplit};
            self_plan_single(a, &s_plan, s_red, s_tab, s_val, &s_plan_bar, 0, true);
            if constexpr (!Q8) {
                const int nblk = max(1, kSpecRows / p.bs);
                if (warp == kConsumerWarps && lane < nblk && (int)blockIdx.x < s_plan.G && s_plan.rows > 0) {
                    const int lbk = s_plan.lb + lane;
                    const int phys = lane == 0 ? s_plan.phys : (lbk < p.maxb ? s_tab[lbk] : -1);
                    if (phys >= 0 && phys < p.num_blocks) {
                        const int r0 = lane == 0 ? s_plan.row : 0;
                        const long long row = ((long long)phys * p.Hkv + kvh) * p.bs + r0;
                        const char* k0 = static_cast<const char*>(p.cache) + (p.layer_off + row * D) * 2;
                        bulk_prefetch_l2(k0, (uint32_t)((p.bs - r0) * D * 2));
                        bulk_prefetch_l2(k0 + p.kv_off * 2, (uint32_t)((p.bs - r0) * D * 2));
                    }
                }
            }
            fence_proxy_async_smem();            // the staged table is read before it is copied again
            __syncthreads();
        }
    }
    // inputs written by earlier kernels (append, plan) are read only after this
    pdl_wait();
    pdl_launch_dependents();    // the combine kernel may start launching
    __syncthreads();
    if constexpr (PAGED) {
        if (p.self_plan) {
            const SelfPlanArgs a{p.table, p.valid, p.pos, p.err, const_cast<int2*>(p.seq_items),
                                 p.maxb, p.num_blocks, p.bs, p.nsplit};
            self_plan_single(a, &s_plan, s_red, s_tab, s_val, &s_plan_bar, 1, false);
        }
    }


    if (warp == kConsumerWarps) {
        // =================== copy-issuing warp ==============================
        // K/V rows read once per call stream through L2 as evict-first; in a
        // paged batch, the blocks that one sequence alone attends (refs)
        const bool evict_first = !(PAGED && p.B > 1);
        const uint64_t pol = l2_policy_evict_first();
        int it = 0, fill = 0, run_off = 0, claims = 0;
        bool ok = true, open = false, hdr_sent = false;
        // the first segment's header goes to the compute warps at once, so that
        // they load q while its first copy is in flight (b = -1: no segment)
        auto publish_first = [&](const MmaSegment& hdr) {
            if (hdr_sent) return;
            hdr_sent = true;
            if (lane == 0) {
                *first_hdr = hdr;
                mbar_arrive(&cbar[3]);
            }
        };
        auto open_stage = [&]() -> bool {
            const int s = it % NST;
            if (it >= NST && !mbar_wait(&empty[s], ((it / NST) - 1) & 1)) {
                if (lane == 0) set_error(p.err, 0x8u /* KVC_DEV_TIMEOUT */);
                return false;
            }
            open = true;
            fill = 0;
            run_off = 0;
            if (lane == 0) meta[s].flags = 0;
            return true;
        };
        auto commit = [&](int extra_flags) {
            const int s = it % NST;
            __syncwarp();
            if (lane == 0) {
                meta[s].nsub = fill;
                meta[s].flags |= extra_flags;
                mbar_arrive(&full[s]);
            }
            open = false;
            ++it;
        };
        // a segment starts on a fresh stage that carries its header; its q rows
        // are prefetched into L2 for the compute warps
        auto begin_segment = [&](const MmaSegment& hdr) -> bool {
            if (open) commit(0);
            if (!open_stage()) return false;
            publish_first(hdr);
            if (lane == 0) {
                meta[it % NST].flags = kSegBegin;
                meta[it % NST].seg = hdr;
                const __nv_bfloat16* qrow =
                    static_cast<const __nv_bfloat16*>(p.q) + ((long long)hdr.b * p.Hq + kvh * p.G + z * GH) * D;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(qrow), "r"((uint32_t)(GH * D * 2))
                             : "memory");
            }
            return true;
        };
        // the next share of this (kv head, q-head group) out of G: first share
        // blockIdx.x, then gridDim.x, gridDim.x + 1, ... claimed through the counter
        auto claim = [&](int G) -> int {
            if (claims++ == 0 && (int)blockIdx.x < G) return blockIdx.x;
            int v = 0;
            if (lane == 0) v = (int)atomicAdd(&p.counters[group], 1u);
            return (int)gridDim.x + __shfl_sync(0xffffffffu, v, 0);
        };
        // A full stage is published only when the next run needs room, so the
        // last stage of a segment is still open here and carries kSegEnd.
        auto end_segment = [&]() { commit(kSegEnd); };
        // free sub-tiles in the open stage (opening a stage when none is open or
        // the open one is full); 0 when the pipeline gave up
        auto ensure_room = [&]() -> int {
            if (open && fill == NSUB) commit(0);
            if (!open && !open_stage()) return 0;
            return NSUB - fill;
        };
        // READ_INCACHE: R(ip theta_i) of the last sub-tile emitted, for
        // i = lane + 32 m, and the step R(16 theta_i) to the next one
        constexpr int kFpl = (HALF + 31) / 32;        // frequencies per lane
        float2 ang[kFpl], adv[kFpl];
        if constexpr (READ) {
#pragma unroll
            for (int m = 0; m < kFpl; ++m) {
                const int i = lane + 32 * m;
                ang[m] = make_float2(1.f, 0.f);
                if (i < HALF) rope_cos_sin(16, p.theta[i], &adv[m].x, &adv[m].y);
            }
        }
        // One run: n consecutive rows (1 <= n <= 16 * room) of this layer's K
        // half from row urow, copied with their V rows by one tensor copy (one
        // per column block without tma_whole) of 16 ceil(n / 16) rows, as that
        // many sub-tiles.  ip0: in-cache position of the first row (READ_INCACHE);
        // exact: its angles computed afresh rather than advanced by 16 from the
        // previous sub-tile's; newrow: run row of the token being appended or -1.
        auto emit_run = [&](long long urow, int n, int ip0, int newrow, bool exact, bool ef) {
            const int s = it % NST;
            const int nsr = (n + 15) >> 4;
            const int R = nsr * 16;
            if constexpr (READ) {
                for (int j = 0; j < nsr; ++j) {
#pragma unroll
                    for (int m = 0; m < kFpl; ++m) {
                        const int i = lane + 32 * m;
                        if (i < HALF) {
                            if (exact && j == 0) {
                                rope_cos_sin((long long)ip0, p.theta[i], &ang[m].x, &ang[m].y);
                            } else {
                                const float2 a = ang[m], d = adv[m];
                                ang[m] = make_float2(a.x * d.x - a.y * d.y, a.y * d.x + a.x * d.y);
                            }
                            const int cp = i >> 3, jj = (i & 7) >> 1, e = i & 1;
                            rot[(s * NSUB + fill + j) * HALF + (jj * S::kCpr + cp) * 2 + e] = ang[m];
                        }
                    }
                }
            }
            if (lane < nsr) {
                const int f = fill + lane;
                const int lo = 16 * lane;
                meta[s].nrows[f] = min(16, n - lo);
                meta[s].ip0[f] = ip0 + lo;
                meta[s].newrow[f] = (newrow >= lo && newrow < lo + 16) ? newrow - lo : -1;
                meta[s].base[f] = run_off + lo * 128;
                meta[s].ld[f] = R;
                if constexpr (Q8) {
                    // the run's scales land in the slot of its first sub-tile, from
                    // row urow rounded down to a multiple of 4
                    meta[s].sbase[f] = fill * S::kScSlotFloats + (int)(urow & 3) + lo;
                    meta[s].sld[f] = kScRunRows;
                }
            }
            if (lane == 0) {
                unsigned char* dst = stage_base + (size_t)s * S::kStageBytes + run_off;
                const CUtensorMap* map = &maps.run[nsr - 1];
                if constexpr (Q8) {
                    mbar_expect_tx(&full[s], (uint32_t)(2 * kScRunRows * 4));
                    tma_load_3d(sc_base + (size_t)s * (S::kScStageBytes / 4) + fill * S::kScSlotFloats, &maps.sc_run,
                                (int)(urow & ~3LL), 0, p.layer, &full[s]);
                }
                mbar_expect_tx(&full[s], (uint32_t)(S::kBoxes * 2 * R * 128));
                if (p.tma_whole) {
                    if (ef)
                        tma_load_5d_hint(dst, map, 0, (int)urow, 0, p.layer, 0, &full[s], pol);
                    else
                        tma_load_5d(dst, map, 0, (int)urow, 0, p.layer, 0, &full[s]);
                } else {
#pragma unroll
                    for (int bx = 0; bx < S::kBoxes; ++bx) {
                        if (ef)
                            tma_load_4d_hint(dst + bx * 2 * R * 128, map, bx * S::kBoxCols, (int)urow, 0, p.layer,
                                             &full[s], pol);
                        else
                            tma_load_4d(dst + bx * 2 * R * 128, map, bx * S::kBoxCols, (int)urow, 0, p.layer,
                                        &full[s]);
                    }
                }
            }
            fill += nsr;
            run_off += S::kBoxes * 2 * R * 128;
        };
        // One sub-tile per calling lane, emitted by the lanes together: n rows
        // (1..16) from K-half row urow, sub-tile `rank` after the stage's
        // current fill (lanes of one call take distinct ranks below the room).
        constexpr int kSubCopy = S::kBoxes * 2 * 16 * 128;
        auto emit_sub_lane = [&](long long urow, int n, int rank, int newrow, bool ef) {
            const int s = it % NST;
            const int f = fill + rank;
            meta[s].nrows[f] = n;
            meta[s].ip0[f] = 0;
            meta[s].newrow[f] = newrow;
            meta[s].base[f] = run_off + rank * kSubCopy;
            meta[s].ld[f] = 16;
            if constexpr (Q8) {
                meta[s].sbase[f] = f * S::kScSlotFloats + (int)(urow & 3);
                meta[s].sld[f] = kScSubRows;
                mbar_expect_tx(&full[s], (uint32_t)(2 * kScSubRows * 4));
                tma_load_3d(sc_base + (size_t)s * (S::kScStageBytes / 4) + f * S::kScSlotFloats, &maps.sc_sub,
                            (int)(urow & ~3LL), 0, p.layer, &full[s]);
            }
            unsigned char* dst = stage_base + (size_t)s * S::kStageBytes + run_off + rank * kSubCopy;
            mbar_expect_tx(&full[s], (uint32_t)kSubCopy);
            if (p.tma_whole) {
                if (ef)
                    tma_load_5d_hint(dst, &maps.run[0], 0, (int)urow, 0, p.layer, 0, &full[s], pol);
                else
                    tma_load_5d(dst, &maps.run[0], 0, (int)urow, 0, p.layer, 0, &full[s]);
            } else {
#pragma unroll
                for (int bx = 0; bx < S::kBoxes; ++bx) {
                    if (ef)
                        tma_load_4d_hint(dst + bx * 2 * 16 * 128, &maps.run[0], bx * S::kBoxCols, (int)urow, 0,
                                         p.layer, &full[s], pol);
                    else
                        tma_load_4d(dst + bx * 2 * 16 * 128, &maps.run[0], bx * S::kBoxCols, (int)urow, 0, p.layer,
                                    &full[s]);
                }
            }
        };

        if constexpr (!PAGED) {
            // stream-K over the sequences: sequence b contributes
            // max(1, ceil(n_live(b) / 16)) sub-tiles (an empty one when t < 0)
            const int C = p.capacity;
            auto seq_tiles = [&](int bb, int* t_out, int* nl_out) -> long long {
                if (bb >= p.B) return 0;
                const int tb = p.pos[bb];
                const int nl = tb < 0 ? 0 : (tb + 1 < C ? tb + 1 : C);
                *t_out = tb;
                *nl_out = nl;
                return (nl > 0 ? (nl + 15) / 16 : 1) + kSeqUnits;
            };
            long long total = 0;
            // up to 32 sequences: each lane keeps its own sequence's figures from
            // this first pass (one read of the positions)
            int c_tb = 0, c_nl = 0;
            long long c_st = 0;
            for (int base = 0; base < p.B; base += 32) {
                int tb = 0, nl = 0;
                long long st = seq_tiles(base + lane, &tb, &nl);
                if (base == 0) {
                    c_tb = tb;
                    c_nl = nl;
                    c_st = st;
                }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) st += __shfl_xor_sync(0xffffffffu, st, off);
                total += st;
            }
            // no more shares than units, so that every share is non-empty and a
            // sequence's partial count is exactly the shares it overlaps
            const int G = (int)(total < p.nsplit ? total : p.nsplit);
            for (int xs = claim(G); xs < G && ok; xs = claim(G)) {
            const long long lo = div_nonneg((long long)xs * total, G);
            const long long hi = div_nonneg((long long)(xs + 1) * total, G);
            long long run = 0;
            for (int base = 0; base < p.B && ok && run < hi; base += 32) {
                int tb = c_tb, nl = c_nl;
                const long long st = p.B <= 32 ? c_st : seq_tiles(base + lane, &tb, &nl);
                long long incl = st;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const long long u = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += u;
                }
                for (int j = 0; j < 32 && ok; ++j) {
                    const int b = base + j;
                    if (b >= p.B) break;
                    const long long Sb = __shfl_sync(0xffffffffu, st, j);
                    const long long Ob = run + __shfl_sync(0xffffffffu, incl, j) - Sb;
                    const int t_b = __shfl_sync(0xffffffffu, tb, j);
                    const int nl_b = __shfl_sync(0xffffffffu, nl, j);
                    if (Ob >= hi) break;
                    if (Ob + Sb <= lo) continue;
                    const int fx = streamk_share_of(Ob, total, G);
                    const int lx = streamk_share_of(Ob + Sb - 1, total, G);
                    MmaSegment hdr;
                    hdr.b = b;
                    hdr.t = t_b;
                    hdr.slot = xs + b;
                    hdr.first_slot = fx + b;
                    hdr.nparts = lx - fx + 1;
                    hdr.new_row = -1;   // the window path marks the new token's run instead
                    if (!(ok = begin_segment(hdr))) break;
                    // units of the sequence: kSeqUnits charged for its segment
                    // start, then one per 16 rows
                    const int u0 = (int)((lo > Ob ? lo : Ob) - Ob), u1 = (int)((hi < Ob + Sb ? hi : Ob + Sb) - Ob);
                    const int r0 = max(0, u0 - kSeqUnits) * 16;
                    const int r1 = min(max(0, u1 - kSeqUnits) * 16, nl_b);
                    const long long base_row = ((long long)b * p.Hkv + kvh) * C;   // row in the K half
                    // slot of the token being decoded: the ring's wrap point, and
                    // (fused append) the row that receives the new K/V
                    int h_slot = 0;
                    if (t_b >= 0)
                        h_slot = t_b < p.sinks ? t_b : p.sinks + (int)((unsigned)(t_b - p.sinks) % (unsigned)p.window);
                    // READ_INCACHE: in-cache positions run on by one per slot between
                    // the sink/window boundary and the ring's wrap; they (and their
                    // angles) are computed afresh at those points and every 32 runs
                    int ip_next = 0, prev_n = 0, since = 0;
                    for (int r = r0; r < r1 && ok;) {
                        const int room = ensure_room();
                        if (!room) {
                            ok = false;
                            break;
                        }
                        int n = min(16 * room, r1 - r);
                        int ip0 = 0;
                        bool exact = true;
                        if constexpr (READ) {
                            // a run never straddles the sink/window boundary or the ring's wrap
                            const int seg_end = r < p.sinks ? p.sinks : (r <= h_slot ? h_slot + 1 : C);
                            n = min(n, seg_end - r);
                            exact = r == r0 || r == p.sinks || r == h_slot + 1 || (prev_n & 15) != 0 || since >= 32;
                            if (exact) {
                                ip0 = incache_of_slot(r, t_b, p.sinks, p.window, C);
                                since = 0;
                            } else {
                                ip0 = ip_next;
                            }
                            ++since;
                            ip_next = ip0 + n;
                            prev_n = n;
                        }
                        const int newrow = (p.k_new && t_b >= 0 && h_slot >= r && h_slot < r + n) ? h_slot - r : -1;
                        emit_run(base_row + r, n, ip0, newrow, exact, evict_first);
                        r += n;
                    }
                    if (ok) end_segment();
                }
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
            }
        } else {
            const bool self = p.self_plan != 0;
            // batch: the shares are cut here from each sequence's attended rows
            // (seq_rows, plan_rows_kernel) laid end to end, as the plan defines
            // them; rows of the first 64 sequences stay in registers
            long long Rt = 0;
            int rows0 = 0, rows1 = 0;
            if (!self) {
                rows0 = lane < p.B ? __ldcg(p.seq_rows + lane) : 0;
                rows1 = 32 + lane < p.B ? __ldcg(p.seq_rows + 32 + lane) : 0;
                long long r = (long long)rows0 + rows1;
                for (int base = 64; base < p.B; base += 32) r += base + lane < p.B ? __ldcg(p.seq_rows + base + lane) : 0;
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
                Rt = r;
            }
            const int G = self ? s_plan.G : paged_share_count(Rt, p.nsplit);
            // self-planned step: the new token's K-half row, when this CTA's
            // share holds it (it is the sequence's last attended row)
            int new_lb = -1, new_r = 0, new_row = -1;
            if (self && p.k_new && s_plan.traw >= 0 && s_plan.tphys >= 0 && s_plan.tphys < p.num_blocks) {
                new_lb = s_plan.traw / p.bs;
                new_r = s_plan.traw % p.bs;
                new_row = (s_plan.tphys * p.Hkv + kvh) * p.bs + new_r;
                if (!s_plan.tattended) {
                    // mapped but not resident: written here, never read by this step
                    if ((int)blockIdx.x == 0 && z == 0) append_token_warp<D, Q8>(p, new_row, kvh, s_plan.traw, lane);
                    new_lb = -1;
                }
            } else if (self && p.k_new && s_plan.traw >= 0 && (int)blockIdx.x == 0 && kvh == 0 && z == 0 &&
                       lane == 0) {
                set_error(p.err, (s_plan.traw / p.bs >= p.maxb) ? 0x4u : (s_plan.tphys < 0 ? 0x2u : 0x1u));
            }
            auto newrow_of = [&](int lbk, int row0, int n) -> int {
                return (lbk == new_lb && new_r >= row0 && new_r < row0 + n) ? new_r - row0 : -1;
            };
            // One segment: sequence itv.x from logical block itv.y, row itv.z, for
            // itv.w attended rows; inf = (t, first partial slot and slot count of
            // the sequence, physical block of itv.y or -2 when not known), `item`
            // its partial slot.
            auto walk_item = [&](const int4 itv, const int4 inf, int item) {
                const int b = itv.x;
                MmaSegment hdr;
                hdr.b = b;
                hdr.t = inf.x;
                hdr.slot = item;
                hdr.first_slot = inf.y;
                hdr.nparts = inf.z;
                hdr.new_row = new_row;
                if (!(ok = begin_segment(hdr))) return;
                const int tt = clamp_paged_t(hdr.t, p.maxb, p.bs);
                const int32_t* trow = p.table + (long long)b * p.maxb;
                int lb = itv.y;
                int rem = itv.w;
                const int last_lb = tt < 0 ? -1 : tt / p.bs;
                // self-planned sequence: the item's first block is attended by
                // construction and its physical block comes with the item, so its
                // copies need no table lookup
                if (inf.w != -2 && rem > 0 && lb <= last_lb && ok) {
                    const int phys = inf.w;
                    if (phys < 0 || phys >= p.num_blocks) {
                        if (lane == 0) index_fault(p.err, 13, phys);
                        ok = false;
                        return;
                    }
                    const int brows = lb == last_lb ? tt - lb * p.bs + 1 : p.bs;
                    const long long blk = ((long long)phys * p.Hkv + kvh) * p.bs;   // row in the K half
                    int row = itv.z;
                    int take = min(brows - row, rem);
                    while (take > 0 && ok) {
                        const int room = ensure_room();
                        if (!room) {
                            ok = false;
                            break;
                        }
                        const int n = min(take, 16 * room);
                        emit_run(blk + row, n, 0, newrow_of(lb, row, n), true, evict_first);
                        take -= n;
                        rem -= n;
                        row += n;
                    }
                    ++lb;
                }
                // blocks of at most 16 rows: one sub-tile each; the lanes take
                // 32 blocks at once and emit them together
                while (p.bs <= 16 && rem > 0 && lb <= last_lb && ok) {
                    const int my_lb = lb + lane;
                    int my_phys = -1, my_rows = 0;
                    uint32_t my_refs = 1u;
                    if (my_lb <= last_lb)
                        my_rows = paged_block_rows_refs(trow, p.valid, p.refs, p.err, my_lb, tt, p.bs, p.num_blocks,
                                                        &my_phys, &my_refs);
                    const bool my_ef = p.refs ? my_refs <= 1u : evict_first;
                    const int row0 = (my_lb == itv.y) ? itv.z : 0;
                    const int avail = my_rows > row0 ? my_rows - row0 : 0;
                    int incl = avail;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const int u = __shfl_up_sync(0xffffffffu, incl, off);
                        if (lane >= off) incl += u;
                    }
                    const int take = max(0, min(avail, rem - (incl - avail)));
                    rem -= min(rem, __shfl_sync(0xffffffffu, incl, 31));
                    const long long urow = ((long long)my_phys * p.Hkv + kvh) * p.bs + row0;
                    unsigned pending = __ballot_sync(0xffffffffu, take > 0);
                    while (pending && ok) {
                        const int room = ensure_room();
                        if (!room) {
                            ok = false;
                            break;
                        }
                        const int rank = __popc(pending & ((1u << lane) - 1u));
                        const bool mine = ((pending >> lane) & 1u) && rank < room;
                        const unsigned emitted = __ballot_sync(0xffffffffu, mine);
                        if (mine) emit_sub_lane(urow, take, rank, newrow_of(my_lb, row0, take), my_ef);
                        __syncwarp();
                        fill += __popc(emitted);
                        run_off += __popc(emitted) * kSubCopy;
                        pending &= ~emitted;
                    }
                    lb += 32;
                }
                while (rem > 0 && lb <= last_lb && ok) {
                    const int my_lb = lb + lane;
                    int my_phys = -1, my_rows = 0;
                    uint32_t my_refs = 1u;
                    if (my_lb <= last_lb)
                        my_rows = paged_block_rows_refs(trow, p.valid, p.refs, p.err, my_lb, tt, p.bs, p.num_blocks,
                                                        &my_phys, &my_refs);
                    const bool my_ef = p.refs ? my_refs <= 1u : evict_first;
                    unsigned mask = __ballot_sync(0xffffffffu, my_rows > 0);
                    while (mask && rem > 0 && ok) {
                        const int src = __ffs(mask) - 1;
                        mask &= mask - 1;
                        const int phys = __shfl_sync(0xffffffffu, my_phys, src);
                        const int brows = __shfl_sync(0xffffffffu, my_rows, src);
                        const bool bef = __shfl_sync(0xffffffffu, (int)my_ef, src) != 0;
                        int row = (lb + src == itv.y) ? itv.z : 0;
                        int take = min(brows - row, rem);
                        const long long blk = ((long long)phys * p.Hkv + kvh) * p.bs;   // row in the K half
                        while (take > 0 && ok) {
                            const int room = ensure_room();
                            if (!room) {
                                ok = false;
                                break;
                            }
                            const int n = min(take, 16 * room);
                            emit_run(blk + row, n, 0, newrow_of(lb + src, row, n), true, bef);
                            take -= n;
                            rem -= n;
                            row += n;
                        }
                    }
                    lb += 32;
                }
                if (ok) end_segment();
            };
            // The first attended block of row s0 of sequence b (position tb):
            // the block of rank s0 / bs, by the directory: the last 32-block
            // group with fewer attended blocks before it than that rank holds it.
            auto first_block = [&](int b, int tb, long long s0, int* lb_out, int* row_out) -> bool {
                const int kb = (int)(s0 / p.bs);
                const int tt = clamp_paged_t(tb, p.maxb, p.bs);
                const int ng = tt < 0 ? 0 : (tt / p.bs) / 32 + 1;
                const int2* drow = p.dir + (long long)b * p.dir_groups;
                int gsel = -1;
                int2 esel = make_int2(0, 0);
                for (int g0 = 0; g0 < ng; g0 += 32) {
                    const int g = g0 + lane;
                    const int2 e = g < ng ? __ldcg(drow + g) : make_int2(0, 0);
                    const unsigned le = __ballot_sync(0xffffffffu, g < ng && e.y <= kb);
                    if (le) {
                        const int src = 31 - __clz(le);
                        gsel = g0 + src;
                        esel.x = __shfl_sync(0xffffffffu, e.x, src);
                        esel.y = __shfl_sync(0xffffffffu, e.y, src);
                    }
                    if (le != 0xffffffffu) break;
                }
                uint32_t mm = (uint32_t)esel.x;
                const int k = kb - esel.y;
                if (gsel < 0 || k < 0 || k >= __popc(mm)) {
                    if (lane == 0) index_fault(p.err, 14, kb);
                    return false;
                }
#pragma unroll 1
                for (int q = 0; q < k; ++q) mm &= mm - 1u;
                *lb_out = gsel * 32 + (__ffs(mm) - 1);
                *row_out = (int)(s0 - (long long)kb * p.bs);
                return true;
            };
            for (int xs = claim(G); xs < G && ok; xs = self ? G : claim(G)) {
                if (self) {
                    // one sequence: share x holds exactly its item x
                    walk_item(make_int4(0, s_plan.lb, s_plan.row, s_plan.rows), make_int4(s_plan.traw, 0, G, s_plan.phys),
                              xs);
                    continue;
                }
                // the sequences that meet share xs, in order (b meets shares
                // paged_seq_shares(...).x .. .y; its segment is slot xs + b): one
                // lane per sequence tests its own, a ballot gathers them
                const long long lo = div_nonneg((long long)xs * Rt, G), hi = div_nonneg((long long)(xs + 1) * Rt, G);
                long long run = 0;
                for (int base = 0; base < p.B && ok; base += 32) {
                    // past share xs: only the empty sequences after the last row
                    // belong to the last share
                    if (run >= hi && hi < Rt) break;
                    const int bb = base + lane;
                    const int r = base == 0 ? rows0 : base == 32 ? rows1
                                : (bb < p.B ? __ldcg(p.seq_rows + bb) : 0);
                    long long incl = r;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const long long u = __shfl_up_sync(0xffffffffu, incl, off);
                        if (lane >= off) incl += u;
                    }
                    const long long Ob = run + incl - r;
                    bool meet;
                    if (r > 0) {
                        meet = Ob < hi && Ob + r > lo;
                    } else {
                        const long long u = Ob < Rt ? Ob : Rt - 1;     // its empty segment's row
                        meet = Rt > 0 ? (u >= lo && u < hi) : xs == 0;
                    }
                    unsigned mset = __ballot_sync(0xffffffffu, bb < p.B && meet);
                    while (mset && ok) {
                        const int j = __ffs(mset) - 1;
                        mset &= mset - 1u;
                        const int b = base + j;
                        const long long Rb = __shfl_sync(0xffffffffu, r, j);
                        const long long Obj = __shfl_sync(0xffffffffu, Ob, j);
                        const int2 fl = paged_seq_shares(Obj, Rb, Rt, G);
                        const int tb = p.pos[b];
                        int lb = 0, row = 0, rows = 0;
                        if (Rb > 0) {
                            const long long s0 = (lo > Obj ? lo : Obj) - Obj;
                            const long long s1 = (hi < Obj + Rb ? hi : Obj + Rb) - Obj;
                            rows = (int)(s1 - s0);
                            if (!first_block(b, tb, s0, &lb, &row)) rows = 0;
                        }
                        walk_item(make_int4(b, lb, row, rows), make_int4(tb, fl.x + b, fl.y - fl.x + 1, -2), xs + b);
                    }
                    run += __shfl_sync(0xffffffffu, incl, 31);
                }
            }
        }
        if (ok) {
            if (open) commit(0);
            if ((ok = open_stage())) {
                __syncwarp();
                if (lane == 0) {
                    meta[it % NST].nsub = -1;
                    mbar_arrive(&full[it % NST]);
                }
            }
        }
        if (!hdr_sent) {
            MmaSegment none;
            none.b = -1;
            none.t = none.slot = none.first_slot = none.nparts = 0;
            none.new_row = -1;
            publish_first(none);
        }
        if (!ok && lane == 0) {
            // never leave with copies still landing in this CTA's shared memory;
            // a stage left open has issued copies: arrive so its phase can end
            if (open) {
                mbar_arrive(&full[it % NST]);
                ++it;
            }
            for (int k = (it > NST ? it - NST : 0); k < it; ++k) mbar_wait(&full[k % NST], (k / NST) & 1);
        }
        return;
    }

    // ====================== compute warps (0 .. 3) ==========================
    const int ctid = tid;
    const int tg = warp / S::kDsplit;     // token group: which sub-tile of each stage
    const int hd = warp % S::kDsplit;     // which half of the output columns (D = 256)
    const int g = lane >> 2, c = lane & 3;
    constexpr int NCT = kConsumerWarps * 32;
    // INT8 column order of Q K^T: k-step ks of lane c takes columns
    // q8_col0(ks) .. + 3 (k-slots 2c, 2c + 1, 2c + 8, 2c + 9) -- any order of the
    // summed columns will do, as long as q and K use the same one
    auto q8_col0 = [&](int ks) {
        const int k2 = ks >> 1;
        return 128 * (k2 >> 2) + 16 * ((k2 & 3) + ((c >> 1) << 2)) + 8 * (c & 1) + 4 * (ks & 1);
    };
    BoundedBarrier csync{&cbar[0], 0u};           // the four compute warps
    BoundedBarrier psync{&cbar[1 + (tg & 1)], 0u}; // the two warps sharing a sub-tile (head_dim 256)

    // READ_INCACHE: this lane rotates chunk pair rcp (pairs i = 8 rcp + j) of
    // rows rrow0 + kRowStep k of its sub-tile; R(rrow0 theta_i) and the step
    // R(kRowStep theta_i) stay in registers (small angles: rrow0, kRowStep < 16)
    constexpr int kRowStep = S::kDsplit * S::kRowGroups;
    const int rcp = lane % S::kCpr;
    const int rrow0 = hd + S::kDsplit * (lane / S::kCpr);
    // packed over the pair couples (8 rcp + 2 q, 8 rcp + 2 q + 1): cos and sin
    float2 r0c[4], r0s[4], stc[4], sts[4];
    if constexpr (READ) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float th = p.theta_f[rcp * 8 + 2 * q + e];
                float c0, s0, c1, s1;
                sincosf((float)rrow0 * th, &s0, &c0);
                sincosf((float)kRowStep * th, &s1, &c1);
                (e ? r0c[q].y : r0c[q].x) = c0;
                (e ? r0s[q].y : r0s[q].x) = s0;
                (e ? stc[q].y : stc[q].x) = c1;
                (e ? sts[q].y : sts[q].x) = s1;
            }
        }
    }

    MmaSegment seg;
    seg.b = seg.t = seg.slot = seg.first_slot = seg.nparts = 0;
    uint32_t qa[S::kKsteps][2];
    // output accumulators: bf16, O = P V in 8-column tiles; INT8, O^T = V^T P^T
    // in 16-column tiles (rows: lane g's columns 16 g + mt and 16 g + 8 + mt,
    // columns: q heads 2c, 2c + 1), half as many
    constexpr int kOt = Q8 ? S::kNt / 2 : S::kNt;
    float o[kOt][4];
    float m_run = -INFINITY, l_run = 0.f;
    // INT8: fp16 tensor-core inputs.  q enters as q * q_scale * 2^-k (per head,
    // k >= 0 keeping it below 2^14: qexp = 2^k returns in the scores); a row's
    // weight enters as p * s_v / S_run, S_run the largest V scale of the segment
    // so far (the accumulator is rescaled when it grows and multiplied back at
    // the end), so weights stay in [0, 1]
    float qexp = 1.f, S_run = 0.f, rS = 0.f;   // rS = 1 / S_run

    // q of sequence seg.b as mma A fragments: row g = q head (zero for g >= GH),
    // per k-step columns 16 ks + 2c (+1) and 16 ks + 8 + 2c (+1); rotated,
    // scaled by softmax_scale * log2(e), rounded to bf16
    auto load_q = [&]() {
        int qpos = seg.t;
        if constexpr (PAGED) {
            qpos = clamp_paged_t(seg.t, p.maxb, p.bs);
            if ((seg.t < 0 || seg.t != qpos) && seg.slot == seg.first_slot && kvh == 0 && z == 0 && ctid == 0)
                set_error(p.err, 0x4u /* KVC_DEV_BAD_POSITION */);
        } else {
            if (seg.t < 0 && seg.slot == seg.first_slot && kvh == 0 && z == 0 && ctid == 0)
                set_error(p.err, 0x4u);
            if (READ) qpos = min(seg.t, p.capacity - 1);
        }
        const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) +
                                    ((long long)seg.b * p.Hq + kvh * p.G + z * GH + g) * D;
        csync.sync(p.err);                      // everyone is done with the previous qcs
        if (p.rope != kRopeNone) {
            for (int i = ctid; i < HALF; i += NCT) {
                float cs, sn;
                rope_cos_sin((long long)qpos, p.theta[i], &cs, &sn);
                qcs[i] = make_float2(cs, sn);
            }
        }
        csync.sync(p.err);
        float qf[S::kKsteps][4];
        if (Q8 && !READ && g < GH) {
            // INT8: k-step ks takes columns q8_col0(ks) .. + 3 (see the Q K^T
            // product); each value is rotated with its pair column
#pragma unroll
            for (int ks = 0; ks < S::kKsteps; ++ks) {
                const int d0 = q8_col0(ks);
                const uint2 w = *reinterpret_cast<const uint2*>(qrow + d0);
                float x[4] = {__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                              __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u)};
                if (p.rope != kRopeNone) {
                    const uint2 wp = *reinterpret_cast<const uint2*>(qrow + (d0 < HALF ? d0 + HALF : d0 - HALF));
                    const float y[4] = {__uint_as_float(wp.x << 16), __uint_as_float(wp.x & 0xffff0000u),
                                        __uint_as_float(wp.y << 16), __uint_as_float(wp.y & 0xffff0000u)};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 cs = qcs[(d0 + e) % HALF];
                        // column i < D/2: x cos - x' sin; column i + D/2: x' sin + x cos
                        x[e] = d0 < HALF ? x[e] * cs.x - y[e] * cs.y : y[e] * cs.y + x[e] * cs.x;
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) qf[ks][e] = x[e];
            }
        } else if (g < GH) {
#pragma unroll
            for (int ks = 0; ks < S::kKsteps; ++ks) {
                const uint32_t lo = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c);
                const uint32_t hi = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * c);
                qf[ks][0] = __uint_as_float(lo << 16);
                qf[ks][1] = __uint_as_float(lo & 0xffff0000u);
                qf[ks][2] = __uint_as_float(hi << 16);
                qf[ks][3] = __uint_as_float(hi & 0xffff0000u);
            }
            if (p.rope != kRopeNone) {
#pragma unroll
                for (int ks = 0; ks < S::kKsteps / 2; ++ks) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = 16 * ks + 2 * c + (e & 1) + 8 * (e >> 1);
                        const float2 cs = qcs[i];
                        const float x1 = qf[ks][e], x2 = qf[ks + S::kKsteps / 2][e];
                        qf[ks][e] = x1 * cs.x - x2 * cs.y;
                        qf[ks + S::kKsteps / 2][e] = x1 * cs.y + x2 * cs.x;
                    }
                }
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < S::kKsteps; ++ks) qf[ks][0] = qf[ks][1] = qf[ks][2] = qf[ks][3] = 0.f;
        }
        if constexpr (Q8 && !READ) {
            float amax = 0.f;
#pragma unroll
            for (int ks = 0; ks < S::kKsteps; ++ks)
#pragma unroll
                for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(qf[ks][e] * p.q_scale));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            int ex = 0;
            frexpf(amax, &ex);                        // amax < 2^ex
            const int k = ex > 14 ? ex - 14 : 0;
            qexp = ldexpf(1.f, k);
            const float qs = ldexpf(p.q_scale, -k);
#pragma unroll
            for (int ks = 0; ks < S::kKsteps; ++ks) {
                qa[ks][0] = pack_f16x2(qf[ks][0] * qs, qf[ks][1] * qs);
                qa[ks][1] = pack_f16x2(qf[ks][2] * qs, qf[ks][3] * qs);
            }
            S_run = 0.f;
            rS = 0.f;
        } else {
#pragma unroll
            for (int ks = 0; ks < S::kKsteps; ++ks) {
                qa[ks][0] = pack_bf16x2(qf[ks][0] * p.q_scale, qf[ks][1] * p.q_scale);
                qa[ks][1] = pack_bf16x2(qf[ks][2] * p.q_scale, qf[ks][3] * p.q_scale);
            }
            if constexpr (Q8) {
                // INT8 with read-time RoPE: bf16 q against the rotated bf16 K
                qexp = 1.f;
                S_run = 0.f;
                rS = 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < kOt; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        m_run = -INFINITY;
        l_run = 0.f;
    };

    // end of a segment: merge the warps and write the segment's partial
    // (m, l, o) per q head; the combine kernel merges a sequence's partials
    auto finish_segment = [&]() {
        if (seg.b < 0) {                          // rejected segment: keep the barrier sequence
            csync.sync(p.err);
            csync.sync(p.err);
            return;
        }
        float lq = l_run;
        lq += __shfl_xor_sync(0xffffffffu, lq, 1);
        lq += __shfl_xor_sync(0xffffffffu, lq, 2);
        csync.sync(p.err);                     // merge buffers free (previous segment done with them)
        if constexpr (Q8) {
            // INT8: this lane holds q heads 2c, 2c + 1 at columns hd * 128 + 16 g + mt (+ 8)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int hh = 2 * c + e;
                if (hh < GH) {
                    float* mo = merge_o + (tg * GH + hh) * D + hd * S::kDl + 16 * g;
#pragma unroll
                    for (int mt = 0; mt < kOt; ++mt) {
                        mo[mt] = o[mt][e] * S_run;
                        mo[8 + mt] = o[mt][2 + e] * S_run;
                    }
                }
            }
        }
        if (g < GH) {
            float* mo = merge_o + (tg * GH + g) * D;
            if constexpr (Q8) {
            } else {
#pragma unroll
                for (int j = 0; j < S::kNt; ++j) {
                    const int col = (hd * S::kNt + j) * 8 + 2 * c;
                    *reinterpret_cast<float2*>(mo + col) = make_float2(o[j][0], o[j][1]);
                }
            }
            if (c == 0 && hd == 0) merge_ml[tg * GH + g] = make_float2(m_run, lq);
        }
        csync.sync(p.err);
        const int qh0 = kvh * p.G + z * GH;
        for (int i4 = ctid; i4 < GH * D / 4; i4 += NCT) {
            const int h = (i4 * 4) / D, d = (i4 * 4) % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < S::kTokenGroups; ++w) M = fmaxf(M, merge_ml[w * GH + h].x);
            float L = 0.f;
            float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < S::kTokenGroups; ++w) {
                const float2 ml = merge_ml[w * GH + h];
                const float e = (ml.x == M) ? 1.f : exp2f(ml.x - M);
                const float4 v = *reinterpret_cast<const float4*>(merge_o + (w * GH + h) * D + d);
                L += ml.y * e;
                O.x += v.x * e;
                O.y += v.y * e;
                O.z += v.z * e;
                O.w += v.w * e;
            }
            const long long slot = (long long)seg.slot * p.Hq + qh0 + h;
            *reinterpret_cast<float4*>(p.part_o + slot * D + d) = O;
            if (d == 0) p.part_ml[slot] = make_float2(M, L);
        }
    };

    // a segment header that fails its checks writes nothing
    auto check_seg = [&](MmaSegment& sg) {
        if (sg.b < 0 || sg.b >= p.B || sg.slot < 0 || sg.slot >= p.max_items || sg.first_slot < 0 ||
            sg.nparts < 1 || sg.first_slot + sg.nparts > p.max_items || sg.slot < sg.first_slot ||
            sg.slot >= sg.first_slot + sg.nparts) {
            if (ctid == 0) index_fault(p.err, 3 + (sg.b < 0 || sg.b >= p.B ? 0 : 8), sg.slot);
            sg.b = -1;
        }
    };
    // q of the first segment, loaded while its first copy is in flight (not
    // with read-time RoPE, whose in-place rotation needs the registers)
    bool preloaded = false;
    if (READ) {
    } else if (mbar_wait(&cbar[3], 0)) {
        MmaSegment first = *first_hdr;
        if (first.b >= 0) {
            check_seg(first);
            if (first.b >= 0) {
                seg = first;
                load_q();
                preloaded = true;
            }
        }
    } else if (lane == 0) {
        set_error(p.err, 0x8u /* KVC_DEV_TIMEOUT */);
    }

    for (int it = 0;; ++it) {
        const int s = it % NST;
        if (!mbar_wait(&full[s], (it / NST) & 1)) {
            if (lane == 0) set_error(p.err, 0x8u);
            break;
        }
        const int nsub = meta[s].nsub;
        if (nsub < 0) break;
        if (nsub > NSUB) {                        // cannot happen: stop rather than read past the stage
            if (ctid == 0) index_fault(p.err, 12, nsub);
            break;
        }
        const int flags = meta[s].flags;
        if (flags & kSegBegin) {
            seg = meta[s].seg;
            check_seg(seg);
            if (preloaded) {                      // the first segment: q is already in registers
                preloaded = false;
            } else {
                if (seg.b >= 0) load_q(); else csync.sync(p.err), csync.sync(p.err);
            }
        }
        if (tg < nsub) {
            const int nrows = meta[s].nrows[tg];
            // the sub-tile's copy lands as [column block][K|V][ld rows][128 bytes]
            const int ld = meta[s].ld[tg];
            const int bstride = 2 * ld * 128;             // between column blocks
            unsigned char* Ks = stage_base + (size_t)s * S::kStageBytes + meta[s].base[tg];
            unsigned char* Vs = Ks + ld * 128;
            const uint32_t ku = smem_u32(Ks), vu = smem_u32(Vs);
            bool wrote = false;

            {
                // fused append (kvc_decode_step): this sub-tile holds the slot of the
                // token being decoded.  Write its K (RoPE baked at t when BAKED) and V
                // to the cache, and over the stale row just copied into shared memory.
                // Window layouts: the token's slot; a self-planned paged sequence:
                // the row the header names.
                const int nr = meta[s].newrow[tg];
                long long new_row = 0;
                if (nr >= 0) {
                    if constexpr (PAGED) {
                        new_row = seg.new_row;
                    } else {
                        const int h_slot = seg.t < p.sinks ? seg.t
                                                           : p.sinks + (int)((unsigned)(seg.t - p.sinks) % (unsigned)p.window);
                        new_row = ((long long)seg.b * p.Hkv + kvh) * p.capacity + h_slot;
                    }
                }
                if (Q8 && nr >= 0) {
                    if (hd == 0) {
                        // INT8: quantise the new rows; codes and scales go to the cache
                        // and over the stale copies in shared memory
                        const long long unit = (long long)seg.b * p.Hkv + kvh;
                        const long long row = new_row;
                        int8_t* kg = const_cast<int8_t*>(static_cast<const int8_t*>(p.cache)) + p.layer_off + row * D;
                        float* ksg = p.scales + p.sc_layer_off + row;
                        int8_t kq[D / 32], vq[D / 32];
                        float sk, sv;
                        q8_store_token_warp<D / 64>(static_cast<const __nv_bfloat16*>(p.k_new) + unit * D,
                                                    static_cast<const __nv_bfloat16*>(p.v_new) + unit * D, kg,
                                                    kg + p.kv_off, ksg, ksg + p.sc_kv_off, p.rope, seg.t, p.theta,
                                                    lane, kq, vq, &sk, &sv);
#pragma unroll
                        for (int m = 0; m < D / 64; ++m) {
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int col = lane + 32 * m + e * HALF;
                                const int off = (col >> 7) * bstride + nr * 128 +
                                                ((((col & 127) >> 4) ^ (nr & 7)) << 4) + (col & 15);
                                Ks[off] = (unsigned char)kq[2 * m + e];
                                Vs[off] = (unsigned char)vq[2 * m + e];
                            }
                        }
                        if (lane == 0) {
                            float* scl = sc_base + (size_t)s * (S::kScStageBytes / 4) + meta[s].sbase[tg];
                            scl[nr] = sk;
                            scl[meta[s].sld[tg] + nr] = sv;
                        }
                    }
                    wrote = true;
                    if constexpr (S::kDsplit == 2) psync.sync(p.err); else __syncwarp();
                } else if (nr >= 0) {
                    if (hd == 0) {
                        const long long unit = (long long)seg.b * p.Hkv + kvh;
                        const __nv_bfloat16* kn = static_cast<const __nv_bfloat16*>(p.k_new) + unit * D;
                        const __nv_bfloat16* vn = static_cast<const __nv_bfloat16*>(p.v_new) + unit * D;
                        __nv_bfloat16* kg = const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(p.cache)) +
                                            p.layer_off + new_row * D;
                        __nv_bfloat16* vg = kg + p.kv_off;
                        for (int i = lane; i < HALF; i += 32) {
                            __nv_bfloat16 k1 = kn[i], k2 = kn[i + HALF];
                            if (p.rope == kRopeBaked) {
                                float cs, sn;
                                rope_cos_sin((long long)seg.t, p.theta[i], &cs, &sn);
                                const float x1 = __bfloat162float(k1), x2 = __bfloat162float(k2);
                                k1 = __float2bfloat16_rn(x1 * cs - x2 * sn);
                                k2 = __float2bfloat16_rn(x1 * sn + x2 * cs);
                            }
                            const __nv_bfloat16 v1 = vn[i], v2 = vn[i + HALF];
                            kg[i] = k1;
                            kg[i + HALF] = k2;
                            vg[i] = v1;
                            vg[i + HALF] = v2;
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int col = i + e * HALF;
                                const int off = (col >> 6) * bstride + nr * 128 +
                                                (((((col & 63) >> 3)) ^ (nr & 7)) << 4) + (col & 7) * 2;
                                *reinterpret_cast<__nv_bfloat16*>(Ks + off) = e ? k2 : k1;
                                *reinterpret_cast<__nv_bfloat16*>(Vs + off) = e ? v2 : v1;
                            }
                        }
                    }
                    wrote = true;
                    if constexpr (S::kDsplit == 2) psync.sync(p.err); else __syncwarp();
                }
            }

            if constexpr (READ && Q8) {
                // INT8: K of the sub-tile as code x row scale, rotated by
                // R((ip0 + r) theta) as below, into the token group's bf16 tile;
                // rows past nrows too (their scores are masked out)
                const float4* rs4 = reinterpret_cast<const float4*>(rot + (s * NSUB + tg) * HALF);
                const float* kscl = sc_base + (size_t)s * (S::kScStageBytes / 4) + meta[s].sbase[tg];
                unsigned char* Kb = krot + (size_t)tg * S::kSub * D * 2;
                float2 cc[4], ss[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 a = rs4[q * S::kCpr + rcp];
                    const float2 ac = make_float2(a.x, a.z), as = make_float2(a.y, a.w);
                    cc[q] = __ffma2_rn(ac, r0c[q], __fmul2_rn(as, make_float2(-r0s[q].x, -r0s[q].y)));
                    ss[q] = __ffma2_rn(as, r0c[q], __fmul2_rn(ac, r0s[q]));
                }
                const int chi = rcp + S::kCpr;
                const int clo = 8 * rcp, chc = 8 * chi;       // first columns of the two chunks
#pragma unroll
                for (int k = 0; k < S::kRowsPerLane; ++k) {
                    const int r = rrow0 + k * kRowStep;
                    const uint2 wl = *reinterpret_cast<const uint2*>(
                        Ks + (clo >> 7) * bstride + r * 128 + ((((clo & 127) >> 4) ^ (r & 7)) << 4) + (clo & 8));
                    const uint2 wh = *reinterpret_cast<const uint2*>(
                        Ks + (chc >> 7) * bstride + r * 128 + ((((chc & 127) >> 4) ^ (r & 7)) << 4) + (chc & 8));
                    const float sc = kscl[r];
                    uint32_t ol[4], oh[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t lw = q < 2 ? wl.x : wl.y, hw = q < 2 ? wh.x : wh.y;
                        const int sh = 16 * (q & 1);
                        const float2 xl = make_float2((float)(int8_t)(lw >> sh) * sc, (float)(int8_t)(lw >> (sh + 8)) * sc);
                        const float2 xh = make_float2((float)(int8_t)(hw >> sh) * sc, (float)(int8_t)(hw >> (sh + 8)) * sc);
                        const float2 yl = __ffma2_rn(xl, cc[q], __fmul2_rn(xh, make_float2(-ss[q].x, -ss[q].y)));
                        const float2 yh = __ffma2_rn(xl, ss[q], __fmul2_rn(xh, cc[q]));
                        ol[q] = pack_bf16x2(yl.x, yl.y);
                        oh[q] = pack_bf16x2(yh.x, yh.y);
                    }
                    *reinterpret_cast<uint4*>(Kb + (rcp >> 3) * (S::kSub * 128) + r * 128 + (((rcp & 7) ^ (r & 7)) << 4)) =
                        make_uint4(ol[0], ol[1], ol[2], ol[3]);
                    *reinterpret_cast<uint4*>(Kb + (chi >> 3) * (S::kSub * 128) + r * 128 + (((chi & 7) ^ (r & 7)) << 4)) =
                        make_uint4(oh[0], oh[1], oh[2], oh[3]);
                    if (k + 1 < S::kRowsPerLane) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 c0 = cc[q];
                            cc[q] = __ffma2_rn(c0, stc[q], __fmul2_rn(ss[q], make_float2(-sts[q].x, -sts[q].y)));
                            ss[q] = __ffma2_rn(ss[q], stc[q], __fmul2_rn(c0, sts[q]));
                        }
                    }
                }
                if constexpr (S::kDsplit == 2) psync.sync(p.err); else __syncwarp();
            }
            if constexpr (READ && !Q8) {
                // rotate the stored (raw) K rows in place by R((ip0 + r) theta):
                // R(ip0 theta) from the stage table times R(r theta), advanced
                // from row to row by the step rotation.  Packed fp32 pairs; rows
                // past nrows are rotated too (their scores are masked out).
                const float4* rs4 = reinterpret_cast<const float4*>(rot + (s * NSUB + tg) * HALF);
                float2 cc[4], ss[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 a = rs4[q * S::kCpr + rcp];
                    const float2 ac = make_float2(a.x, a.z), as = make_float2(a.y, a.w);
                    cc[q] = __ffma2_rn(ac, r0c[q], __fmul2_rn(as, make_float2(-r0s[q].x, -r0s[q].y)));
                    ss[q] = __ffma2_rn(as, r0c[q], __fmul2_rn(ac, r0s[q]));
                }
                const int chi = rcp + S::kCpr;
                const int lo_off = (rcp >> 3) * bstride, hi_off = (chi >> 3) * bstride;
#pragma unroll
                for (int k = 0; k < S::kRowsPerLane; ++k) {
                    const int r = rrow0 + k * kRowStep;
                    uint4* plo = reinterpret_cast<uint4*>(Ks + lo_off + r * 128 + ((((rcp & 7) ^ (r & 7))) << 4));
                    uint4* phi = reinterpret_cast<uint4*>(Ks + hi_off + r * 128 + ((((chi & 7) ^ (r & 7))) << 4));
                    const uint4 wl = *plo, wh = *phi;
                    const uint32_t lw[4] = {wl.x, wl.y, wl.z, wl.w}, hw[4] = {wh.x, wh.y, wh.z, wh.w};
                    uint32_t ol[4], oh[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 xl = make_float2(__uint_as_float(lw[q] << 16), __uint_as_float(lw[q] & 0xffff0000u));
                        const float2 xh = make_float2(__uint_as_float(hw[q] << 16), __uint_as_float(hw[q] & 0xffff0000u));
                        const float2 yl = __ffma2_rn(xl, cc[q], __fmul2_rn(xh, make_float2(-ss[q].x, -ss[q].y)));
                        const float2 yh = __ffma2_rn(xl, ss[q], __fmul2_rn(xh, cc[q]));
                        ol[q] = pack_bf16x2(yl.x, yl.y);
                        oh[q] = pack_bf16x2(yh.x, yh.y);
                    }
                    *plo = make_uint4(ol[0], ol[1], ol[2], ol[3]);
                    *phi = make_uint4(oh[0], oh[1], oh[2], oh[3]);
                    if (k + 1 < S::kRowsPerLane) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 c0 = cc[q];
                            cc[q] = __ffma2_rn(c0, stc[q], __fmul2_rn(ss[q], make_float2(-sts[q].x, -sts[q].y)));
                            ss[q] = __ffma2_rn(ss[q], stc[q], __fmul2_rn(c0, sts[q]));
                        }
                    }
                }
                wrote = true;
                if constexpr (S::kDsplit == 2) psync.sync(p.err); else __syncwarp();
            }
            if (!Q8 && nrows < S::kSub) {
                // rows past nrows may hold anything (NaN): zero this warp's V columns there
                // (INT8 codes are always finite; their weights are zeroed instead)
                constexpr int BPW = S::kBoxes / S::kDsplit;
                const int per_box = (S::kSub - nrows) * 8;
                for (int idx = lane; idx < per_box * BPW; idx += 32) {
                    const int bxl = idx / per_box, rem = idx % per_box;
                    const int r = nrows + rem / 8, ch = rem % 8;
                    *reinterpret_cast<uint4*>(Vs + (hd * BPW + bxl) * bstride + r * 128 + ch * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                wrote = true;
                __syncwarp();
            }

            // ---- S = Q K^T over the 16 rows: two 8-token n-tiles --------------
            float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            uint4 vw[2][2];          // INT8: V code chunks of tokens 2c, 2c + 1, 2c + 8, 2c + 9
            if constexpr (Q8 && READ) {
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                    const int ta = 2 * c + 8 * hlf;
                    vw[hlf][0] = *reinterpret_cast<const uint4*>(Vs + hd * bstride + ta * 128 + ((g ^ (ta & 7)) << 4));
                    vw[hlf][1] = *reinterpret_cast<const uint4*>(Vs + hd * bstride + (ta + 1) * 128 +
                                                                 ((g ^ ((ta + 1) & 7)) << 4));
                }
            }
            if constexpr (Q8 && !READ) {
                // INT8: lane (g, c) reads 8 code bytes of rows g and g + 8 at columns
                // q8_col0(2 k2) .. + 7 and turns them into the B fragments of k-steps
                // 2 k2 and 2 k2 + 1 (the 16-byte chunks k2 mod 4 and k2 mod 4 + 4 of a
                // 128-column block: a half-warp's reads fall on 8 distinct chunks)
                uint2 kw[D / 32][2];
#pragma unroll
                for (int k2 = 0; k2 < D / 32; ++k2) {
                    const int ch = (k2 & 3) + ((c >> 1) << 2);
                    const int off = (k2 >> 2) * bstride + ((ch ^ (g & 7)) << 4) + ((c & 1) << 3);
                    kw[k2][0] = *reinterpret_cast<const uint2*>(Ks + off + g * 128);
                    kw[k2][1] = *reinterpret_cast<const uint2*>(Ks + off + (g + 8) * 128);
                }
                // the V chunks P V will need, loaded now so that their latency hides
                // behind Q K^T and the softmax
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                    const int ta = 2 * c + 8 * hlf;          // tokens ta, ta + 1 -> B register hlf
                    vw[hlf][0] = *reinterpret_cast<const uint4*>(Vs + hd * bstride + ta * 128 + ((g ^ (ta & 7)) << 4));
                    vw[hlf][1] = *reinterpret_cast<const uint4*>(Vs + hd * bstride + (ta + 1) * 128 +
                                                                 ((g ^ ((ta + 1) & 7)) << 4));
                }
#pragma unroll
                for (int k2 = 0; k2 < D / 32; ++k2) {
#pragma unroll
                    for (int s2 = 0; s2 < 2; ++s2) {
                        const uint32_t a = (s2 ? kw[k2][0].y : kw[k2][0].x) ^ 0x80808080u;
                        const uint32_t e = (s2 ? kw[k2][1].y : kw[k2][1].x) ^ 0x80808080u;
                        const int ks = 2 * k2 + s2;
                        mma_f16_16816(sa[0], qa[ks][0], 0u, qa[ks][1], 0u, q8_f16x2(a, 0x4140u), q8_f16x2(a, 0x4342u));
                        mma_f16_16816(sa[1], qa[ks][0], 0u, qa[ks][1], 0u, q8_f16x2(e, 0x4140u), q8_f16x2(e, 0x4342u));
                    }
                }
            } else {
                const int tok = ((lane >> 4) << 3) + (lane & 7);
                const int chs = (lane >> 3) & 1;
                // bf16 K: the stage's rows, or (INT8 + READ) the rotated tile
                const uint32_t kbase = Q8 ? smem_u32(krot + (size_t)tg * S::kSub * D * 2) : ku;
                const int kstride = Q8 ? S::kSub * 128 : bstride;
#pragma unroll
                for (int ks = 0; ks < S::kKsteps; ++ks) {
                    const int bx = ks >> 2;
                    const int ch = ((ks & 3) << 1) + chs;
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kbase + bx * kstride + tok * 128 + ((ch ^ (tok & 7)) << 4), b0, b1, b2, b3);
                    mma_bf16_16816(sa[0], qa[ks][0], 0u, qa[ks][1], 0u, b0, b1);
                    mma_bf16_16816(sa[1], qa[ks][0], 0u, qa[ks][1], 0u, b2, b3);
                }
            }

            // ---- online softmax on row g (this lane's q head) ----------------
            float sv[4] = {sa[0][0], sa[0][1], sa[1][0], sa[1][1]};
            const int tk0 = 2 * c;
            float vsc[4] = {1.f, 1.f, 1.f, 1.f};
            if constexpr (Q8) {
                // scores of a row times its K scale; its V scale goes into the
                // weight (zero past nrows, whose scales may be anything)
                const float* scl = sc_base + (size_t)s * (S::kScStageBytes / 4) + meta[s].sbase[tg];
                const float* vscl = scl + meta[s].sld[tg];
                const int tk[4] = {tk0, tk0 + 1, tk0 + 8, tk0 + 9};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if constexpr (!READ) sv[e] *= scl[tk[e]] * qexp;   // (READ: the K scale is in the tile)
                    vsc[e] = tk[e] < nrows ? vscl[tk[e]] : 0.f;
                }
            }
            if (tk0 >= nrows) sv[0] = -INFINITY;
            if (tk0 + 1 >= nrows) sv[1] = -INFINITY;
            if (tk0 + 8 >= nrows) sv[2] = -INFINITY;
            if (tk0 + 9 >= nrows) sv[3] = -INFINITY;
            float mx = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mn = fmaxf(m_run, mx);
            const float alpha = (mn == m_run || g >= GH) ? 1.f : exp2f(m_run - mn);
            float pe[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) pe[e] = (sv[e] == -INFINITY || g >= GH) ? 0.f : exp2f(sv[e] - mn);
            l_run = l_run * alpha + ((pe[0] + pe[1]) + (pe[2] + pe[3]));
            m_run = mn;
            float ofac = alpha;
            uint32_t pa0, pa2;
            if constexpr (Q8) {
                // a V scale above S_run anywhere: the 16 rows' largest (lanes of one c
                // share their rows) becomes S_run, the accumulator scaled down to it
                const float lmax = fmaxf(fmaxf(vsc[0], vsc[1]), fmaxf(vsc[2], vsc[3]));
                if (__any_sync(0xffffffffu, lmax > S_run)) {
                    float smax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, 1));
                    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 2));
                    ofac *= S_run / smax;
                    S_run = smax;
                    rS = __frcp_rn(S_run);
                }
                pa0 = pack_f16x2(pe[0] * vsc[0] * rS, pe[1] * vsc[1] * rS);
                pa2 = pack_f16x2(pe[2] * vsc[2] * rS, pe[3] * vsc[3] * rS);
            } else {
                pa0 = pack_bf16x2(pe[0], pe[1]);
                pa2 = pack_bf16x2(pe[2], pe[3]);
            }
            if (__any_sync(0xffffffffu, ofac != 1.f)) {
                if constexpr (Q8) {
                    // columns are q heads 2c and 2c + 1: their factors come from lanes 8c, 8c + 4
                    const float f0 = __shfl_sync(0xffffffffu, ofac, 8 * c);
                    const float f1 = __shfl_sync(0xffffffffu, ofac, 8 * c + 4);
#pragma unroll
                    for (int mt = 0; mt < kOt; ++mt) {
                        o[mt][0] *= f0;
                        o[mt][2] *= f0;
                        o[mt][1] *= f1;
                        o[mt][3] *= f1;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < S::kNt; ++j) {
                        o[j][0] *= ofac;
                        o[j][1] *= ofac;
                    }
                }
            }

            // ---- O += P V over this warp's output columns ---------------------
            if constexpr (Q8) {
                // INT8: O^T += V^T P^T.  Lane (g, c) holds 16 code bytes (columns
                // hd * 128 + 16 g .. + 15) of tokens 2c, 2c + 1, 2c + 8, 2c + 9 (loaded with
                // K, in vw); A rows g and g + 8 of m-tile mt are columns 16 g + mt and
                // 16 g + 8 + mt, k = tokens; B = P^T is the softmax fragment as it is.
                uint32_t x0[16], x1[16];        // byte j of tokens (2c, 2c + 1) and (2c + 8, 2c + 9)
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const uint32_t a0 = (q4 == 0 ? vw[0][0].x : q4 == 1 ? vw[0][0].y : q4 == 2 ? vw[0][0].z : vw[0][0].w) ^ 0x80808080u;
                    const uint32_t b0 = (q4 == 0 ? vw[0][1].x : q4 == 1 ? vw[0][1].y : q4 == 2 ? vw[0][1].z : vw[0][1].w) ^ 0x80808080u;
                    const uint32_t a1 = (q4 == 0 ? vw[1][0].x : q4 == 1 ? vw[1][0].y : q4 == 2 ? vw[1][0].z : vw[1][0].w) ^ 0x80808080u;
                    const uint32_t b1 = (q4 == 0 ? vw[1][1].x : q4 == 1 ? vw[1][1].y : q4 == 2 ? vw[1][1].z : vw[1][1].w) ^ 0x80808080u;
                    // [a0 b0 a1 b1] and [a2 b2 a3 b3] of the two token rows
                    const uint32_t lo0 = __byte_perm(a0, b0, 0x5140u), hi0 = __byte_perm(a0, b0, 0x7362u);
                    const uint32_t lo1 = __byte_perm(a1, b1, 0x5140u), hi1 = __byte_perm(a1, b1, 0x7362u);
#pragma unroll
                    for (int jb = 0; jb < 4; ++jb) {
                        const uint32_t sel = (jb & 1) ? 0x4342u : 0x4140u;
                        x0[4 * q4 + jb] = q8_f16x2(jb < 2 ? lo0 : hi0, sel);
                        x1[4 * q4 + jb] = q8_f16x2(jb < 2 ? lo1 : hi1, sel);
                    }
                }
#pragma unroll
                for (int mt = 0; mt < kOt; ++mt)
                    mma_f16_16816(o[mt], x0[mt], x0[8 + mt], x1[mt], x1[8 + mt], pa0, pa2);
            } else {
                const int tok = (((lane >> 3) & 1) << 3) + (lane & 7);
                const int chs = lane >> 4;
#pragma unroll
                for (int j = 0; j < S::kNt; j += 2) {
                    const int dt = hd * S::kNt + j;        // global 8-column tile
                    const int bx = dt >> 3;
                    const int ch = (dt & 7) + chs;
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_trans(vu + bx * bstride + tok * 128 + ((ch ^ (tok & 7)) << 4), v0, v1, v2, v3);
                    mma_bf16_16816(o[j], pa0, 0u, pa2, 0u, v0, v1);
                    mma_bf16_16816(o[j + 1], pa0, 0u, pa2, 0u, v2, v3);
                }
            }
            if (wrote) fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (flags & kSegEnd) finish_segment();
    }
}

template <int D, int GH, bool PAGED, bool READ, bool Q8>
cudaError_t launch_decode_mma_t(const DecodeParams& p, const KvTensorMaps& maps, dim3 grid, cudaStream_t stream) {
    using SM = MmaSmem<D, GH, READ, Q8, PAGED>;
    // the resident CTAs per SM that __launch_bounds__ plans for must fit in
    // shared memory (228 KB per SM, 1 KB of it reserved per CTA)
    constexpr int kCtasPerSm = decode_ctas_per_sm(Q8, PAGED, READ, D);
    static_assert(kCtasPerSm * (SM::kTotal + 1024) <= 233472, "shared memory for the planned CTAs per SM");
    auto kern = decode_mma_kernel<D, GH, PAGED, READ, Q8>;
    // few (sequence, kv head, group) units: narrow column chunks, more CTAs
    // each; many: 128 columns a CTA (measured: 64-column chunks 0.5 us slower
    // on the 64-sequence paged batch, 16-column ones 14 us)
    const long long units = (long long)p.B * p.Hkv * p.nsub;
    const bool narrow = units * (D / 16) <= 1216;
    constexpr int kWide = D >= 128 ? 128 : 64;
    auto comb = narrow ? combine_streamk_kernel<D, GH, PAGED, 16> : combine_streamk_kernel<D, GH, PAGED, kWide>;
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_relaxed) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM::kTotal);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_relaxed);
    }
    // both launches may begin while the previous kernel in the stream drains;
    // each waits (griddepcontrol.wait) before touching that kernel's outputs
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = SM::kTotal;
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p, maps);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t ccfg = {};
    ccfg.gridDim = dim3(p.B, p.Hkv * p.nsub, D / (narrow ? 16 : kWide));
    ccfg.blockDim = dim3(kCombineThreads);
    ccfg.dynamicSmemBytes = 0;
    ccfg.stream = stream;
    ccfg.attrs = &attr;
    ccfg.numAttrs = 1;
    return cudaLaunchKernelEx(&ccfg, comb, p);
}

}  // namespace kvc
