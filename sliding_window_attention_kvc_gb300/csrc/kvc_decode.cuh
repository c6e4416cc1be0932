// Split-K decode attention over a ring / sink+ring / paged KV cache.
//
// One CTA = one work item (a contiguous share of one sequence's attended
// rows) x one kv head x one group of up to 4 q heads.  Warp 4 issues 1-D bulk
// copies (cp.async.bulk, the TMA engine) of K and V rows into a 4-stage
// shared-memory ring guarded by mbarriers; warps 0-3 compute.  Each compute
// lane owns 2 x 16 bytes of a row (dims [c, c + CH) and [D/2 + c, D/2 + c + CH),
// i.e. whole RoPE pairs), so a row is read from shared memory exactly once,
// conflict-free, and q . k is finished with a shuffle butterfly over the
// lanes of the row.  Every lane group keeps its own fp32 online softmax
// (running max m in log2 units, running sum l, unnormalised output o); the
// groups are merged at the end and the CTA writes one partial (m, l, o) per q
// head.  The last CTA to finish a (sequence, kv head, q-head group) - found
// with an atomic ticket, no waiting - combines the partials:
//     M = max m_i,  out = sum o_i 2^(m_i - M) / sum l_i 2^(m_i - M).
//
// Attended sets ([ring] 2.2 and 6, [sink] cache-set equation, [pool] "kernel
// forgets absent blocks"): for RING / SINK_RING, the live slots are exactly
// 0 .. min(t, C-1) and every live slot is attended, so a work item is a slot
// range; for PAGED, rows of blocks that are unmapped or not valid are never
// copied and rows past t are cut from the last block.
#pragma once

#include <atomic>

#include "kvc_device.cuh"

namespace kvc {

template <typename Elt, int D>
struct DecodeShape {
    static constexpr int kElt = EltTraits<Elt>::kBytes;
    static constexpr int kCh = 16 / kElt;                  // elements per 16-byte chunk
    static constexpr int kDpl = 2 * kCh;                   // dims per lane
    static constexpr int kLpr = D / kDpl;                  // lanes per row
    static constexpr int kRgPerWarp = 32 / kLpr;           // row groups per warp
    static constexpr int kRowGroups = kConsumerWarps * kRgPerWarp;
    static constexpr int kRpg = 2;                         // rows per row group per stage
    static constexpr int kT = kRowGroups * kRpg;           // rows per stage
    static constexpr int kRowBytes = D * kElt;
    static constexpr int kStageBytes = 2 * kT * kRowBytes; // K rows then V rows
    static constexpr int kHalf = D / 2;
    static_assert(kLpr >= 2 && kLpr <= 32 && (32 % kLpr) == 0, "unsupported head_dim");
};

struct alignas(16) StageMeta {
    int nrows;   // rows in the stage; -1 = end of the stream
    int ipb;     // READ_INCACHE: in-cache position of row 0
    int pad[2];
};

template <typename Elt, int D, int GH, bool READ>
struct DecodeSmem {
    using S = DecodeShape<Elt, D>;
    static constexpr size_t kStages = 0;
    static constexpr size_t kBars = kStages + (size_t)kvc::kStages * S::kStageBytes;
    static constexpr size_t kMeta = kBars + 2 * kvc::kStages * sizeof(uint64_t);
    static constexpr size_t kRot = kMeta + kvc::kStages * sizeof(StageMeta);
    static constexpr size_t kTab = kRot + (READ ? (size_t)kvc::kStages * S::kHalf * sizeof(float2) : 0);
    static constexpr size_t kQcs = kTab + (READ ? (size_t)S::kT * S::kHalf * sizeof(float2) : 0);
    static constexpr size_t kMergeO = kQcs + (size_t)S::kHalf * sizeof(float2);
    static constexpr size_t kMergeML = kMergeO + (size_t)kConsumerWarps * GH * D * sizeof(float);
    static constexpr size_t kFlag = kMergeML + (size_t)kConsumerWarps * GH * sizeof(float2);
    static constexpr size_t kTotal = kFlag + 16;
};

// Attended rows of logical block lb of a paged sequence whose current
// position is t (already clamped to the table): 0 when the block is unmapped
// or not resident, the rows up to t for the last block, else block_size.
__device__ __forceinline__ int paged_block_rows(const int32_t* table_row, const uint32_t* valid, uint32_t* err,
                                                int lb, int t, int bs, int num_blocks, int* phys_out) {
    const int last = t / bs;
    if (t < 0 || lb > last) return 0;
    const int phys = table_row[lb];
    *phys_out = phys;
    if (phys < 0) return 0;
    if (phys >= num_blocks) {
        set_error(err, 0x1u /* KVC_DEV_BAD_BLOCK */);
        return 0;
    }
    if (valid && !((valid[phys >> 5] >> (phys & 31)) & 1u)) return 0;
    return lb == last ? (t - lb * bs + 1) : bs;
}

// The same, with the block's reader count of this step (refs, null: 1)
// loaded beside its valid word.
__device__ __forceinline__ int paged_block_rows_refs(const int32_t* table_row, const uint32_t* valid,
                                                     const uint32_t* refs, uint32_t* err, int lb, int t, int bs,
                                                     int num_blocks, int* phys_out, uint32_t* refs_out) {
    const int last = t / bs;
    *refs_out = 1u;
    if (t < 0 || lb > last) return 0;
    const int phys = table_row[lb];
    *phys_out = phys;
    if (phys < 0) return 0;
    if (phys >= num_blocks) {
        set_error(err, 0x1u /* KVC_DEV_BAD_BLOCK */);
        return 0;
    }
    const uint32_t w = valid ? valid[phys >> 5] : 0xffffffffu;
    *refs_out = refs ? __ldcg(refs + phys) : 1u;
    if (!((w >> (phys & 31)) & 1u)) return 0;
    return lb == last ? (t - lb * bs + 1) : bs;
}

// n / d for n >= 0, d > 0: a 32-bit division when both fit.
__device__ __forceinline__ long long div_nonneg(long long n, long long d) {
    if (n >= 0 && n < 0x100000000LL && d > 0 && d < 0x100000000LL) return (long long)((unsigned)n / (unsigned)d);
    return n / d;
}

// Share holding unit u of a stream-K partition of `total` units into
// `shares` contiguous ranges [floor(x total / shares), floor((x + 1) total / shares)).
__device__ __forceinline__ int streamk_share_of(long long u, long long total, int shares) {
    return (int)div_nonneg((u + 1) * shares - 1, total);
}

// Paged stream-K plan: G shares of the R attended rows of the batch laid end to
// end (no more shares than rows, at least one).  Sequence b, with O_b rows
// before it and R_b rows, meets shares first .. last; a sequence with no
// attended row gets the share that holds row O_b (row R - 1 past the end) for
// its empty segment.  Its segment with share x writes partial slot x + b.
__device__ __forceinline__ int paged_share_count(long long R, int shares) {
    return (int)(R < shares ? (R > 0 ? R : 1) : shares);
}
__device__ __forceinline__ int2 paged_seq_shares(long long Ob, long long Rb, long long R, int G) {
    if (Rb > 0) return make_int2(streamk_share_of(Ob, R, G), streamk_share_of(Ob + Rb - 1, R, G));
    const int x = R > 0 ? streamk_share_of(Ob < R ? Ob : R - 1, R, G) : 0;
    return make_int2(x, x);
}

__device__ __forceinline__ int clamp_paged_t(int t, int maxb, int bs) {
    const long long lim = (long long)maxb * bs - 1;
    return t > lim ? (int)lim : t;
}

// In-cache position of live slot s of a sink+ring cache at time t
// ([sink] "RoPE cache position shifting"): sinks keep their index; the window
// token in slot s is p = t - ((t - s) mod W), shifted left by max(0, t-C+1).
__device__ __forceinline__ int incache_of_slot(int s, int t, int S, int W, int C) {
    if (s < S) return s;
    const int p = t - (int)(((long long)t - s) % W);
    const int shift = t - C + 1;
    return shift > 0 ? p - shift : p;
}

template <typename Elt, int D, int GH, bool PAGED, bool READ>
__global__ void __launch_bounds__(kDecodeThreads, 2) decode_kernel(const __grid_constant__ DecodeParams p) {
    using S = DecodeShape<Elt, D>;
    using SM = DecodeSmem<Elt, D, GH, READ>;
    using TR = EltTraits<Elt>;
    constexpr int NST = kvc::kStages;
    constexpr int CH = S::kCh, DPL = S::kDpl, LPR = S::kLpr, T = S::kT, NRG = S::kRowGroups;
    constexpr int HALF = S::kHalf;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* stage_base = smem + SM::kStages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kBars);
    uint64_t* empty = full + NST;
    StageMeta* meta = reinterpret_cast<StageMeta*>(smem + SM::kMeta);
    float2* rot = reinterpret_cast<float2*>(smem + SM::kRot);
    float2* tab = reinterpret_cast<float2*>(smem + SM::kTab);
    float2* qcs = reinterpret_cast<float2*>(smem + SM::kQcs);
    float* merge_o = reinterpret_cast<float*>(smem + SM::kMergeO);
    float2* merge_ml = reinterpret_cast<float2*>(smem + SM::kMergeML);
    int* flag = reinterpret_cast<int*>(smem + SM::kFlag);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int item = blockIdx.x, kvh = blockIdx.y, z = blockIdx.z;

    // ---- which sequence, which rows --------------------------------------
    int b, first_item, nparts;
    int4 pitem = make_int4(0, 0, 0, 0);
    if constexpr (PAGED) {
        if (item >= *p.n_items) return;
        pitem = p.items[item];
        if (pitem.x < 0) return;          // index left unused by the plan
        b = pitem.x;
        const int2 si = p.seq_items[b];
        first_item = si.x;
        nparts = si.y;
    } else {
        b = item / p.nsplit;
        first_item = b * p.nsplit;
        nparts = p.nsplit;
    }
    int t = p.pos[b];

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_fence_init();
    }
    __syncthreads();

    const Elt* cache = static_cast<const Elt*>(p.cache);

    if (warp == kConsumerWarps) {
        // =================== copy-issuing warp ==============================
        int it = 0;
        bool ok = true;
        auto open_stage = [&](int s) -> bool {
            if (it >= NST) {
                if (!mbar_wait(&empty[s], ((it / NST) - 1) & 1)) {
                    if (lane == 0) set_error(p.err, 0x8u /* KVC_DEV_TIMEOUT */);
                    return false;
                }
            }
            return true;
        };
        if constexpr (!PAGED) {
            const int C = p.capacity;
            int n_live = t < 0 ? 0 : (t + 1 < C ? t + 1 : C);
            const int split = item - first_item;
            const int chunk = (n_live + p.nsplit - 1) / p.nsplit;
            const int r0 = min(n_live, split * chunk);
            const int r1 = min(n_live, r0 + chunk);
            const long long unit = ((long long)b * p.Hkv + kvh) * C;
            const Elt* kbase = cache + p.layer_off + unit * D;
            const Elt* vbase = kbase + p.kv_off;
            int h_slot = 0;
            if constexpr (READ) {
                if (t >= 0) h_slot = t < p.sinks ? t : p.sinks + (int)(((long long)t - p.sinks) % p.window);
            }
            for (int r = r0; r < r1 && ok;) {
                int n = min(T, r1 - r);
                int ipb = 0;
                if constexpr (READ) {
                    const int seg_end = r < p.sinks ? p.sinks : (r <= h_slot ? h_slot + 1 : C);
                    n = min(n, seg_end - r);
                    ipb = incache_of_slot(r, t, p.sinks, p.window, C);
                }
                const int s = it % NST;
                if (!(ok = open_stage(s))) break;
                if constexpr (READ) {
                    for (int i = lane; i < HALF; i += 32) {
                        float c, sn;
                        rope_cos_sin((long long)ipb, p.theta[i], &c, &sn);
                        rot[s * HALF + i] = make_float2(c, sn);
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    meta[s].nrows = n;
                    meta[s].ipb = ipb;
                    const uint32_t bytes = (uint32_t)n * S::kRowBytes;
                    unsigned char* dst = stage_base + (size_t)s * S::kStageBytes;
                    mbar_expect_tx(&full[s], 2 * bytes);
                    bulk_load(dst, kbase + (long long)r * D, bytes, &full[s]);
                    bulk_load(dst + T * S::kRowBytes, vbase + (long long)r * D, bytes, &full[s]);
                    mbar_arrive(&full[s]);
                }
                r += n;
                ++it;
            }
        } else {
            const int tt = clamp_paged_t(t, p.maxb, p.bs);
            const int32_t* trow = p.table + (long long)b * p.maxb;
            int lb = pitem.y;
            int row_first = pitem.z;
            int rem = pitem.w;
            int fill = 0;
            bool open = false;
            const int last_lb = tt < 0 ? -1 : tt / p.bs;
            while (rem > 0 && lb <= last_lb && ok) {
                const int my_lb = lb + lane;
                int my_phys = -1;
                int my_rows = 0;
                if (my_lb <= last_lb)
                    my_rows = paged_block_rows(trow, p.valid, p.err, my_lb, tt, p.bs, p.num_blocks, &my_phys);
                unsigned mask = __ballot_sync(0xffffffffu, my_rows > 0);
                while (mask && rem > 0 && ok) {
                    const int src = __ffs(mask) - 1;
                    mask &= mask - 1;
                    const int phys = __shfl_sync(0xffffffffu, my_phys, src);
                    const int brows = __shfl_sync(0xffffffffu, my_rows, src);
                    int row = (lb + src == pitem.y) ? row_first : 0;
                    int take = min(brows - row, rem);
                    const long long blk = ((long long)phys * p.Hkv + kvh) * p.bs;
                    const Elt* kb = cache + p.layer_off + blk * D;
                    const Elt* vb = kb + p.kv_off;
                    while (take > 0) {
                        const int s = it % NST;
                        if (!open) {
                            if (!(ok = open_stage(s))) break;
                            open = true;
                            fill = 0;
                        }
                        const int n = min(take, T - fill);
                        if (lane == 0) {
                            const uint32_t bytes = (uint32_t)n * S::kRowBytes;
                            unsigned char* dst = stage_base + (size_t)s * S::kStageBytes + (size_t)fill * S::kRowBytes;
                            mbar_expect_tx(&full[s], 2 * bytes);
                            bulk_load(dst, kb + (long long)row * D, bytes, &full[s]);
                            bulk_load(dst + T * S::kRowBytes, vb + (long long)row * D, bytes, &full[s]);
                        }
                        fill += n;
                        take -= n;
                        rem -= n;
                        row += n;
                        if (fill == T) {
                            if (lane == 0) {
                                meta[s].nrows = T;
                                mbar_arrive(&full[s]);
                            }
                            open = false;
                            ++it;
                        }
                    }
                }
                lb += 32;
            }
            if (open && ok) {
                const int s = it % NST;
                if (lane == 0) {
                    meta[s].nrows = fill;
                    mbar_arrive(&full[s]);
                }
                ++it;
            }
        }
        // end-of-stream marker
        if (ok) {
            const int s = it % NST;
            if ((ok = open_stage(s)) && lane == 0) {
                meta[s].nrows = -1;
                mbar_arrive(&full[s]);
            }
        }
        if (!ok && lane == 0) {
            // Do not leave the CTA with copies still landing in its shared
            // memory: wait (bounded) for every stage that may hold one.
            for (int k = (it > NST ? it - NST : 0); k < it; ++k) mbar_wait(&full[k % NST], (k / NST) & 1);
        }
        return;
    }

    // ====================== compute warps (0 .. 3) ==========================
    const int ctid = tid;                 // 0 .. 127
    const int rgw = lane / LPR;           // row group within the warp
    const int sl = lane % LPR;            // lane within the row
    const int rg = warp * S::kRgPerWarp + rgw;

    int qpos = 0;
    if (!PAGED) {
        if (t < 0) {
            if (item == first_item && kvh == 0 && z == 0 && ctid == 0) set_error(p.err, 0x4u);
        }
        qpos = t;
        if (READ) qpos = t < p.capacity - 1 ? t : p.capacity - 1;
    } else {
        if ((t < 0 || t > clamp_paged_t(t, p.maxb, p.bs)) && item == first_item && kvh == 0 && z == 0 && ctid == 0)
            set_error(p.err, 0x4u);
        qpos = clamp_paged_t(t, p.maxb, p.bs);
    }
    if (p.rope != kRopeNone) {
        for (int i = ctid; i < HALF; i += kConsumerWarps * 32) {
            float c, sn;
            rope_cos_sin((long long)qpos, p.theta[i], &c, &sn);
            qcs[i] = make_float2(c, sn);
        }
    }
    if constexpr (READ) {
        for (int idx = ctid; idx < T * HALF; idx += kConsumerWarps * 32) {
            const int r = idx / HALF, i = idx % HALF;
            float c, sn;
            sincosf((float)r * p.theta_f[i], &sn, &c);
            tab[idx] = make_float2(c, sn);
        }
    }
    named_sync(1, kConsumerWarps * 32);

    // q for the GH heads of this CTA: rotated, scaled by softmax_scale*log2(e)
    float q[GH][DPL];
    {
        const Elt* qb = static_cast<const Elt*>(p.q);
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            const int qh = kvh * p.G + z * GH + h;
            const Elt* row = qb + ((long long)b * p.Hq + qh) * D;
            const uint4 wa = *reinterpret_cast<const uint4*>(row + sl * CH);
            const uint4 wb = *reinterpret_cast<const uint4*>(row + HALF + sl * CH);
            float fa[CH], fb[CH];
            TR::unpack(wa, fa);
            TR::unpack(wb, fb);
            if (p.rope != kRopeNone) {
#pragma unroll
                for (int j = 0; j < CH; ++j) {
                    const float2 cs = qcs[sl * CH + j];
                    const float x1 = fa[j], x2 = fb[j];
                    fa[j] = x1 * cs.x - x2 * cs.y;
                    fb[j] = x1 * cs.y + x2 * cs.x;
                }
            }
#pragma unroll
            for (int j = 0; j < CH; ++j) {
                q[h][j] = fa[j] * p.q_scale;
                q[h][CH + j] = fb[j] * p.q_scale;
            }
        }
    }

    float m[GH], l[GH], o[GH][DPL];
#pragma unroll
    for (int h = 0; h < GH; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int j = 0; j < DPL; ++j) o[h][j] = 0.f;
    }

    for (int it = 0;; ++it) {
        const int s = it % NST;
        if (!mbar_wait(&full[s], (it / NST) & 1)) {
            if (lane == 0) set_error(p.err, 0x8u);
            break;
        }
        const int nrows = meta[s].nrows;
        if (nrows < 0) break;
        const unsigned char* Ks = stage_base + (size_t)s * S::kStageBytes;
        const unsigned char* Vs = Ks + T * S::kRowBytes;

        float sc[S::kRpg][GH];
#pragma unroll
        for (int k = 0; k < S::kRpg; ++k) {
            const int r = rg + k * NRG;
            const bool vr = r < nrows;
            float kf[DPL];
            if (vr) {
                const uint4 wa = *reinterpret_cast<const uint4*>(Ks + r * S::kRowBytes + sl * 16);
                const uint4 wb = *reinterpret_cast<const uint4*>(Ks + r * S::kRowBytes + (sl + LPR) * 16);
                TR::unpack(wa, kf);
                TR::unpack(wb, kf + CH);
            } else {
#pragma unroll
                for (int j = 0; j < DPL; ++j) kf[j] = 0.f;
            }
            if constexpr (READ) {
                if (vr) {
                    const float2* rs = rot + s * HALF + sl * CH;
                    const float2* tr = tab + r * HALF + sl * CH;
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        const float2 a = rs[j], bb = tr[j];
                        const float c = a.x * bb.x - a.y * bb.y;
                        const float sn = a.y * bb.x + a.x * bb.y;
                        const float x1 = kf[j], x2 = kf[CH + j];
                        kf[j] = x1 * c - x2 * sn;
                        kf[CH + j] = x1 * sn + x2 * c;
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                float d = 0.f;
#pragma unroll
                for (int j = 0; j < DPL; ++j) d = fmaf(q[h][j], kf[j], d);
#pragma unroll
                for (int off = LPR / 2; off >= 1; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
                sc[k][h] = vr ? d : -INFINITY;
            }
        }

        float pk[S::kRpg][GH];
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            float mn = m[h];
#pragma unroll
            for (int k = 0; k < S::kRpg; ++k) mn = fmaxf(mn, sc[k][h]);
            float lsum = 0.f;
#pragma unroll
            for (int k = 0; k < S::kRpg; ++k) {
                pk[k][h] = sc[k][h] == -INFINITY ? 0.f : exp2f(sc[k][h] - mn);
                lsum += pk[k][h];
            }
            if (mn != m[h]) {
                const float alpha = exp2f(m[h] - mn);   // m = -inf gives 0
                l[h] *= alpha;
#pragma unroll
                for (int j = 0; j < DPL; ++j) o[h][j] *= alpha;
                m[h] = mn;
            }
            l[h] += lsum;
        }

#pragma unroll
        for (int k = 0; k < S::kRpg; ++k) {
            const int r = rg + k * NRG;
            if (r < nrows) {
                float vf[DPL];
                const uint4 wa = *reinterpret_cast<const uint4*>(Vs + r * S::kRowBytes + sl * 16);
                const uint4 wb = *reinterpret_cast<const uint4*>(Vs + r * S::kRowBytes + (sl + LPR) * 16);
                TR::unpack(wa, vf);
                TR::unpack(wb, vf + CH);
#pragma unroll
                for (int h = 0; h < GH; ++h) {
#pragma unroll
                    for (int j = 0; j < DPL; ++j) o[h][j] = fmaf(pk[k][h], vf[j], o[h][j]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---- merge the row groups of this warp ---------------------------------
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            const float mo = __shfl_xor_sync(0xffffffffu, m[h], off);
            const float lo = __shfl_xor_sync(0xffffffffu, l[h], off);
            const float mn = fmaxf(m[h], mo);
            const float a = (m[h] == mn) ? 1.f : exp2f(m[h] - mn);
            const float c = (mo == mn) ? 1.f : exp2f(mo - mn);
            l[h] = l[h] * a + lo * c;
#pragma unroll
            for (int j = 0; j < DPL; ++j) {
                const float oo = __shfl_xor_sync(0xffffffffu, o[h][j], off);
                o[h][j] = o[h][j] * a + oo * c;
            }
            m[h] = mn;
        }
    }
    if (rgw == 0) {
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            float* mo = merge_o + (warp * GH + h) * D;
#pragma unroll
            for (int j = 0; j < CH; ++j) {
                mo[sl * CH + j] = o[h][j];
                mo[HALF + sl * CH + j] = o[h][CH + j];
            }
            if (sl == 0) merge_ml[warp * GH + h] = make_float2(m[h], l[h]);
        }
    }
    named_sync(1, kConsumerWarps * 32);

    // ---- merge the warps, write this CTA's partial ------------------------
    for (int idx = ctid; idx < GH * D; idx += kConsumerWarps * 32) {
        const int h = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, merge_ml[w * GH + h].x);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float2 ml = merge_ml[w * GH + h];
            const float e = (ml.x == M) ? 1.f : exp2f(ml.x - M);
            L += ml.y * e;
            O += merge_o[(w * GH + h) * D + d] * e;
        }
        const int qh = kvh * p.G + z * GH + h;
        const long long slot = (long long)item * p.Hq + qh;
        p.part_o[slot * D + d] = O;
        if (d == 0) p.part_ml[slot] = make_float2(M, L);
    }
    __threadfence();
    named_sync(1, kConsumerWarps * 32);
    const long long cidx = ((long long)b * p.Hkv + kvh) * p.nsub + z;
    if (ctid == 0) {
        const unsigned ticket = atomicAdd(&p.counters[cidx], 1u);
        *flag = (ticket == (unsigned)(nparts - 1));
    }
    named_sync(1, kConsumerWarps * 32);
    if (*flag) {
        // ---- last CTA of this (sequence, kv head, group): combine ---------
        __threadfence();
        Elt* out = static_cast<Elt*>(p.out);
        for (int idx = ctid; idx < GH * D; idx += kConsumerWarps * 32) {
            const int h = idx / D, d = idx % D;
            const int qh = kvh * p.G + z * GH + h;
            float M = -INFINITY;
            for (int k = 0; k < nparts; ++k)
                M = fmaxf(M, __ldcg(&p.part_ml[(long long)(first_item + k) * p.Hq + qh]).x);
            float L = 0.f, O = 0.f;
            for (int k = 0; k < nparts; ++k) {
                const long long slot = (long long)(first_item + k) * p.Hq + qh;
                const float2 ml = __ldcg(&p.part_ml[slot]);
                const float e = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
                L += ml.y * e;
                O += __ldcg(&p.part_o[slot * D + d]) * e;
            }
            out[((long long)b * p.Hq + qh) * D + d] = TR::from_f32(L > 0.f ? O / L : 0.f);
        }
        if (ctid == 0) p.counters[cidx] = 0u;
    }
}

template <typename Elt, int D, int GH, bool PAGED, bool READ>
cudaError_t launch_decode_t(const DecodeParams& p, dim3 grid, cudaStream_t stream) {
    using SM = DecodeSmem<Elt, D, GH, READ>;
    auto kern = decode_kernel<Elt, D, GH, PAGED, READ>;
    // The shared-memory opt-in is per device: remember which devices have it.
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
    kern<<<grid, kDecodeThreads, SM::kTotal, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kvc
