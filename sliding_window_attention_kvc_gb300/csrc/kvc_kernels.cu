// Append (with fused RoPE), paged work planning, and block-table / residency
// updates.
#include "kvc_decode.cuh"

namespace kvc {

// ---------------------------------------------------------------------------
// kvc_append: one CTA per (token, sequence); each thread rotates one RoPE
// pair (i, i + D/2) of one kv head.  Slot maps: [ring] 3.3 / 5.1 (p mod W),
// [sink] (S pinned sinks, then a ring), [share] 3.1 (block table).  RoPE is
// baked into K only ([pool] "RoPE baked into K rows": V is never rotated).
// ---------------------------------------------------------------------------
// Write one token's K (RoPE baked at `pos` when rope == kRopeBaked) and V
// rows for every kv head: K of head h at kc + h * head_stride, V kv_off
// elements further; k_src / v_src are the token's [Hkv, D] rows.  Threads
// first .. first + nthreads - 1 of the calling CTA (all by default) split the
// (head, pair) work.
template <typename Elt>
__device__ __forceinline__ void write_token_rows(Elt* kc, long long kv_off, long long head_stride, const Elt* ks,
                                                 const Elt* vs, int Hkv, int D, int rope, long long pos,
                                                 const unsigned long long* theta, int first = 0, int nthreads = 0) {
    using TR = EltTraits<Elt>;
    const int half = D / 2;
    Elt* vc = kc + kv_off;
    if (nthreads <= 0) nthreads = blockDim.x;
    for (int idx = (int)threadIdx.x - first; idx < Hkv * half; idx += nthreads) {
        const int h = idx / half, i = idx % half;
        const Elt* kr = ks + (long long)h * D;
        const Elt* vr = vs + (long long)h * D;
        Elt* kd = kc + h * head_stride;
        Elt* vd = vc + h * head_stride;
        const Elt k1 = kr[i], k2 = kr[i + half];
        if (rope == kRopeBaked) {
            float c, s;
            rope_cos_sin(pos, theta[i], &c, &s);
            const float x1 = TR::to_f32(k1), x2 = TR::to_f32(k2);
            kd[i] = TR::from_f32(x1 * c - x2 * s);
            kd[i + half] = TR::from_f32(x1 * s + x2 * c);
        } else {
            kd[i] = k1;
            kd[i + half] = k2;
        }
        vd[i] = vr[i];
        vd[i + half] = vr[i + half];
    }
}

// INT8 cache ([primer] 5.1, quantised cache): one warp per kv head stores
// the token's K (RoPE baked at `pos`) and V rows as codes and row scales.
// kc: K codes of kv head 0; ksc: its K scale; heads head_stride codes and
// sc_head_stride scales apart; V kv_off codes and sc_kv_off scales further.
template <int NP>
__device__ __forceinline__ void q8_write_token_rows(int8_t* kc, long long kv_off, long long head_stride, float* ksc,
                                                    long long sc_kv_off, long long sc_head_stride,
                                                    const __nv_bfloat16* ks, const __nv_bfloat16* vs, int Hkv,
                                                    int rope, long long pos, const unsigned long long* theta) {
    constexpr int D = 64 * NP;
    const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int h = threadIdx.x >> 5; h < Hkv; h += nw) {
        int8_t kq[2 * NP], vq[2 * NP];
        float sk, sv;
        int8_t* kd = kc + h * head_stride;
        float* sd = ksc + h * sc_head_stride;
        q8_store_token_warp<NP>(ks + (long long)h * D, vs + (long long)h * D, kd, kd + kv_off, sd, sd + sc_kv_off,
                                rope, pos, theta, lane, kq, vq, &sk, &sv);
    }
}

// Elt: the cache's element type; int8_t = INT8 cache, fed bf16 rows.
template <typename Elt>
__global__ void __launch_bounds__(256) append_kernel(const __grid_constant__ AppendParams p) {
    const int i_tok = blockIdx.x, b = blockIdx.y;
    const int t0 = p.pos[b];
    const long long pos = (long long)t0 + i_tok;
    if (pos < 0) return;                       // left padding
    const long long last = (long long)t0 + p.n_new - 1;
    const int D = p.D;

    long long row_base;                        // element offset of (row, kv head 0) in the K half
    long long head_stride;                     // elements between kv heads
    if (p.layout != kPaged) {
        // a window token overwritten by a later token of this call is skipped
        if (pos >= p.sinks && pos + p.window <= last) return;
        const long long slot = pos < p.sinks ? pos : p.sinks + (pos - p.sinks) % p.window;
        row_base = ((long long)b * p.Hkv * p.capacity + slot) * D;
        head_stride = (long long)p.capacity * D;
    } else {
        const long long lb = pos / p.bs;
        if (lb >= p.maxb) {
            if (threadIdx.x == 0) set_error(p.err, 0x4u /* KVC_DEV_BAD_POSITION */);
            return;
        }
        const int phys = p.table[(long long)b * p.maxb + lb];
        if (phys < 0 || phys >= p.num_blocks) {
            if (threadIdx.x == 0) set_error(p.err, phys < 0 ? 0x2u : 0x1u);
            return;
        }
        row_base = ((long long)phys * p.Hkv * p.bs + (pos % p.bs)) * D;
        head_stride = (long long)p.bs * D;
    }
    if constexpr (sizeof(Elt) == 1) {
        int8_t* kc = static_cast<int8_t*>(p.cache) + p.layer_off + row_base;
        float* sc = p.scales + p.sc_layer_off + row_base / D;
        const __nv_bfloat16* ks = static_cast<const __nv_bfloat16*>(p.k_new) + ((long long)b * p.n_new + i_tok) * p.Hkv * D;
        const __nv_bfloat16* vs = static_cast<const __nv_bfloat16*>(p.v_new) + ((long long)b * p.n_new + i_tok) * p.Hkv * D;
        if (D == 128)
            q8_write_token_rows<2>(kc, p.kv_off, head_stride, sc, p.sc_kv_off, head_stride / D, ks, vs, p.Hkv, p.rope,
                                   pos, p.theta);
        else
            q8_write_token_rows<4>(kc, p.kv_off, head_stride, sc, p.sc_kv_off, head_stride / D, ks, vs, p.Hkv, p.rope,
                                   pos, p.theta);
    } else {
        Elt* kc = static_cast<Elt*>(p.cache) + p.layer_off + row_base;
        const Elt* ks = static_cast<const Elt*>(p.k_new) + ((long long)b * p.n_new + i_tok) * p.Hkv * D;
        const Elt* vs = static_cast<const Elt*>(p.v_new) + ((long long)b * p.n_new + i_tok) * p.Hkv * D;
        write_token_rows<Elt>(kc, p.kv_off, head_stride, ks, vs, p.Hkv, D, p.rope, pos, p.theta);
    }
}

// kvc_prefill: the chunk's K (RoPE baked at its position, as an append stores
// it) and V rows of token blockIdx.x of sequence blockIdx.y, into the staging
// buffers [B][T][Hkv][D] (bf16).  Left-padding positions stage nothing.
__global__ void __launch_bounds__(256) prefill_stage_kernel(const __grid_constant__ AppendParams p,
                                                            __nv_bfloat16* kst, __nv_bfloat16* vst) {
    const int i_tok = blockIdx.x, b = blockIdx.y;
    const long long pos = (long long)p.pos[b] + i_tok;
    if (pos < 0) return;
    const long long row = ((long long)b * p.n_new + i_tok) * p.Hkv * p.D;
    write_token_rows<__nv_bfloat16>(kst + row, (long long)(vst - kst), p.D,
                                    static_cast<const __nv_bfloat16*>(p.k_new) + row,
                                    static_cast<const __nv_bfloat16*>(p.v_new) + row, p.Hkv, p.D, p.rope, pos,
                                    p.theta);
}

// INT8 cache: the chunk's rows as the cache will read them back, bf16 of
// code * row scale (the quantisation kvc_append applies: K rotated first when
// BAKED), so the chunk's tokens attend one another as the decode steps would.
// One warp per (token, kv head).
template <int NP>
__global__ void __launch_bounds__(256) prefill_stage_q8_kernel(const __grid_constant__ AppendParams p,
                                                               __nv_bfloat16* kst, __nv_bfloat16* vst) {
    constexpr int D = 64 * NP, HALF = 32 * NP;
    const int i_tok = blockIdx.x, b = blockIdx.y;
    const long long pos = (long long)p.pos[b] + i_tok;
    if (pos < 0) return;
    const int lane = threadIdx.x & 31;
    for (int hk = threadIdx.x >> 5; hk < p.Hkv; hk += blockDim.x >> 5) {
        const long long row = (((long long)b * p.n_new + i_tok) * p.Hkv + hk) * D;
        const __nv_bfloat16* kr = static_cast<const __nv_bfloat16*>(p.k_new) + row;
        const __nv_bfloat16* vr = static_cast<const __nv_bfloat16*>(p.v_new) + row;
        float kx[2 * NP], vx[2 * NP];
#pragma unroll
        for (int m = 0; m < NP; ++m) {
            const int i = lane + 32 * m;
            float x1 = __bfloat162float(kr[i]), x2 = __bfloat162float(kr[i + HALF]);
            if (p.rope == kRopeBaked) {
                float c, sn;
                rope_cos_sin(pos, p.theta[i], &c, &sn);
                const float y1 = x1 * c - x2 * sn, y2 = x1 * sn + x2 * c;
                x1 = y1;
                x2 = y2;
            }
            kx[2 * m] = x1;
            kx[2 * m + 1] = x2;
            vx[2 * m] = __bfloat162float(vr[i]);
            vx[2 * m + 1] = __bfloat162float(vr[i + HALF]);
        }
        int8_t kq[2 * NP], vq[2 * NP];
        const float sk = q8_quantize_lane<2 * NP>(kx, kq);
        const float sv = q8_quantize_lane<2 * NP>(vx, vq);
#pragma unroll
        for (int m = 0; m < NP; ++m) {
            const int i = lane + 32 * m;
            kst[row + i] = __float2bfloat16_rn((float)kq[2 * m] * sk);
            kst[row + i + HALF] = __float2bfloat16_rn((float)kq[2 * m + 1] * sk);
            vst[row + i] = __float2bfloat16_rn((float)vq[2 * m] * sv);
            vst[row + i + HALF] = __float2bfloat16_rn((float)vq[2 * m + 1] * sv);
        }
    }
}

cudaError_t launch_prefill_stage(const AppendParams& p, void* kst, void* vst, cudaStream_t stream) {
    __nv_bfloat16* k = static_cast<__nv_bfloat16*>(kst);
    __nv_bfloat16* v = static_cast<__nv_bfloat16*>(vst);
    if (p.scales) {                       // INT8 cache
        if (p.D == 128)
            prefill_stage_q8_kernel<2><<<dim3(p.n_new, p.B), 256, 0, stream>>>(p, k, v);
        else if (p.D == 256)
            prefill_stage_q8_kernel<4><<<dim3(p.n_new, p.B), 256, 0, stream>>>(p, k, v);
        else
            return cudaErrorInvalidValue;
    } else {
        prefill_stage_kernel<<<dim3(p.n_new, p.B), 256, 0, stream>>>(p, k, v);
    }
    return cudaGetLastError();
}

cudaError_t launch_append(int dtype, const AppendParams& p, cudaStream_t stream) {
    dim3 grid(p.n_new, p.B);
    if (dtype == 0)
        append_kernel<float><<<grid, 256, 0, stream>>>(p);
    else if (dtype == 1)
        append_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(p);
    else
        append_kernel<int8_t><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Paged work plan (stream-K).  The attended rows of all sequences, laid end
// to end, are cut into G <= `ctas` nearly equal contiguous shares
// [floor(x R / G), floor((x + 1) R / G)); the intersection of share x with
// sequence b is work item x + b (items of one sequence, and of one share, get
// consecutive indices; a share boundary that falls exactly on a sequence
// boundary leaves one index unused, marked -1).  The tensor-core decode of a
// batch cuts these shares itself from plan_rows_kernel's per-sequence rows
// (below); the fp32 decode, one CTA per item, takes them from two kernels,
// one CTA per sequence each, chained by programmatic dependent launch:
//   plan_count_kernel  R_b = attended rows of sequence b (blocks lb <= t_b / bs
//                      that are mapped and valid; [pool] "kernel forgets
//                      absent blocks").  With a new token to append
//                      (kvc_decode_step) it first writes that token's K/V.
//                      The last CTA to finish (an atomic ticket, no waiting)
//                      takes O_b = sum of R before b, R, G, and each sequence's
//                      first item and item count (a sequence with no attended
//                      row gets one empty item, for its zero output).
//   plan_items_kernel  the sequence-local prefix of rows per block; each item
//                      of sequence b is written by the thread whose blocks hold
//                      its first row.
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 256;
constexpr int kPlanPerThread = 16;

// Block-wide inclusive scan of one value per thread (kPlanThreads threads);
// returns the thread's inclusive prefix and the block total in *total.
template <typename T>
__device__ __forceinline__ T plan_block_scan(T v, T* s_warp, T* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int NW = kPlanThreads / 32;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const T u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
    }
    if (lane == 31) s_warp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        T x = lane < NW ? s_warp[lane] : T(0);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const T u = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += u;
        }
        if (lane < NW) s_warp[lane] = x;
    }
    __syncthreads();
    const T r = v + (warp > 0 ? s_warp[warp - 1] : T(0));
    *total = s_warp[NW - 1];
    __syncthreads();
    return r;
}

// Attended rows of kPlanPerThread logical blocks lb[j] < nb of one sequence
// (as paged_block_rows) whose table entries phys[j] are already loaded: every
// valid-bit load is issued before any is used.
__device__ __forceinline__ void plan_rows_of(const uint32_t* valid, uint32_t* err, const int* lb, int t, int nb,
                                             int bs, int num_blocks, const int* phys, int* rows) {
    uint32_t word[kPlanPerThread];
#pragma unroll
    for (int j = 0; j < kPlanPerThread; ++j) {
        const bool in = lb[j] < nb && phys[j] >= 0 && phys[j] < num_blocks;
        word[j] = (in && valid) ? __ldg(valid + (phys[j] >> 5)) : 0xffffffffu;
    }
#pragma unroll
    for (int j = 0; j < kPlanPerThread; ++j) {
        int r = 0;
        if (lb[j] < nb && phys[j] >= num_blocks) {
            set_error(err, 0x1u /* KVC_DEV_BAD_BLOCK */);
        } else if (lb[j] < nb && phys[j] >= 0 && ((word[j] >> (phys[j] & 31)) & 1u)) {
            r = lb[j] == t / bs ? (t - lb[j] * bs + 1) : bs;
        }
        rows[j] = r;
    }
}

// The same, loading the table entries first (all in flight together).
__device__ __forceinline__ void plan_block_rows(const int32_t* trow, const uint32_t* valid, uint32_t* err,
                                                const int* lb, int t, int nb, int bs, int num_blocks, int* rows,
                                                int* phys) {
#pragma unroll
    for (int j = 0; j < kPlanPerThread; ++j) phys[j] = lb[j] < nb ? __ldg(trow + lb[j]) : -1;
    plan_rows_of(valid, err, lb, t, nb, bs, num_blocks, phys, rows);
}

__device__ __forceinline__ void plan_pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void plan_pdl_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// The step's new token (kvc_decode_step) of sequence b at position traw, to
// row traw mod bs of logical block traw / bs.
// INT8 cache: the new token's rows at element row_base of the layer's K half.
// Kept out of line: inlined, it slowed the bf16 plan kernel by several us.
__device__ __noinline__ void plan_append_q8(const PlanParams& p, long long row_base, long long tok, int traw) {
    int8_t* kc = static_cast<int8_t*>(p.cache) + p.layer_off + row_base;
    float* sc = p.scales + p.sc_layer_off + row_base / p.D;
    const __nv_bfloat16* ks = static_cast<const __nv_bfloat16*>(p.k_new) + tok;
    const __nv_bfloat16* vs = static_cast<const __nv_bfloat16*>(p.v_new) + tok;
    const long long hs = (long long)p.bs * p.D;
    if (p.D == 128)
        q8_write_token_rows<2>(kc, p.kv_off, hs, sc, p.sc_kv_off, p.bs, ks, vs, p.Hkv, p.rope, traw, p.theta);
    else
        q8_write_token_rows<4>(kc, p.kv_off, hs, sc, p.sc_kv_off, p.bs, ks, vs, p.Hkv, p.rope, traw, p.theta);
}

__device__ __forceinline__ void plan_append(const PlanParams& p, int b, int traw, int known_phys = -2) {
    if (!p.k_new || traw < 0) return;
    const long long lb = traw / p.bs;
    if (lb >= p.maxb) {
        if (threadIdx.x == 0) set_error(p.err, 0x4u /* KVC_DEV_BAD_POSITION */);
        return;
    }
    const int phys = known_phys >= -1 ? known_phys : p.table[(long long)b * p.maxb + lb];
    if (phys < 0 || phys >= p.num_blocks) {
        if (threadIdx.x == 0) set_error(p.err, phys < 0 ? 0x2u : 0x1u);
        return;
    }
    const long long row_base = ((long long)phys * p.Hkv * p.bs + (traw % p.bs)) * p.D;
    const long long tok = (long long)b * p.Hkv * p.D;
    if (p.elt == 1)
        plan_append_q8(p, row_base, tok, traw);
    else if (p.elt == 4)
        write_token_rows<float>(static_cast<float*>(p.cache) + p.layer_off + row_base, p.kv_off,
                                (long long)p.bs * p.D, static_cast<const float*>(p.k_new) + tok,
                                static_cast<const float*>(p.v_new) + tok, p.Hkv, p.D, p.rope, traw, p.theta);
    else
        write_token_rows<__nv_bfloat16>(static_cast<__nv_bfloat16*>(p.cache) + p.layer_off + row_base, p.kv_off,
                                        (long long)p.bs * p.D, static_cast<const __nv_bfloat16*>(p.k_new) + tok,
                                        static_cast<const __nv_bfloat16*>(p.v_new) + tok, p.Hkv, p.D, p.rope, traw,
                                        p.theta);
}

// First item and item count of a sequence with O_b rows before it and R_b rows.
__device__ __forceinline__ int2 plan_seq_items(int b, long long Ob, long long Rb, long long R, int G) {
    const int2 fl = paged_seq_shares(Ob, Rb, R, G);
    return make_int2(fl.x + b, fl.y - fl.x + 1);
}

// The items of sequence b (O_b, R_b; shares of R rows into G) whose first row
// lies in this thread's blocks lb0 .. lb0 + kPlanPerThread - 1, which hold its
// sequence-local rows [rs, re); v = their inclusive prefix from rs, ph = their
// physical blocks.  Each item gets its record (seq, first block, first row,
// rows) and, for the decode's copy warp, (t_b, first slot and count of the
// sequence's partials, physical block of its first block).  Share x
// starts at floor(x R / G), inside [O_b + rs, O_b + re) iff
// ceil((O_b + rs) G / R) <= x < ceil((O_b + re) G / R); the sequence's first
// item starts at its row 0 when its share began in an earlier sequence.
__device__ __forceinline__ void plan_write_items(const PlanParams& p, int b, int tb, long long Ob, long long Rb,
                                                 long long R, int G, int2 si, int lb0, const int* v, const int* ph,
                                                 long long rs, long long re) {
    if (re <= rs) return;
    const int fx = si.x - b, lx = fx + si.y - 1;
    const long long A = Ob + rs, Bnd = Ob + re;
    int x0 = (int)((A * G + R - 1) / R), x1 = (int)((Bnd * G + R - 1) / R);
    if (x0 < fx) x0 = fx;
    if (x1 > lx + 1) x1 = lx + 1;
    if (rs == 0 && (long long)fx * R / G < Ob && x0 > fx) x0 = fx;
    for (int x = x0; x < x1; ++x) {
        const long long lo = (long long)x * R / G, hi = (long long)(x + 1) * R / G;
        const long long s0 = (lo > Ob ? lo : Ob) - Ob;
        const long long s1 = (hi < Ob + Rb ? hi : Ob + Rb) - Ob;
        if (s1 <= s0 || s0 < rs || s0 >= re) continue;
        // first block j whose prefix exceeds s0 (unrolled: v and ph stay in registers)
        int j = 0, phj = ph[0];
        long long before = rs;
#pragma unroll
        for (int jj = 0; jj < kPlanPerThread - 1; ++jj) {
            if (rs + v[jj] <= s0) {
                j = jj + 1;
                before = rs + v[jj];
                phj = ph[jj + 1];
            }
        }
        const int i = x + b;
        if (x < 0 || x >= p.ctas || i >= p.max_items) {
            index_fault(p.err, 6, i);
            continue;
        }
        p.items[i] = make_int4(b, lb0 + j, (int)(s0 - before), (int)(s1 - s0));
        p.item_info[i] = make_int4(tb, si.x, si.y, phj);
        atomicMin(&p.cta_items[x].x, i);
        atomicAdd(&p.cta_items[x].y, 1);
    }
}

__device__ __forceinline__ void plan_write_empty_item(const PlanParams& p, int b, int tb, int2 si) {
    const int fx = si.x - b;
    if (fx < 0 || fx >= p.ctas || si.x >= p.max_items) {
        index_fault(p.err, 6, si.x);
        return;
    }
    p.items[si.x] = make_int4(b, 0, 0, 0);
    p.item_info[si.x] = make_int4(tb, si.x, si.y, -1);
    atomicMin(&p.cta_items[fx].x, si.x);
    atomicAdd(&p.cta_items[fx].y, 1);
}

__device__ __forceinline__ void plan_init_items(const PlanParams& p) {
    for (int i = threadIdx.x; i < p.max_items; i += kPlanThreads) p.items[i] = make_int4(-1, 0, 0, 0);
    for (int i = threadIdx.x; i < p.ctas; i += kPlanThreads) p.cta_items[i] = make_int2(0x7fffffff, 0);
}

__device__ __forceinline__ void plan_write_header(const PlanParams& p, long long R, int G) {
    p.n_items[0] = G + p.B;
    p.n_items[1] = G;
    *reinterpret_cast<long long*>(p.n_items + 2) = R;
}

// Shares of R rows: no more than the CTAs, and no empty share.
__device__ __forceinline__ int plan_shares(long long R, int ctas) { return paged_share_count(R, ctas); }

__global__ void __launch_bounds__(kPlanThreads) plan_count_kernel(const __grid_constant__ PlanParams p) {
    __shared__ int s_wi[32];
    __shared__ long long s_wl[32];
    __shared__ int s_last;
    const int tid = threadIdx.x;
    const int b = blockIdx.x;
    plan_pdl_wait();            // positions, table, valid bits may come from the previous kernel
    // the next kernel (the decode kernel, or plan_items_kernel) may launch now:
    // it waits for this grid to complete before it reads anything
    plan_pdl_launch();
    const int32_t* trow = p.table + (long long)b * p.maxb;
    constexpr int kChunk = kPlanThreads * kPlanPerThread;
    __shared__ int s_tok_phys;

    if (gridDim.x == 1 && p.maxb <= kChunk) {
        // one sequence whose blocks fit one pass: the whole plan here (the
        // host launches no plan_items_kernel in this case; same test).  The
        // table is loaded in full without waiting for the position.
        const int lb0 = tid * kPlanPerThread;
        int lbs[kPlanPerThread], v[kPlanPerThread], ph[kPlanPerThread];
#pragma unroll
        for (int j = 0; j < kPlanPerThread; ++j) {
            lbs[j] = lb0 + j;
            ph[j] = lb0 + j < p.maxb ? __ldg(trow + lb0 + j) : -1;
        }
        if (tid == 0) s_tok_phys = -2;
        const int traw = __ldg(p.pos);
        const int t = clamp_paged_t(traw, p.maxb, p.bs);
        const int nb = t < 0 ? 0 : t / p.bs + 1;
        plan_rows_of(p.valid, p.err, lbs, t, nb, p.bs, p.num_blocks, ph, v);
        int tsum = 0;
#pragma unroll
        for (int j = 0; j < kPlanPerThread; ++j) {
            tsum += v[j];
            v[j] = tsum;
        }
        int R32 = 0;
        const int incl = plan_block_scan<int>(tsum, s_wi, &R32);   // (its barriers order the slot's reset)
#pragma unroll
        for (int j = 0; j < kPlanPerThread; ++j)
            if (traw >= 0 && lbs[j] == traw / p.bs) s_tok_phys = ph[j];
        const long long R = R32;
        const int G = plan_shares(R, p.ctas);
        const int2 si = plan_seq_items(0, 0, R, R, G);
        plan_init_items(p);
        if (tid == 0) {
            p.seq_rows[0] = R32;
            p.seq_off[0] = 0;
            p.seq_items[0] = si;
            plan_write_header(p, R, G);
        }
        __syncthreads();
        if (R > 0)
            plan_write_items(p, 0, traw, 0, R, R, G, si, lb0, v, ph, incl - tsum, incl);
        else if (tid == 0)
            plan_write_empty_item(p, 0, traw, si);
        plan_append(p, b, traw, s_tok_phys);
        return;
    }

    const int traw = p.pos[b];
    const int t = clamp_paged_t(traw, p.maxb, p.bs);
    const int nb = t < 0 ? 0 : t / p.bs + 1;

    // R_b
    int sum = 0;
    for (int base = 0; base < nb; base += kChunk) {
        int lbs[kPlanPerThread], v[kPlanPerThread], ph[kPlanPerThread];
#pragma unroll
        for (int j = 0; j < kPlanPerThread; ++j) lbs[j] = base + j * kPlanThreads + tid;
        plan_block_rows(trow, p.valid, p.err, lbs, t, nb, p.bs, p.num_blocks, v, ph);
#pragma unroll
        for (int j = 0; j < kPlanPerThread; ++j) sum += v[j];
    }
    plan_append(p, b, traw);
    int rb = 0;
    plan_block_scan<int>(sum, s_wi, &rb);
    if (tid == 0) p.seq_rows[b] = rb;

    // the last CTA to get here: offsets, G, and each sequence's first item
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(p.ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    plan_init_items(p);
    long long run = 0;
    for (int base = 0; base < p.B; base += kPlanThreads) {
        const int bb = base + tid;
        const long long r = bb < p.B ? (long long)__ldcg(&p.seq_rows[bb]) : 0;
        long long chunk = 0;
        const long long incl = plan_block_scan<long long>(r, s_wl, &chunk);
        if (bb < p.B) p.seq_off[bb] = run + incl - r;
        run += chunk;
    }
    const long long R = run;
    const int G = plan_shares(R, p.ctas);
    __syncthreads();
    for (int bb = tid; bb < p.B; bb += kPlanThreads)
        p.seq_items[bb] = plan_seq_items(bb, __ldcg(&p.seq_off[bb]), __ldcg(&p.seq_rows[bb]), R, G);
    if (tid == 0) {
        plan_write_header(p, R, G);
        *p.ticket = 0u;                       // ready for the next plan
    }
}

__global__ void __launch_bounds__(kPlanThreads) plan_items_kernel(const __grid_constant__ PlanParams p) {
    __shared__ int s_wi[32];
    const int tid = threadIdx.x;
    const int b = blockIdx.x;
    // Positions, table and valid bits were final when plan_count_kernel passed
    // its own wait (this grid launches only after that): the rows of the first
    // pass are loaded before waiting for plan_count_kernel's results.
    const int32_t* trow = p.table + (long long)b * p.maxb;
    const int traw = __ldg(p.pos + b);
    const int t = clamp_paged_t(traw, p.maxb, p.bs);
    const int nb = t < 0 ? 0 : t / p.bs + 1;
    constexpr int kChunk = kPlanThreads * kPlanPerThread;
    int lbs[kPlanPerThread], v[kPlanPerThread], ph[kPlanPerThread];
#pragma unroll
    for (int j = 0; j < kPlanPerThread; ++j) lbs[j] = tid * kPlanPerThread + j;
    plan_block_rows(trow, p.valid, nullptr, lbs, t, nb, p.bs, p.num_blocks, v, ph);
    // No early trigger here: the decode grid fills every SM (two CTAs each)
    // and must not launch while plan CTAs still hold registers, or its last
    // CTAs start only when others finish.
    plan_pdl_wait();
    const int G = __ldcg(&p.n_items[1]);
    const long long R = __ldcg(reinterpret_cast<const long long*>(p.n_items + 2));
    const long long Ob = __ldcg(&p.seq_off[b]);
    const long long Rb = __ldcg(&p.seq_rows[b]);
    const int2 si = __ldcg(&p.seq_items[b]);
    if (Rb <= 0) {              // one empty item
        if (tid == 0) plan_write_empty_item(p, b, traw, si);
        return;
    }
    int carry = 0;
    for (int base = 0; base < nb; base += kChunk) {
        const int lb0 = base + tid * kPlanPerThread;
        if (base > 0) {
#pragma unroll
            for (int j = 0; j < kPlanPerThread; ++j) lbs[j] = lb0 + j;
            plan_block_rows(trow, p.valid, nullptr, lbs, t, nb, p.bs, p.num_blocks, v, ph);
        }
        int tsum = 0;
#pragma unroll
        for (int j = 0; j < kPlanPerThread; ++j) {
            tsum += v[j];
            v[j] = tsum;
        }
        int chunk = 0;
        const int incl = plan_block_scan<int>(tsum, s_wi, &chunk);
        plan_write_items(p, b, traw, Ob, Rb, R, G, si, lb0, v, ph, carry + incl - tsum, carry + incl);
        carry += chunk;
    }
}

// Rows and attended-block directory of each sequence, for the tensor-core
// decode, whose CTAs cut their own shares from them (one CTA per sequence):
//   seq_rows[b]      R_b, as plan_count_kernel counts it;
//   dir[b][g]        (bits i: logical block 32 g + i is attended, attended
//                    blocks of b before block 32 g), for g <= t_b / bs / 32.
//   refs[q]          += 1 for each sequence that attends physical block q:
//                    blocks read by one sequence stream through L2 as
//                    evict-first, shared ones (prefixes) stay for their
//                    other readers.
// Every attended block but a sequence's last holds bs rows, so its row r lies
// in the attended block of rank r / bs, which the directory finds with one
// search over g and one bit select.  With a new token to append
// (kvc_decode_step) the CTA writes it first, as plan_count_kernel does.
__global__ void __launch_bounds__(kPlanThreads) plan_rows_kernel(const __grid_constant__ PlanParams p) {
    constexpr int NW = kPlanThreads / 32;
    constexpr int kGroups = NW * kPlanPerThread;      // 32-block groups of one pass
    constexpr int kChunk = kPlanThreads * kPlanPerThread;
    constexpr int kAppPairs = 4;                      // bf16 append: (kv head, pair) units per thread
    __shared__ int s_grp[kGroups];
    __shared__ int s_wi[32];
    __shared__ int s_pass;
    __shared__ int s_tok_phys;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    plan_pdl_wait();            // positions, table, valid bits may come from the previous kernel
    // the decode kernel may launch now: it waits for this grid to complete
    // before it reads anything
    plan_pdl_launch();
    const int32_t* trow = p.table + (long long)b * p.maxb;
    // Issued together, before any is used: the position, the table entries of
    // the first pass (all of them, not only those the position reaches) and,
    // on a bf16 cache, the step's new token.
    const int traw = p.pos[b];
    int ph0[kPlanPerThread];
#pragma unroll
    for (int j = 0; j < kPlanPerThread; ++j) {
        const int lb = j * kPlanThreads + tid;
        ph0[j] = lb < p.maxb ? __ldg(trow + lb) : -1;
    }
    const int half = p.D / 2;
    const bool app16 = p.k_new && p.elt == 2 && p.Hkv * half <= kAppPairs * kPlanThreads;
    __nv_bfloat162 kx[kAppPairs], vx[kAppPairs];      // (x_i, x_{i + D/2}) of unit tid + u kPlanThreads
    if (app16) {
        const __nv_bfloat16* ks = static_cast<const __nv_bfloat16*>(p.k_new) + (long long)b * p.Hkv * p.D;
        const __nv_bfloat16* vs = static_cast<const __nv_bfloat16*>(p.v_new) + (long long)b * p.Hkv * p.D;
#pragma unroll
        for (int u = 0; u < kAppPairs; ++u) {
            const int idx = tid + u * kPlanThreads;
            if (idx < p.Hkv * half) {
                const int off = (idx / half) * p.D + idx % half;
                kx[u] = __halves2bfloat162(ks[off], ks[off + half]);
                vx[u] = __halves2bfloat162(vs[off], vs[off + half]);
            }
        }
    }
    if (tid == 0) s_tok_phys = -2;
    __syncthreads();
    const int t = clamp_paged_t(traw, p.maxb, p.bs);
    const int nb = t < 0 ? 0 : t / p.bs + 1;
    const int tok_lb = traw >= 0 ? traw / p.bs : -1;
    int2* drow = p.dir + (long long)b * p.dir_groups;
    int sum = 0, before = 0;
    for (int base = 0; base < nb; base += kChunk) {
        // thread tid takes blocks base + j kPlanThreads + tid: warp w's lanes
        // cover the 32 blocks of group (base + j kPlanThreads) / 32 + w
        int lbs[kPlanPerThread], v[kPlanPerThread], ph[kPlanPerThread];
#pragma unroll
        for (int j = 0; j < kPlanPerThread; ++j) lbs[j] = base + j * kPlanThreads + tid;
        if (base == 0) {
#pragma unroll
            for (int j = 0; j < kPlanPerThread; ++j) ph[j] = lbs[j] < nb ? ph0[j] : -1;
            plan_rows_of(p.valid, p.err, lbs, t, nb, p.bs, p.num_blocks, ph, v);
        } else {
            plan_block_rows(trow, p.valid, p.err, lbs, t, nb, p.bs, p.num_blocks, v, ph);
        }
        uint32_t m[kPlanPerThread];
#pragma unroll
        for (int j = 0; j < kPlanPerThread; ++j) {
            if (lbs[j] == tok_lb) s_tok_phys = ph[j];        // the new token's block
            if (v[j] > 0) atomicAdd(p.refs + ph[j], 1u);
            sum += v[j];
            m[j] = __ballot_sync(0xffffffffu, v[j] > 0);
            if (lane == 0) s_grp[j * NW + warp] = __popc(m[j]);
        }
        __syncthreads();
        if (warp == 0) {
            // exclusive prefix of the pass's groups in block order (4 per lane)
            int c[kGroups / 32], tot = 0;
#pragma unroll
            for (int k = 0; k < kGroups / 32; ++k) {
                c[k] = s_grp[lane * (kGroups / 32) + k];
                tot += c[k];
            }
            int incl = tot;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += u;
            }
            int ex = before + incl - tot;
#pragma unroll
            for (int k = 0; k < kGroups / 32; ++k) {
                s_grp[lane * (kGroups / 32) + k] = ex;
                ex += c[k];
            }
            if (lane == 31) s_pass = incl;
        }
        __syncthreads();
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < kPlanPerThread; ++j) {
                const int lb0 = base + j * kPlanThreads + warp * 32;
                if (lb0 < nb) drow[lb0 >> 5] = make_int2((int)m[j], s_grp[j * NW + warp]);
            }
        }
        before += s_pass;
        __syncthreads();
    }
    const int tok_phys = s_tok_phys;
    if (!app16) {
        plan_append(p, b, traw, tok_phys);
    } else if (traw >= 0) {
        // the new token's rows from the registers loaded above (as plan_append)
        const int phys = tok_lb < p.maxb ? (tok_phys >= -1 ? tok_phys : __ldg(trow + tok_lb)) : -1;
        if (tok_lb >= p.maxb || phys < 0 || phys >= p.num_blocks) {
            if (tid == 0) set_error(p.err, tok_lb >= p.maxb ? 0x4u : (phys < 0 ? 0x2u : 0x1u));
        } else {
            __nv_bfloat16* kc = static_cast<__nv_bfloat16*>(p.cache) + p.layer_off +
                                ((long long)phys * p.Hkv * p.bs + traw % p.bs) * p.D;
            const long long hs = (long long)p.bs * p.D;
#pragma unroll
            for (int u = 0; u < kAppPairs; ++u) {
                const int idx = tid + u * kPlanThreads;
                if (idx < p.Hkv * half) {
                    const int h = idx / half, i = idx % half;
                    __nv_bfloat16* kd = kc + h * hs;
                    __nv_bfloat16* vd = kd + p.kv_off;
                    __nv_bfloat16 k1 = kx[u].x, k2 = kx[u].y;
                    if (p.rope == kRopeBaked) {
                        float c, sn;
                        rope_cos_sin((long long)traw, p.theta[i], &c, &sn);
                        const float x1 = __bfloat162float(k1), x2 = __bfloat162float(k2);
                        k1 = __float2bfloat16_rn(x1 * c - x2 * sn);
                        k2 = __float2bfloat16_rn(x1 * sn + x2 * c);
                    }
                    kd[i] = k1;
                    kd[i + half] = k2;
                    vd[i] = vx[u].x;
                    vd[i + half] = vx[u].y;
                }
            }
        }
    }
    int rb = 0;
    plan_block_scan<int>(sum, s_wi, &rb);
    if (tid == 0) p.seq_rows[b] = rb;
}

cudaError_t launch_plan_rows(const PlanParams& p, cudaStream_t stream) {
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.B);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, plan_rows_kernel, p);
}

cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream) {
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.B);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, plan_count_kernel, p);
    if (e != cudaSuccess) return e;
    // one sequence of at most kPlanThreads * kPlanPerThread blocks: planned in one kernel
    if (p.B == 1 && (long long)p.maxb <= (long long)kPlanThreads * kPlanPerThread) return cudaSuccess;
    return cudaLaunchKernelEx(&cfg, plan_items_kernel, p);
}

// ---------------------------------------------------------------------------
// block table / residency scatter ([share] 5.1 block manager, [pool] valid mask)
// ---------------------------------------------------------------------------
__global__ void table_write_kernel(const __grid_constant__ TableParams p) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    const int s = p.seq[i], lb = p.lb[i], ph = p.phys[i];
    if (s < 0 || s >= p.B || lb < 0 || lb >= p.maxb || ph < -1 || ph >= p.num_blocks) {
        set_error(p.err, 0x10u /* KVC_DEV_BAD_ENTRY */);
        return;
    }
    p.table[(long long)s * p.maxb + lb] = ph;
    if (ph >= 0 && p.valid) atomicOr(&p.valid[ph >> 5], 1u << (ph & 31));
}

__global__ void valid_write_kernel(const __grid_constant__ TableParams p) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    const int ph = p.phys[i];
    if (ph < 0 || ph >= p.num_blocks) {
        set_error(p.err, 0x10u);
        return;
    }
    const uint32_t bit = 1u << (ph & 31);
    if (p.value[i])
        atomicOr(&p.valid[ph >> 5], bit);
    else
        atomicAnd(&p.valid[ph >> 5], ~bit);
}

cudaError_t launch_table_write(const TableParams& p, cudaStream_t stream) {
    table_write_kernel<<<(p.n + 255) / 256, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_valid_write(const TableParams& p, cudaStream_t stream) {
    valid_write_kernel<<<(p.n + 255) / 256, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kvc
