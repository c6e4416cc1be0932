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
template <typename Elt>
__global__ void __launch_bounds__(256) append_kernel(const __grid_constant__ AppendParams p) {
    using TR = EltTraits<Elt>;
    const int i_tok = blockIdx.x, b = blockIdx.y;
    const int t0 = p.pos[b];
    const long long pos = (long long)t0 + i_tok;
    if (pos < 0) return;                       // left padding
    const long long last = (long long)t0 + p.n_new - 1;
    const int D = p.D, half = D / 2;

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
    Elt* kc = static_cast<Elt*>(p.cache) + p.layer_off + row_base;
    Elt* vc = kc + p.kv_off;
    const Elt* ks = static_cast<const Elt*>(p.k_new) + ((long long)b * p.n_new + i_tok) * p.Hkv * D;
    const Elt* vs = static_cast<const Elt*>(p.v_new) + ((long long)b * p.n_new + i_tok) * p.Hkv * D;

    for (int idx = threadIdx.x; idx < p.Hkv * half; idx += blockDim.x) {
        const int h = idx / half, i = idx % half;
        const Elt* kr = ks + (long long)h * D;
        const Elt* vr = vs + (long long)h * D;
        Elt* kd = kc + h * head_stride;
        Elt* vd = vc + h * head_stride;
        const Elt k1 = kr[i], k2 = kr[i + half];
        if (p.rope == kRopeBaked) {
            float c, s;
            rope_cos_sin((double)pos, p.theta[i], &c, &s);
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

cudaError_t launch_append(int dtype, const AppendParams& p, cudaStream_t stream) {
    dim3 grid(p.n_new, p.B);
    if (dtype == 0)
        append_kernel<float><<<grid, 256, 0, stream>>>(p);
    else
        append_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Paged work plan: split each sequence's attended rows into work items of
// nearly equal size, in proportion to its length, so one long sequence (a
// 256K-token pool) or a batch of mixed lengths keeps every SM busy.
//   1. rows[b][lb] = attended rows of logical block lb (0 if unmapped, not
//      valid, or past t), then an inclusive prefix sum per sequence;
//   2. n_b = 1 + floor(R_b * extra / R) items for sequence b (R_b its rows,
//      R the batch total, extra = max_items - B), first item by prefix sum;
//   3. item k of b starts at row floor(k R_b / n_b) of b's attended rows,
//      located by binary search in the prefix.
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ PlanParams p) {
    __shared__ long long s_total;
    __shared__ int s_carry;
    __shared__ int s_warp[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // 1. rows per block
    for (long long idx = tid; idx < (long long)p.B * p.maxb; idx += kPlanThreads) {
        const int b = (int)(idx / p.maxb), lb = (int)(idx % p.maxb);
        const int t = clamp_paged_t(p.pos[b], p.maxb, p.bs);
        int phys = -1;
        p.rows[idx] = paged_block_rows(p.table + (long long)b * p.maxb, p.valid, p.err, lb, t, p.bs,
                                       p.num_blocks, &phys);
    }
    if (tid == 0) {
        s_total = 0;
        s_carry = 0;
    }
    __syncthreads();
    // inclusive prefix per sequence: one warp per sequence
    for (int b = warp; b < p.B; b += kPlanThreads / 32) {
        int run = 0;
        int32_t* r = p.rows + (long long)b * p.maxb;
        for (int base = 0; base < p.maxb; base += 32) {
            const int lb = base + lane;
            int v = lb < p.maxb ? r[lb] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += u;
            }
            if (lb < p.maxb) r[lb] = run + v;
            run += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) atomicAdd((unsigned long long*)&s_total, (unsigned long long)run);
    }
    __syncthreads();

    // 2. items per sequence and first item (block-wide exclusive scan)
    const long long R = s_total;
    const int extra = p.max_items - p.B;
    for (int base = 0; base < p.B; base += kPlanThreads) {
        const int b = base + tid;
        int n = 0;
        if (b < p.B) {
            const long long Rb = p.rows[(long long)b * p.maxb + p.maxb - 1];
            n = 1 + (R > 0 ? (int)((Rb * (long long)extra) / R) : 0);
        }
        // exclusive scan of n over the block
        int v = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += u;
        }
        if (lane == 31) s_warp[warp] = v;
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
        const int incl = v + (warp > 0 ? s_warp[warp - 1] : 0) + s_carry;
        if (b < p.B) p.seq_items[b] = make_int2(incl - n, n);
        __syncthreads();
        if (tid == kPlanThreads - 1) s_carry = incl;
        __syncthreads();
    }
    if (tid == 0) *p.n_items = s_carry;

    // 3. item boundaries: one warp per sequence, lanes over its items
    for (int b = warp; b < p.B; b += kPlanThreads / 32) {
        const int32_t* pre = p.rows + (long long)b * p.maxb;
        const long long Rb = pre[p.maxb - 1];
        const int2 si = p.seq_items[b];
        for (int k = lane; k < si.y; k += 32) {
            const long long start = (long long)k * Rb / si.y;
            const long long stop = (long long)(k + 1) * Rb / si.y;
            int lb = 0, off = 0;
            if (stop > start) {
                // first block whose inclusive prefix exceeds `start`
                int lo = 0, hi = p.maxb - 1;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (pre[mid] > start) hi = mid; else lo = mid + 1;
                }
                lb = lo;
                off = (int)(start - (lb > 0 ? pre[lb - 1] : 0));
            }
            p.items[si.x + k] = make_int4(b, lb, off, (int)(stop - start));
        }
    }
}

cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream) {
    plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
    return cudaGetLastError();
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
