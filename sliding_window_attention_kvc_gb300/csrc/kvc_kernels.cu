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
            rope_cos_sin((long long)pos, p.theta[i], &c, &s);
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
// Paged work plan (stream-K).  The attended rows of all sequences, laid end
// to end, are cut into `ctas` nearly equal contiguous shares; the
// intersection of share x with sequence b is work item x + b (items of one
// sequence, and of one share, get consecutive indices; a share boundary that
// falls exactly on a sequence boundary leaves one index unused, marked -1).
//   1. rows[b][lb] = attended rows of logical block lb (0 if unmapped, not
//      valid, or past t); a block-wide inclusive scan over the flattened
//      [B][max_blocks] array turns it into P, so sequence b starts at
//      O_b = P[b * maxb - 1] and holds R_b = P[(b + 1) * maxb - 1] - O_b rows;
//   2. per sequence: the shares overlapping [O_b, O_b + R_b) (a sequence with
//      no attended row still gets one empty item, for its zero output), each
//      item's first block and row by binary search in P.
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;
constexpr int kPlanPerThread = 8;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ PlanParams p) {
    __shared__ int s_warp[32];
    __shared__ int s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long n = (long long)p.B * p.maxb;

    for (int i = tid; i < p.max_items; i += kPlanThreads) p.items[i] = make_int4(-1, 0, 0, 0);
    for (int i = tid; i < p.ctas; i += kPlanThreads) p.cta_items[i] = make_int2(0x7fffffff, 0);
    if (tid == 0) s_carry = 0;
    __syncthreads();

    // 1. rows per block and their block-wide inclusive scan, in chunks
    for (long long base = 0; base < n; base += (long long)kPlanThreads * kPlanPerThread) {
        int v[kPlanPerThread];
        int tsum = 0;
#pragma unroll
        for (int j = 0; j < kPlanPerThread; ++j) {
            const long long idx = base + (long long)tid * kPlanPerThread + j;
            int r = 0;
            if (idx < n) {
                const int b = (int)(idx / p.maxb), lb = (int)(idx % p.maxb);
                const int t = clamp_paged_t(p.pos[b], p.maxb, p.bs);
                int phys = -1;
                r = paged_block_rows(p.table + (long long)b * p.maxb, p.valid, p.err, lb, t, p.bs, p.num_blocks,
                                     &phys);
            }
            tsum += r;
            v[j] = tsum;
        }
        int w = tsum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += u;
        }
        if (lane == 31) s_warp[warp] = w;
        __syncthreads();
        if (warp == 0) {
            int x = s_warp[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += u;
            }
            s_warp[lane] = x;
        }
        __syncthreads();
        const int before = s_carry + (warp > 0 ? s_warp[warp - 1] : 0) + (w - tsum);
#pragma unroll
        for (int j = 0; j < kPlanPerThread; ++j) {
            const long long idx = base + (long long)tid * kPlanPerThread + j;
            if (idx < n) p.rows[idx] = before + v[j];
        }
        __syncthreads();
        if (tid == 0) s_carry += s_warp[31];
        __syncthreads();
    }
    const long long R = s_carry;
    const int G = (int)(R < p.ctas ? (R > 0 ? R : 1) : p.ctas);   // no empty shares

    // 2a. per sequence: offset, rows, first and last share
    for (int b = tid; b < p.B; b += kPlanThreads) {
        const int32_t* P = p.rows;
        const long long Ob = b > 0 ? P[(long long)b * p.maxb - 1] : 0;
        const long long Rb = P[(long long)(b + 1) * p.maxb - 1] - Ob;
        int fx, lx;
        if (Rb > 0) {
            fx = streamk_share_of(Ob, R, G);
            lx = streamk_share_of(Ob + Rb - 1, R, G);
        } else {
            fx = lx = R > 0 ? streamk_share_of(Ob < R ? Ob : R - 1, R, G) : 0;
        }
        p.seq_items[b] = make_int2(fx + b, lx - fx + 1);
    }
    __syncthreads();
    // 2b. one thread per item index i = x + b: its sequence by binary search
    // over the sequences' first items, then its first block and row
    for (int i = tid; i < G + p.B && i < p.max_items; i += kPlanThreads) {
        int lo_s = 0, hi_s = p.B - 1;
        while (lo_s < hi_s) {                 // last sequence whose first item <= i
            const int mid = (lo_s + hi_s + 1) >> 1;
            if (p.seq_items[mid].x <= i) lo_s = mid; else hi_s = mid - 1;
        }
        const int b = lo_s;
        const int2 si = p.seq_items[b];
        if (i < si.x || i >= si.x + si.y) continue;      // unused index (stays -1)
        const int x = i - b;
        if (x < 0 || x >= p.ctas) {
            index_fault(p.err, 6, i);
            continue;
        }
        const int32_t* P = p.rows;
        const long long Ob = b > 0 ? P[(long long)b * p.maxb - 1] : 0;
        const long long Rb = P[(long long)(b + 1) * p.maxb - 1] - Ob;
        const long long lo = (long long)x * R / G, hi = (long long)(x + 1) * R / G;
        const long long s0 = (lo > Ob ? lo : Ob) - Ob;
        const long long s1 = (hi < Ob + Rb ? hi : Ob + Rb) - Ob;
        int lb = 0, off = 0;
        if (s1 > s0) {
            // first block whose (sequence-local) inclusive prefix exceeds s0
            int lo_b = 0, hi_b = p.maxb - 1;
            const int32_t* Pb = P + (long long)b * p.maxb;
            while (lo_b < hi_b) {
                const int mid = (lo_b + hi_b) >> 1;
                if (Pb[mid] - Ob > s0) hi_b = mid; else lo_b = mid + 1;
            }
            lb = lo_b;
            off = (int)(s0 - ((lb > 0 ? Pb[lb - 1] : Ob) - Ob));
        }
        p.items[i] = make_int4(b, lb, off, (int)(s1 > s0 ? s1 - s0 : 0));
        atomicMin(&p.cta_items[x].x, i);
        atomicAdd(&p.cta_items[x].y, 1);
    }
    if (tid == 0) *p.n_items = G + p.B;
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
