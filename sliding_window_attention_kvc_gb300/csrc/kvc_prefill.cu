// Chunked prefill attention for bf16 caches at head_dim 64 (head_dim 128 runs
// on the tcgen05 kernel of kvc_prefill_tc.cu) ([pool] "the real cost of long
// context": prefill in chunks of 128-256 tokens, one mechanism with the paged
// pool; [ring] 3.1 and 5.2: during prefill the window is a mask on the score
// matrix).
//
// Token i of a chunk (position t = pos0[b] + i) attends its layout's set A(t):
// the window t-W+1 .. t (with pinned sinks 0 .. S-1), or every p <= t whose
// block is mapped and valid.  Keys before pos0 come from the cache as it
// stands; keys of the chunk come from the staged rows (K rotated as an append
// stores it), so that a ring slot the chunk will overwrite is still read.
// kvc_prefill appends the chunk afterwards.
//
// One CTA: 64 (token, q head) rows of one kv head of one sequence -- 64 / G
// tokens of the chunk times the G q heads of the group -- as four warps of 16
// rows.  Keys stream through shared memory in tiles of 64 rows (K and V),
// double-buffered with cp.async, gathered row by row (ring slots, sink slots,
// paged blocks, staged chunk rows).  S = Q K^T and O += P V are mma.sync
// m16n8k16 (bf16 in, fp32 accumulate) on ldmatrix fragments of 128-byte-swizzled
// rows; the softmax is online, in base 2, per row.
#include "kvc_decode.cuh"

namespace kvc {

constexpr int kPfRows = 64;       // (token, q head) rows per CTA
constexpr int kPfKeys = 64;       // keys per tile
constexpr int kPfThreads = 128;

template <int D>
struct PfShape {
    static constexpr int kChunks = D / 8;                  // 16-byte chunks per row
    static constexpr int kTile = kPfKeys * D * 2;          // K (or V) of one tile
    static constexpr int kBuf = 2 * kTile;                 // K and V
    static constexpr int kSmem = 2 * kBuf + 2 * kPfKeys * 4 + 2 * kPfKeys * 8;   // two buffers, row flags, row sources
    static constexpr int kKsteps = D / 16;
    static constexpr int kNt = D / 8;                      // output 8-column tiles
};

// Byte offset of 16-byte chunk ch of row r in a swizzled tile (rows of D * 2
// bytes; the chunk index's low three bits are xor-ed with the row's).
template <int D>
__device__ __forceinline__ int pf_off(int r, int ch) {
    return r * (D * 2) + ((ch ^ (r & 7)) << 4);
}

__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst_smem)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Three CTAs per SM (168 registers a thread): measured 163 -> 169 TFLOP/s on
// ring chunks, 185 -> 236 on the paged batch, against two at 173 registers.
// READ: read-time RoPE (a separate instance, so the none/baked kernel carries
// none of its code or registers).
template <int D, bool READ>
__global__ void __launch_bounds__(kPfThreads, 3) prefill_kernel(const __grid_constant__ PrefillParams p) {
    using S = PfShape<D>;
    extern __shared__ __align__(128) unsigned char pf_smem[];
    int* rowok = reinterpret_cast<int*>(pf_smem + 2 * S::kBuf);      // [2][kPfKeys]
    // each key row's source, per buffer: element offset of its K row in the
    // cache (>= 0), -(offset of its staged row) - 2, or -1 (no row)
    long long* rowsrc = reinterpret_cast<long long*>(pf_smem + 2 * S::kBuf + 2 * kPfKeys * 4);   // [2][kPfKeys]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    const int h = blockIdx.y, b = blockIdx.z;
    const int G = p.G;
    const int tq = kPfRows / G;                       // tokens per CTA
    const int i0 = blockIdx.x * tq;
    const int pos0 = p.pos0[b];
    const int C = p.capacity;

    // this lane's two rows (g and g + 8 of the warp's 16): token, q head, position
    int row_i[2], row_t[2], row_h[2];
    bool row_ok[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int R = warp * 16 + g + 8 * e;
        const int tl = R / G;
        row_i[e] = i0 + tl;
        row_h[e] = h * G + R % G;
        row_t[e] = pos0 + row_i[e];
        row_ok[e] = tl < tq && row_i[e] < p.T;
    }
    // the CTA's positions: first and last of its tokens (left padding clipped)
    const int i_last = min(i0 + tq, p.T) - 1;
    const int t_hi = pos0 + i_last;
    const int t_lo = max(pos0 + i0, 0);
    // every row of the CTA is a chunk token at a position >= 0 (no padding,
    // no rows past the chunk's end): interior tiles may skip the per-key tests
    const bool all_rows = pos0 + i0 >= 0 && i0 + tq <= p.T;

    // q fragments (A of Q K^T): rows g, g + 8; columns 16 ks + 2c (+1), + 8;
    // rotated (RoPE) at the token's position t, or at min(t, C - 1) for the
    // sink keys of read-time RoPE (sinks_ip), scaled by q_scale, bf16
    constexpr bool read_rope = READ;
    uint32_t qa[S::kKsteps][4];
    auto load_q = [&](bool sinks_ip) {
        float qf[2][S::kKsteps][4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) +
                                        (((long long)b * p.T + (row_ok[e] ? row_i[e] : 0)) * p.Hq + row_h[e]) * D;
#pragma unroll
            for (int ks = 0; ks < S::kKsteps; ++ks) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t w = 0u;
                    if (row_ok[e]) w = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 * hf + 2 * c);
                    qf[e][ks][2 * hf] = __uint_as_float(w << 16);
                    qf[e][ks][2 * hf + 1] = __uint_as_float(w & 0xffff0000u);
                }
            }
            if (p.rope != kRopeNone && row_ok[e] && row_t[e] >= 0) {
                const long long qpos = sinks_ip ? min(row_t[e], C - 1) : row_t[e];
#pragma unroll
                for (int ks = 0; ks < S::kKsteps / 2; ++ks) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int i = 16 * ks + 8 * (k >> 1) + 2 * c + (k & 1);
                        float cs, sn;
                        rope_cos_sin(qpos, p.theta[i], &cs, &sn);
                        const float x1 = qf[e][ks][k], x2 = qf[e][ks + S::kKsteps / 2][k];
                        qf[e][ks][k] = x1 * cs - x2 * sn;
                        qf[e][ks + S::kKsteps / 2][k] = x1 * sn + x2 * cs;
                    }
                }
            }
        }
#pragma unroll
        for (int ks = 0; ks < S::kKsteps; ++ks) {
            qa[ks][0] = pack_bf16x2(qf[0][ks][0] * p.q_scale, qf[0][ks][1] * p.q_scale);
            qa[ks][1] = pack_bf16x2(qf[1][ks][0] * p.q_scale, qf[1][ks][1] * p.q_scale);
            qa[ks][2] = pack_bf16x2(qf[0][ks][2] * p.q_scale, qf[0][ks][3] * p.q_scale);
            qa[ks][3] = pack_bf16x2(qf[1][ks][2] * p.q_scale, qf[1][ks][3] * p.q_scale);
        }
    };

    // key ranges: window layouts [0, min(S, t_hi + 1)) and [max(S, t_lo - W + 1), t_hi];
    // paged [0, t_hi]
    const bool paged = p.layout == kPaged;
    int r0b = 0, r0e = 0, r1b = 0, r1e = 0;
    if (i_last >= i0 && t_hi >= 0) {
        if (paged) {
            r1b = 0;
            r1e = t_hi + 1;
        } else {
            r0e = min(p.sinks, t_hi + 1);
            r1b = max(p.sinks, t_lo - p.window + 1);
            r1e = t_hi + 1;
        }
    }
    const int n0 = (r0e - r0b + kPfKeys - 1) / kPfKeys;
    // read-time RoPE: a window key at distance t - p from the query, a sink key
    // at min(t, C - 1) - p ([sink] "RoPE cache position shifting"): keys are
    // rotated at their own positions in shared memory, the query at t, or at
    // min(t, C - 1) for the sink tiles, which come first
    load_q(read_rope && n0 > 0);
    const int ntiles = n0 + (r1e > r1b ? (r1e - r1b + kPfKeys - 1) / kPfKeys : 0);
    auto tile_base = [&](int k) { return k < n0 ? r0b + k * kPfKeys : r1b + (k - n0) * kPfKeys; };
    auto tile_end = [&](int k) { return k < n0 ? r0e : r1e; };

    const long long unit = (long long)b * p.Hkv + h;
    const __nv_bfloat16* cache = static_cast<const __nv_bfloat16*>(p.cache);
    const __nv_bfloat16* kst = static_cast<const __nv_bfloat16*>(p.kst);
    const __nv_bfloat16* vst = static_cast<const __nv_bfloat16*>(p.vst);

    // gather tile k into buffer k & 1: first one thread per key row finds the
    // row's source; then thread tid copies chunk tid % kChunks of rows
    // tid / kChunks + n * (128 / kChunks)
    auto load_tile = [&](int k) {
        unsigned char* Kb = pf_smem + (k & 1) * S::kBuf;
        unsigned char* Vb = Kb + S::kTile;
        int* ok = rowok + (k & 1) * kPfKeys;
        long long* src = rowsrc + (k & 1) * kPfKeys;
        if (tid < kPfKeys) {
            const int r = tid;
            const int pk = tile_base(k) + r;
            long long sv = -1;
            bool good = pk < tile_end(k) && pk >= 0;
            if (good && paged) {
                const int lb = pk / p.bs;
                int phys = lb < p.maxb ? p.table[(long long)b * p.maxb + lb] : -1;
                if (phys >= p.num_blocks) {
                    set_error(p.err, 0x1u /* KVC_DEV_BAD_BLOCK */);
                    phys = -1;
                }
                good = phys >= 0 && (!p.valid || ((p.valid[phys >> 5] >> (phys & 31)) & 1u));
                if (good && pk < pos0) sv = p.layer_off + (((long long)phys * p.Hkv + h) * p.bs + pk % p.bs) * D;
            } else if (good && pk < pos0) {
                const int slot = pk < p.sinks ? pk : p.sinks + (int)((unsigned)(pk - p.sinks) % (unsigned)p.window);
                sv = p.layer_off + (unit * C + slot) * D;
            }
            if (good && pk >= pos0)                      // a row of the chunk itself
                sv = -((((long long)b * p.T + (pk - pos0)) * p.Hkv + h) * D) - 2;
            src[r] = good ? sv : -1;
            ok[r] = good ? 1 : 0;
        }
        __syncthreads();
        constexpr int kRowsPerPass = kPfThreads / S::kChunks;
        const int ch = tid % S::kChunks;
        for (int r = tid / S::kChunks; r < kPfKeys; r += kRowsPerPass) {
            const long long sv = src[r];
            if (sv == -1) {
                *reinterpret_cast<uint4*>(Kb + pf_off<D>(r, ch)) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(Vb + pf_off<D>(r, ch)) = make_uint4(0u, 0u, 0u, 0u);
            } else {
                const __nv_bfloat16* ks = sv >= 0 ? cache + sv : kst + (-sv - 2);
                const __nv_bfloat16* vs = sv >= 0 ? ks + p.kv_off : vst + (-sv - 2);
                cp_async16(Kb + pf_off<D>(r, ch), ks + ch * 8);
                cp_async16(Vb + pf_off<D>(r, ch), vs + ch * 8);
            }
        }
    };

    float o[S::kNt][4];
#pragma unroll
    for (int n = 0; n < S::kNt; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    if (ntiles > 0) load_tile(0);
    cp_async_commit();
    for (int k = 0; k < ntiles; ++k) {
        if (k + 1 < ntiles) load_tile(k + 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const unsigned char* Kb = pf_smem + (k & 1) * S::kBuf;
        const unsigned char* Vb = Kb + S::kTile;
        const int* ok = rowok + (k & 1) * kPfKeys;
        const int base = tile_base(k);
        if constexpr (READ) {
            if (k == n0 && n0 > 0) load_q(false);      // past the sink tiles: q at t
            // rotate the raw K rows of the tile at their positions base + r: thread
            // tid takes rotation pair i = tid % (D/2) of rows r0 .. r0 + kRun - 1,
            // one exact angle, then the step R(theta_i) from row to row
            constexpr int HALF = D / 2, kRun = kPfKeys * HALF / kPfThreads;
            const int i = tid % HALF, r0 = (tid / HALF) * kRun;
            float c0, s0, cst, sst;
            rope_cos_sin((long long)(base + r0), p.theta[i], &c0, &s0);
            rope_cos_sin(1, p.theta[i], &cst, &sst);
            unsigned char* Kw = const_cast<unsigned char*>(Kb);
            for (int r = r0; r < r0 + kRun; ++r) {
                __nv_bfloat16* lo = reinterpret_cast<__nv_bfloat16*>(Kw + pf_off<D>(r, i >> 3) + (i & 7) * 2);
                __nv_bfloat16* hi = reinterpret_cast<__nv_bfloat16*>(Kw + pf_off<D>(r, (i + HALF) >> 3) + (i & 7) * 2);
                const float x1 = __bfloat162float(*lo), x2 = __bfloat162float(*hi);
                *lo = __float2bfloat16_rn(x1 * c0 - x2 * s0);
                *hi = __float2bfloat16_rn(x1 * s0 + x2 * c0);
                const float cn = c0 * cst - s0 * sst;
                s0 = s0 * cst + c0 * sst;
                c0 = cn;
            }
            __syncthreads();
        }

        // ---- S = Q K^T: 16 rows x 64 keys (8 n-tiles) -----------------------
        float s[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
        {
            const int tok = ((lane >> 4) << 3) + (lane & 7);
            const int chs = (lane >> 3) & 1;
#pragma unroll
            for (int ks = 0; ks < S::kKsteps; ++ks) {
#pragma unroll
                for (int jp = 0; jp < 4; ++jp) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(smem_u32(Kb + pf_off<D>(16 * jp + tok, 2 * ks + chs)), b0, b1, b2, b3);
                    mma_bf16_16816(s[2 * jp], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                    mma_bf16_16816(s[2 * jp + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
                }
            }
        }

        // ---- masks, online softmax per row ----------------------------------
        // A tile inside every row's window and below every row's position needs
        // no per-key test (window layouts), or only the keys' own validity (paged)
        const bool interior = all_rows && k >= n0 && base + kPfKeys <= r1e && base + kPfKeys - 1 <= t_lo &&
                              (paged || base >= t_hi - p.window + 1);
#pragma unroll
        for (int e = 0; e < 2; ++e) {              // row g (e = 0), g + 8 (e = 1)
            const int t = row_t[e];
            float mx = -INFINITY;
            if (interior) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        float& v = s[j][2 * e + u];
                        if (paged && !ok[8 * j + 2 * c + u]) v = -INFINITY;
                        mx = fmaxf(mx, v);
                    }
                }
            } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int col = 8 * j + 2 * c + u;
                    const int pk = base + col;
                    bool allowed = row_ok[e] && ok[col] && pk <= t;
                    if (!paged) allowed = allowed && (pk < p.sinks || pk > t - p.window);
                    float& v = s[j][2 * e + u];
                    v = allowed ? v : -INFINITY;
                    mx = fmaxf(mx, v);
                }
            }
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mn = fmaxf(m_run[e], mx);
            const float alpha = (mn == -INFINITY || mn == m_run[e]) ? 1.f : exp2f(m_run[e] - mn);
            float ls = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    float& v = s[j][2 * e + u];
                    v = (v == -INFINITY) ? 0.f : exp2f(v - mn);
                    ls += v;
                }
            }
            l_run[e] = l_run[e] * alpha + ls;
            m_run[e] = mn;
            if (alpha != 1.f) {
#pragma unroll
                for (int n = 0; n < S::kNt; ++n) {
                    o[n][2 * e] *= alpha;
                    o[n][2 * e + 1] *= alpha;
                }
            }
        }

        // ---- O += P V: 4 k-steps of 16 keys ---------------------------------
        {
            const int tok = (((lane >> 3) & 1) << 3) + (lane & 7);
            const int chs = lane >> 4;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t a0 = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
                const uint32_t a1 = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
                const uint32_t a2 = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
                const uint32_t a3 = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
                for (int jp = 0; jp < S::kNt / 2; ++jp) {
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_trans(smem_u32(Vb + pf_off<D>(16 * kk + tok, 2 * jp + chs)), v0, v1, v2, v3);
                    mma_bf16_16816(o[2 * jp], a0, a1, a2, a3, v0, v1);
                    mma_bf16_16816(o[2 * jp + 1], a0, a1, a2, a3, v2, v3);
                }
            }
        }
        __syncthreads();           // the buffer is refilled by the next iteration's load
    }
    cp_async_wait<0>();

    // ---- normalise and write -----------------------------------------------
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        float l = l_run[e];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        if (!row_ok[e]) continue;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) +
                             (((long long)b * p.T + row_i[e]) * p.Hq + row_h[e]) * D + 2 * c;
#pragma unroll
        for (int n = 0; n < S::kNt; ++n)
            *reinterpret_cast<uint32_t*>(dst + 8 * n) = pack_bf16x2(o[n][2 * e] * inv, o[n][2 * e + 1] * inv);
    }
}

template <int D, bool READ>
cudaError_t launch_prefill_t(const PrefillParams& p, cudaStream_t stream) {
    using S = PfShape<D>;
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_relaxed) & bit)) {
        e = cudaFuncSetAttribute(prefill_kernel<D, READ>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmem);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_relaxed);
    }
    const int tq = kPfRows / p.G;
    dim3 grid((p.T + tq - 1) / tq, p.Hkv, p.B);
    prefill_kernel<D, READ><<<grid, kPfThreads, S::kSmem, stream>>>(p);
    return cudaGetLastError();
}

// head_dim 128 runs on the tcgen05 kernel (kvc_prefill_tc.cu), head_dim 64 here.
cudaError_t launch_prefill(int head_dim, int g, const PrefillParams& p, cudaStream_t stream) {
    if (g < 1 || g > kPfRows) return cudaErrorInvalidValue;
    const bool read = p.rope == kRopeRead;
    if (head_dim == 64) return read ? launch_prefill_t<64, true>(p, stream) : launch_prefill_t<64, false>(p, stream);
    if (head_dim == 128) return launch_prefill_tc(p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace kvc
