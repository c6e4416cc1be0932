// Chunked prefill attention at head_dim 128 on the fifth-generation tensor
// cores (tcgen05): the same operation as prefill_kernel ([pool] chunked
// prefill; [ring] 3.1 and 5.2, the window as a mask on the score matrix), with
// both products issued as tcgen05.mma and accumulated in tensor memory.
//
// One CTA: 128 (token, q head) rows of one kv head of one sequence -- 128 / G
// tokens times the G q heads of the group -- one thread and one TMEM lane per
// row.  Shared memory holds Q (rotated, scaled, bf16) and two buffers of
// 64-key K and V tiles, gathered row by row with cp.async (ring slots, sinks,
// paged blocks, staged chunk rows).  Every operand tile is stored in 64-column
// blocks of 128-byte rows, 16-byte chunks xor-swizzled by the row's low three
// bits (the 128-byte swizzle of the tensor-core shared-memory descriptors).
// Per tile:
//   S  = Q K^T       tcgen05.mma M=128 N=64 K=128 into TMEM columns 128..191
//   softmax          each thread loads its row of S (tcgen05.ld), masks it,
//                    updates its running max and sum (base 2) and writes its
//                    bf16 probabilities over the K tile, which S no longer needs
//   O  = O a + P V   O lives in TMEM columns 0..127; a row is rescaled in place
//                    (tcgen05.ld / st) only when its reference max moved (by
//                    more than 8 in base 2); P V is tcgen05.mma M=128 N=128
//                    K=64, V as an N-major operand
// Completion of each product is tracked by an mbarrier (tcgen05.commit); every
// wait is bounded and the decision to stop is taken by the whole CTA.
#include "kvc_decode.cuh"

namespace kvc {

namespace {

constexpr int kTcRows = 128;       // (token, q head) rows per CTA = threads = TMEM lanes
constexpr int kTcKeys = 64;        // keys per tile
constexpr int kTcD = 128;          // head_dim of this kernel
constexpr int kTcThreads = 128;

constexpr int kTcQ = kTcRows * kTcD * 2;            // Q tile (32 KiB)
constexpr int kTcKV = kTcKeys * kTcD * 2;           // K (or V) tile (16 KiB)
constexpr int kTcP = kTcRows * kTcKeys * 2;         // P tile (16 KiB), written over the K tile
static_assert(kTcP == kTcKV, "P is written over the K tile it was computed from");
constexpr int kTcOffBuf = kTcQ;                     // buffer j: K at kTcOffBuf + 2 j kTcKV, V after it
constexpr int kTcOffMeta = kTcOffBuf + 2 * 2 * kTcKV;
// meta: rowok [2][64] int, rowsrc [2][64] long long, two mbarriers, TMEM address
constexpr int kTcMeta = 2 * kTcKeys * 4 + 2 * kTcKeys * 8 + 2 * 8 + 16;
constexpr int kTcSmem = kTcOffMeta + kTcMeta + 1024;   // + room to align the base to 1024 bytes
constexpr int kTcOCol = 0;                          // O: TMEM columns [0, 128)
constexpr int kTcSCol = 128;                        // S: TMEM columns [128, 192)
constexpr int kTcTmemCols = 256;
constexpr float kTcLazy = 8.f;                      // lazy rescale threshold (log2 units)
// two CTAs fit an SM by shared memory (228 KiB, 1 KiB reserved per CTA) and
// three do not, so the CTAs of one SM never ask for more than its 512 columns
static_assert(2 * (kTcSmem + 1024) <= 228 * 1024 && 3 * (kTcSmem + 1024) > 228 * 1024, "occupancy");
static_assert(2 * kTcTmemCols <= 512, "TMEM columns of the resident CTAs");

// Byte offset of 16-byte chunk ch (of kTcD / 8) of row r in a tile of R rows.
template <int R>
__device__ __forceinline__ int tc_off(int r, int ch) {
    return (ch >> 3) * (R * 128) + r * 128 + (((ch ^ r) & 7) << 4);
}

// Shared-memory matrix descriptor: start, leading and stride byte offsets
// (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t tc_sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: f32 accumulator, bf16 A and B, A
// K-major, B K-major (0) or N-major (1), N / 8 and M / 16.
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N, int b_n_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_n_major << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive 32-bit TMEM columns of this thread's lane (its warp's 32 lanes)
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tc_cp_async16(void* dst_smem, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst_smem)), "l"(src) : "memory");
}
__device__ __forceinline__ void tc_cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void tc_cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

}  // namespace

template <bool READ>
__global__ void __launch_bounds__(kTcThreads, 2) prefill_tc_kernel(const __grid_constant__ PrefillParams p) {
    constexpr int D = kTcD;
    extern __shared__ unsigned char tc_raw[];
    const uint32_t raw_u = smem_u32(tc_raw);
    unsigned char* sm = tc_raw + (((raw_u + 1023u) & ~1023u) - raw_u);
    const uint32_t sm_u = smem_u32(sm);
    unsigned char* Qs = sm;
    int* rowok = reinterpret_cast<int*>(sm + kTcOffMeta);                                    // [2][64]
    // each key row's source, per buffer: element offset of its K row in the
    // cache (>= 0), -(offset of its staged row) - 2, or -1 (no row)
    long long* rowsrc = reinterpret_cast<long long*>(sm + kTcOffMeta + 2 * kTcKeys * 4);     // [2][64]
    uint64_t* bar_s = reinterpret_cast<uint64_t*>(sm + kTcOffMeta + 2 * kTcKeys * 12);
    uint64_t* bar_o = bar_s + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_s + 2);

    const int tid = threadIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    const int G = p.G;
    const int tq = kTcRows / G;                       // tokens per CTA
    const int i0 = blockIdx.x * tq;
    const int pos0 = p.pos0[b];
    const int C = p.capacity;

    // this thread's row: token, q head, position
    const int tl = tid / G;
    const int row_i = i0 + tl;
    const int row_h = h * G + tid % G;
    const int row_t = pos0 + row_i;
    const bool row_ok = tl < tq && row_i < p.T;
    const int i_last = min(i0 + tq, p.T) - 1;
    const int t_hi = pos0 + i_last;
    const int t_lo = max(pos0 + i0, 0);
    const bool all_rows = pos0 + i0 >= 0 && i0 + tq <= p.T;

    if (tid == 0) {
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        mbar_fence_init();
    }
    if (tid < 32) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }

    // Q row of this thread: rotated (RoPE) at t, or at min(t, C - 1) for the
    // sink tiles of read-time RoPE (sinks_ip), scaled by q_scale, bf16
    auto write_q = [&](bool sinks_ip) {
        const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) +
                                    (((long long)b * p.T + (row_ok ? row_i : 0)) * p.Hq + row_h) * D;
        const bool rot = p.rope != kRopeNone && row_ok && row_t >= 0;
        const long long qpos = sinks_ip ? min(row_t, C - 1) : row_t;
#pragma unroll 1
        for (int cb = 0; cb < D / 16; ++cb) {         // chunk cb (elements 8 cb ..) and its rotation partner
            uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
            if (row_ok) {
                lo = *reinterpret_cast<const uint4*>(qrow + 8 * cb);
                hi = *reinterpret_cast<const uint4*>(qrow + D / 2 + 8 * cb);
            }
            const uint32_t lw[4] = {lo.x, lo.y, lo.z, lo.w}, hw[4] = {hi.x, hi.y, hi.z, hi.w};
            uint32_t lo2[4], hi2[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float x[2] = {__uint_as_float(lw[e] << 16), __uint_as_float(lw[e] & 0xffff0000u)};
                float y[2] = {__uint_as_float(hw[e] << 16), __uint_as_float(hw[e] & 0xffff0000u)};
                if (rot) {
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        float cs, sn;
                        rope_cos_sin(qpos, p.theta[8 * cb + 2 * e + u], &cs, &sn);
                        const float x1 = x[u], x2 = y[u];
                        x[u] = x1 * cs - x2 * sn;
                        y[u] = x1 * sn + x2 * cs;
                    }
                }
                lo2[e] = pack_bf16x2(x[0] * p.q_scale, x[1] * p.q_scale);
                hi2[e] = pack_bf16x2(y[0] * p.q_scale, y[1] * p.q_scale);
            }
            *reinterpret_cast<uint4*>(Qs + tc_off<kTcRows>(tid, cb)) = make_uint4(lo2[0], lo2[1], lo2[2], lo2[3]);
            *reinterpret_cast<uint4*>(Qs + tc_off<kTcRows>(tid, cb + D / 16)) =
                make_uint4(hi2[0], hi2[1], hi2[2], hi2[3]);
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
    const int n0 = (r0e - r0b + kTcKeys - 1) / kTcKeys;
    // read-time RoPE: a window key at distance t - p from the query, a sink key
    // at min(t, C - 1) - p ([sink] "RoPE cache position shifting"): keys are
    // rotated at their own positions in shared memory, the query at t, or at
    // min(t, C - 1) for the sink tiles, which come first
    write_q(READ && n0 > 0);
    const int ntiles = n0 + (r1e > r1b ? (r1e - r1b + kTcKeys - 1) / kTcKeys : 0);
    auto tile_base = [&](int k) { return k < n0 ? r0b + k * kTcKeys : r1b + (k - n0) * kTcKeys; };
    auto tile_end = [&](int k) { return k < n0 ? r0e : r1e; };

    const long long unit = (long long)b * p.Hkv + h;
    const __nv_bfloat16* cache = static_cast<const __nv_bfloat16*>(p.cache);
    const __nv_bfloat16* kst = static_cast<const __nv_bfloat16*>(p.kst);
    const __nv_bfloat16* vst = static_cast<const __nv_bfloat16*>(p.vst);

    // gather tile k into buffer k & 1: one thread per key row finds the row's
    // source, then thread tid copies chunk tid % 16 of rows tid / 16 + 8 n
    auto load_tile = [&](int k) {
        unsigned char* Kb = sm + kTcOffBuf + (k & 1) * 2 * kTcKV;
        unsigned char* Vb = Kb + kTcKV;
        int* ok = rowok + (k & 1) * kTcKeys;
        long long* src = rowsrc + (k & 1) * kTcKeys;
        if (tid < kTcKeys) {
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
        constexpr int kChunks = D / 8;
        const int ch = tid % kChunks;
        for (int r = tid / kChunks; r < kTcKeys; r += kTcThreads / kChunks) {
            const long long sv = src[r];
            if (sv == -1) {
                *reinterpret_cast<uint4*>(Kb + tc_off<kTcKeys>(r, ch)) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(Vb + tc_off<kTcKeys>(r, ch)) = make_uint4(0u, 0u, 0u, 0u);
            } else {
                const __nv_bfloat16* ks = sv >= 0 ? cache + sv : kst + (-sv - 2);
                const __nv_bfloat16* vs = sv >= 0 ? ks + p.kv_off : vst + (-sv - 2);
                tc_cp_async16(Kb + tc_off<kTcKeys>(r, ch), ks + ch * 8);
                tc_cp_async16(Vb + tc_off<kTcKeys>(r, ch), vs + ch * 8);
            }
        }
    };

    if (ntiles > 0) load_tile(0);
    tc_cp_async_commit();
    if (ntiles > 1) load_tile(1);
    tc_cp_async_commit();

    tc_fence_before();
    __syncthreads();                                  // barriers initialised, TMEM address written
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = tmem + ((uint32_t)(tid & ~31) << 16);   // this warp's 32 lanes

    constexpr uint32_t kIdescS = tc_idesc(kTcRows, kTcKeys, 0);
    constexpr uint32_t kIdescO = tc_idesc(kTcRows, kTcD, 1);
    float m_run = -INFINITY, l_run = 0.f;
    int issued_s = -1, issued_o = -1;                 // last tile whose S / P V was issued
    bool dead = false;

    for (int k = 0; k < ntiles; ++k) {
        tc_cp_async_wait_all();                       // tile k (the only group that can be pending)
        fence_proxy_async_smem();                     // visible to the tensor cores' reads
        __syncthreads();
        unsigned char* Kb = sm + kTcOffBuf + (k & 1) * 2 * kTcKV;
        const int* ok = rowok + (k & 1) * kTcKeys;
        const int base = tile_base(k);
        if constexpr (READ) {
            if (k == n0 && n0 > 0) write_q(false);   // past the sink tiles: q at t (S of the last sink tile is done)
            // rotate the raw K rows of the tile at their positions base + r: thread
            // tid takes rotation pair i = tid % (D/2) of rows r0 .. r0 + kRun - 1,
            // one exact angle, then the step R(theta_i) from row to row
            constexpr int HALF = D / 2, kRun = kTcKeys * HALF / kTcThreads;
            const int i = tid % HALF, r0 = (tid / HALF) * kRun;
            float c0, s0, cst, sst;
            rope_cos_sin((long long)(base + r0), p.theta[i], &c0, &s0);
            rope_cos_sin(1, p.theta[i], &cst, &sst);
            for (int r = r0; r < r0 + kRun; ++r) {
                __nv_bfloat16* lo = reinterpret_cast<__nv_bfloat16*>(Kb + tc_off<kTcKeys>(r, i >> 3) + (i & 7) * 2);
                __nv_bfloat16* hi =
                    reinterpret_cast<__nv_bfloat16*>(Kb + tc_off<kTcKeys>(r, (i + HALF) >> 3) + (i & 7) * 2);
                const float x1 = __bfloat162float(*lo), x2 = __bfloat162float(*hi);
                *lo = __float2bfloat16_rn(x1 * c0 - x2 * s0);
                *hi = __float2bfloat16_rn(x1 * s0 + x2 * c0);
                const float cn = c0 * cst - s0 * sst;
                s0 = s0 * cst + c0 * sst;
                c0 = cn;
            }
            fence_proxy_async_smem();
            __syncthreads();
        }

        // ---- S = Q K^T (M 128, N 64, K 128: eight steps of 16) ---------------
        if (tid == 0) {
            tc_fence_after();
            const uint32_t kb_u = sm_u + kTcOffBuf + (k & 1) * 2 * kTcKV;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t within = (ks & 3) * 32;
                tc_mma(tmem + kTcSCol, tc_sdesc(sm_u + (ks >> 2) * (kTcRows * 128) + within, 16, 1024),
                       tc_sdesc(kb_u + (ks >> 2) * (kTcKeys * 128) + within, 16, 1024), kIdescS, ks > 0);
            }
            tc_commit(bar_s);
        }
        issued_s = k;
        // P V of tile k - 1 (queued before S) completes first: O may be rescaled
        // below, and buffer (k + 1) & 1 (tile k - 1's K/P and V) takes tile k + 1
        // now, while S, the softmax and P V of tile k run
        if (k > 0) {
            if (__syncthreads_or(!mbar_wait(bar_o, (k - 1) & 1))) {
                dead = true;
                break;
            }
            tc_fence_after();
            if (k + 1 < ntiles) load_tile(k + 1);
            tc_cp_async_commit();
        }
        if (__syncthreads_or(!mbar_wait(bar_s, k & 1))) {
            dead = true;
            break;
        }
        tc_fence_after();
        float s[kTcKeys];
        tc_ld32(lane_base + kTcSCol, s);
        tc_ld32(lane_base + kTcSCol + 32, s + 32);
        tc_wait_ld();

        // ---- masks, online softmax of this thread's row ----------------------
        // a tile inside every row's window and below every row's position needs
        // no per-key test (window layouts), or only the keys' own validity (paged)
        const bool interior = all_rows && k >= n0 && base + kTcKeys <= r1e && base + kTcKeys - 1 <= t_lo &&
                              (paged || base >= t_hi - p.window + 1);
        float mx = -INFINITY;
        if (interior) {
#pragma unroll
            for (int j = 0; j < kTcKeys; ++j) {
                if (paged && !ok[j]) s[j] = -INFINITY;
                mx = fmaxf(mx, s[j]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < kTcKeys; ++j) {
                const int pk = base + j;
                bool allowed = row_ok && ok[j] && pk <= row_t;
                if (!paged) allowed = allowed && (pk < p.sinks || pk > row_t - p.window);
                s[j] = allowed ? s[j] : -INFINITY;
                mx = fmaxf(mx, s[j]);
            }
        }
        // the row's reference max moves only when the tile's max exceeds it by
        // more than kTcLazy (base 2): probabilities stay below 2^kTcLazy, and O
        // and l share the reference, so the result is unchanged while most
        // tiles skip the rescale of O
        float mn = m_run, alpha = 1.f;
        if (mx > m_run + kTcLazy) {
            mn = mx;
            alpha = m_run == -INFINITY ? 1.f : exp2f(m_run - mn);   // no attended key yet: O's row is zero
        }
        float ls = 0.f;
#pragma unroll
        for (int j = 0; j < kTcKeys; ++j) {
            s[j] = (s[j] == -INFINITY) ? 0.f : exp2f(s[j] - mn);
            ls += s[j];
        }
        l_run = l_run * alpha + ls;
        m_run = mn;

        if (k > 0) {
            // tcgen05.ld / st are warp-wide: a warp rescales when any of its rows
            // needs it (alpha is 1 for the others)
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    float ov[32];
                    tc_ld32(lane_base + kTcOCol + 32 * c4, ov);
                    tc_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) ov[j] *= alpha;
                    tc_st32(lane_base + kTcOCol + 32 * c4, ov);
                }
                tc_wait_st();
            }
        }

        // P (bf16) over the K tile: row tid, 64 keys = 8 chunks of 16 bytes
#pragma unroll
        for (int ch = 0; ch < kTcKeys / 8; ++ch) {
            const uint4 w = make_uint4(pack_bf16x2(s[8 * ch], s[8 * ch + 1]), pack_bf16x2(s[8 * ch + 2], s[8 * ch + 3]),
                                       pack_bf16x2(s[8 * ch + 4], s[8 * ch + 5]),
                                       pack_bf16x2(s[8 * ch + 6], s[8 * ch + 7]));
            *reinterpret_cast<uint4*>(Kb + tc_off<kTcRows>(tid, ch)) = w;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- O += P V (M 128, N 128, K 64: four steps of 16 keys) -----------
        if (tid == 0) {
            tc_fence_after();
            const uint32_t p_u = sm_u + kTcOffBuf + (k & 1) * 2 * kTcKV;
            const uint32_t v_u = p_u + kTcKV;
#pragma unroll
            for (int ks = 0; ks < kTcKeys / 16; ++ks)
                tc_mma(tmem + kTcOCol, tc_sdesc(p_u + ks * 32, 16, 1024),
                       tc_sdesc(v_u + ks * 16 * 128, kTcKeys * 128, 1024), kIdescO, (k > 0 || ks > 0));
            tc_commit(bar_o);
        }
        issued_o = k;
    }

    // ---- normalise and write ---------------------------------------------------
    bool have_o = false;
    if (!dead && ntiles > 0) {
        if (__syncthreads_or(!mbar_wait(bar_o, (ntiles - 1) & 1)))
            dead = true;
        else
            have_o = true;
    }
    if (dead) {
        // a product did not complete in time: report it, and give the ones in
        // flight one more bounded wait before the columns are freed
        if (tid == 0) set_error(p.err, 0x8u /* KVC_DEV_TIMEOUT */);
        if (issued_s >= 0) mbar_wait(bar_s, issued_s & 1);
        if (issued_o >= 0) mbar_wait(bar_o, issued_o & 1);
    }
    tc_cp_async_wait_all();
    tc_fence_after();
    if (!dead) {                                      // uniform: every thread takes part in the warp-wide loads
        const float inv = (have_o && l_run > 0.f) ? 1.f / l_run : 0.f;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + (((long long)b * p.T + row_i) * p.Hq + row_h) * D;
#pragma unroll 1
        for (int c4 = 0; c4 < D / 32; ++c4) {
            float ov[32];
            if (have_o) {
                tc_ld32(lane_base + kTcOCol + 32 * c4, ov);
                tc_wait_ld();
            }
            if (row_ok) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = have_o ? pack_bf16x2(ov[8 * q + 2 * e] * inv, ov[8 * q + 2 * e + 1] * inv) : 0u;
                    *reinterpret_cast<uint4*>(dst + 32 * c4 + 8 * q) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid < 32)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols)
                     : "memory");
}

template <bool READ>
static cudaError_t launch_prefill_tc_t(const PrefillParams& p, cudaStream_t stream) {
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_relaxed) & bit)) {
        e = cudaFuncSetAttribute(prefill_tc_kernel<READ>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_relaxed);
    }
    const int tq = kTcRows / p.G;
    dim3 grid((p.T + tq - 1) / tq, p.Hkv, p.B);
    prefill_tc_kernel<READ><<<grid, kTcThreads, kTcSmem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_prefill_tc(const PrefillParams& p, cudaStream_t stream) {
    if (p.G < 1 || p.G > kTcRows) return cudaErrorInvalidValue;
    return p.rope == kRopeRead ? launch_prefill_tc_t<true>(p, stream) : launch_prefill_tc_t<false>(p, stream);
}

}  // namespace kvc
