// Chunked prefill attention on the tcgen05 tensor cores, warp-specialised
// ([pool] chunked prefill of 128-256 tokens; [ring] 3.1 and 5.2, the window as
// a mask on the score matrix; [sink] "RoPE cache position shifting").
//
// One CTA per SM: NQ tiles of 128 (token, q head) rows of one kv head of one
// sequence (NQ = 2 for head_dim 64 and 128, 1 for 256), one TMEM lane per row.
// Roles (warps):
//   0      producer: cuts the keys into 64-row tiles and loads each by TMA into
//          a ring of shared-memory stages ([column block][K|V][64 rows][128 B],
//          128-byte swizzle).  Ring and sink+ring caches are cut in slot space
//          (64 consecutive slots, one box), each slot holding the position it
//          had after position pos0 - 1; paged caches in blocks (the mapped and
//          valid blocks, packed 64 / bs to a tile); then the chunk's own rows
//          from the staged copy, 64 tokens to a tile.  It records each row's
//          position (-1: no key).
//   1      issues every tcgen05.mma (one thread):  S_i = Q_i K^T  into one of
//          two S buffers per Q tile, then O_i += P_i V; S of tile j + 1 is
//          issued before P V of tile j, so the softmax of one tile overlaps the
//          products of the next.
//   2-3    fix-up: zero the V rows of absent keys (they may hold anything) and,
//          for read-time RoPE, rotate the raw K rows at their positions.
//   4-7    softmax of Q tile 0 (one thread per row): masks (window, sinks,
//   (8-11)  causal), online softmax in base 2 with a lazy reference max (moved
//          only when a tile's max exceeds it by more than 8: probabilities stay
//          below 2^8), bf16 P into shared memory, O rescaled in TMEM when the
//          reference moved; at the end O / l to the output.
// Every wait is bounded (~1 s); a timeout sets KVC_DEV_TIMEOUT and every role
// stops; the CTA waits for its copies and products before freeing TMEM.
#include <atomic>

#include "kvc_decode.cuh"

namespace kvc {

namespace {

constexpr int kWsKeys = 64;                 // keys per tile
constexpr int kWsRows = 128;                // rows per Q tile (TMEM lanes)
constexpr int kWsSoftmax0 = 4;              // first softmax warp
constexpr float kWsLazy = 8.f;

enum : int { kTileSlot = 0, kTileSink = 1, kTileBlocks = 2, kTileStage = 3, kTileEnd = 4 };

template <int D>
struct WsShape {
    static constexpr int NQ = D == 256 ? 1 : 2;
    static constexpr int STAGES = D == 64 ? 4 : (D == 128 ? 4 : 2);
    static constexpr int CB = D / 64;                          // 64-column blocks of a row
    static constexpr int QBytes = kWsRows * D * 2;             // one Q tile
    static constexpr int KVBlock = 2 * kWsKeys * 128;          // one column block of K and V
    static constexpr int StageBytes = CB * KVBlock;            // K and V of 64 keys
    static constexpr int OffQ = 0;
    static constexpr int OffStage = OffQ + NQ * QBytes;
    static constexpr int OffP = OffStage + STAGES * StageBytes;   // (P lives in tensor memory)
    // INT8 caches: row scales of each stage's cache tile, [stage][K|V][68]:
    // copied from a row that is a multiple of 4 (whole 16-byte copies), the
    // tile's first row sc_off after it
    static constexpr int ScRows = kWsKeys + 4;
    static constexpr int OffScale = OffP;
    static constexpr int OffMeta = OffScale + STAGES * 2 * ScRows * 4;
    static constexpr int TmemCols = 512;
    static constexpr int SCol0 = NQ * D;                       // S buffers after the O tiles
    static_assert(NQ * D + NQ * 2 * kWsKeys <= TmemCols, "TMEM columns");
    // 4 control warps, then 4 softmax warps per Q tile (one thread per row)
    static constexpr int Threads = 32 * (kWsSoftmax0 + 4 * NQ);
};

// How the softmax masks a tile's keys: every key seen by every row of the
// CTA (no test), the chunk's own rows (key k at position kbase + k: a range
// test), or key by key from pos[].
enum : int { kMaskNone = 0, kMaskRange = 1, kMaskKeys = 2 };

struct alignas(16) WsStageMeta {
    int kind;
    int any_absent;          // some row has no key (its V is zeroed)
    int mask;                // kMaskNone / kMaskRange / kMaskKeys
    int kbase;               // kMaskRange: position of key 0
    int sc_off;              // INT8 cache tile: row 0's scale in the stage's scale area
    int pos[kWsKeys];        // position of each row, -1 = none
};

// the barriers follow the stages' records: whole 16-byte records keep them aligned
static_assert(sizeof(WsStageMeta) % 16 == 0, "stage records keep the barriers aligned");

struct WsBars {
    uint64_t full[4], ready[4], empty[4];
    uint64_t s_full[2][2], s_free[2][2], p_full[2], o_done[2], q_ready[2], fin;
    uint64_t fixb;           // INT8 with read-time RoPE: the fix-up threads, between expansion and rotation
    uint32_t tmem;
    int ntiles;              // set when the producer's end marker reaches the MMA thread
    int abort;
};

template <int D>
constexpr int ws_smem_bytes() {
    using S = WsShape<D>;
    return S::OffMeta + S::STAGES * (int)sizeof(WsStageMeta) + (int)sizeof(WsBars) + 1024;
}

// tile offsets inside a stage
__device__ __forceinline__ int ws_off(int r, int ch) {    // K row r, 16-byte chunk ch (of the row's D/8)
    return (ch >> 3) * (2 * kWsKeys * 128) + r * 128 + (((ch ^ r) & 7) << 4);
}

__device__ __forceinline__ uint64_t ws_sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__host__ __device__ constexpr uint32_t ws_idesc(int M, int N, int b_n_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_n_major << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void ws_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// The same with A from tensor memory (a_tmem: lane = row, two 16-bit elements
// along K per 32-bit column).
__device__ __forceinline__ void ws_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void ws_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void ws_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void ws_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void ws_ld32(uint32_t taddr, float* v) {
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

__device__ __forceinline__ void ws_st32(uint32_t taddr, const float* v) {
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

__device__ __forceinline__ void ws_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void ws_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^a and 2^b in one special-function op: the arguments rounded to fp16
// (ex2.approx.f16x2) and the results widened to fp32.  Softmax arguments here
// are <= 8 (the lazy reference max), so fp16 keeps them to 2^-8 or better --
// finer than the bf16 rounding P gets for P V; a masked key's -inf gives 0.
__device__ __forceinline__ float2 ws_ex2_pair(float a, float b) {
    float2 r;
    asm("{\n\t.reg .b32 h;\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.f16x2.f32 h, %3, %2;\n\t"
        "ex2.approx.f16x2 h, h;\n\t"
        "mov.b32 {lo, hi}, h;\n\t"
        "cvt.f32.f16 %0, lo;\n\t"
        "cvt.f32.f16 %1, hi;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a), "f"(b));
    return r;
}

// try_wait with a suspend-time hint: a thread whose phase is not complete
// sleeps until it completes (or the hint, 0.1 ms, runs out) instead of coming
// back to re-issue the test, which would take issue slots from the softmax warps
__device__ __forceinline__ bool ws_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, 100000;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// A bounded wait that also gives up once another role has given up.
__device__ __forceinline__ bool ws_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (ws_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!ws_try_wait(bar, parity)) {
        if (*abort || clock64() - t0 > kWaitCycles) return false;
    }
    return true;
}

}  // namespace

template <int D, bool READ, bool Q8>
__global__ void __launch_bounds__(WsShape<D>::Threads, 1)
    prefill_ws_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ PrefillMaps maps) {
    static_assert(!Q8 || D >= 128, "INT8 rows are whole 128-code boxes");
    using S = WsShape<D>;
    constexpr int NQ = S::NQ, NST = S::STAGES, CB = S::CB;
    extern __shared__ unsigned char ws_raw[];
    const uint32_t raw_u = smem_u32(ws_raw);
    unsigned char* sm = ws_raw + (((raw_u + 1023u) & ~1023u) - raw_u);
    const uint32_t sm_u = smem_u32(sm);
    WsStageMeta* meta = reinterpret_cast<WsStageMeta*>(sm + S::OffMeta);
    WsBars* bars = reinterpret_cast<WsBars*>(sm + S::OffMeta + NST * sizeof(WsStageMeta));
    volatile int* abort = &bars->abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y, b = blockIdx.z;
    const int G = p.G;
    const int tq = kWsRows / G;                      // tokens per Q tile
    const int i0 = blockIdx.x * tq * NQ;             // first token of the CTA
    const int pos0 = p.pos0[b];
    const int C = p.capacity;
    const bool paged = p.layout == kPaged;
    const int i_last = min(i0 + tq * NQ, p.T) - 1;   // last token of the CTA
    const int t_hi = pos0 + i_last;                  // its position
    const int t_lo = max(pos0 + i0, 0);
    const int t0 = pos0 - 1;                         // the cache holds positions <= t0
    // read-time RoPE: sink keys are scored with q at min(t, C - 1), so they form
    // a tile of their own, first (only cached sinks: chunk tokens below C need none)
    const bool sink_tile = READ && !paged && p.sinks > 0 && t0 >= 0 && t_hi >= 0;

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->ready[s], 64);
            mbar_init(&bars->empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            for (int u = 0; u < 2; ++u) {
                mbar_init(&bars->s_full[i][u], 1);
                mbar_init(&bars->s_free[i][u], 4);
            }
            mbar_init(&bars->p_full[i], kWsRows);
            mbar_init(&bars->o_done[i], 1);
            mbar_init(&bars->q_ready[i], kWsRows);
        }
        mbar_init(&bars->fin, 1);
        mbar_init(&bars->fixb, 64);
        bars->ntiles = 0x7fffffff;
        bars->abort = 0;
        mbar_fence_init();
        if (p.layout == kPaged)
            tma_prefetch_desc(&maps.block);
        else
            tma_prefetch_desc(&maps.slot);
        tma_prefetch_desc(&maps.stage);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars->tmem)),
                     "r"(S::TmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    ws_fence_before();
    __syncthreads();
    ws_fence_after();
    const uint32_t tmem = bars->tmem;
    const long long unit = (long long)b * p.Hkv + h;
    // INT8 cache tiles: the codes of 128 columns (hh) of K or V (kv) land in the
    // stage's upper column blocks, 64 rows of 128 bytes, and are expanded in
    // place (see the fix-up role); their row scales go to the scale area
    auto code_at = [&](int s, int hh, int kv) -> unsigned char* {
        return sm + S::OffStage + s * S::StageBytes + (CB / 2 + hh) * S::KVBlock + kv * (kWsKeys * 128);
    };
    float* sc_area = reinterpret_cast<float*>(sm + S::OffScale);
    auto give_up = [&]() {
        if (!*abort) {
            bars->abort = 1;
            set_error(p.err, 0x8u /* KVC_DEV_TIMEOUT */);
        }
    };

    if (warp == 0) {
        // ============================ producer ==============================
        int idx = 0;
        bool ok = true;
        // next stage: wait until the MMA thread is done with its last tile
        auto acquire = [&]() -> int {
            const int s = idx % NST;
            if (idx >= NST && !ws_wait(&bars->empty[s], ((idx / NST) - 1) & 1, abort)) {
                if (lane == 0) give_up();
                ok = false;
            }
            return s;
        };
        auto unit_base = [&]() { return (long long)unit * C; };
        // window layouts: slot tiles.  Slot s holds the latest position <= t0
        // with that slot (p = s for sinks), or none.
        auto slot_pos = [&](int s, bool sinks_only, bool no_sinks) -> int {
            if (s >= C || t0 < 0) return -1;
            if (s < p.sinks) return (no_sinks || s > t0) ? -1 : s;
            if (sinks_only || s > t0) return -1;
            const int q = t0 - (int)((unsigned)(t0 - s) % (unsigned)p.window);
            // window keys any token of the CTA can see
            return q >= t_lo - p.window + 1 ? q : -1;
        };
        auto issue_slot_tile = [&](int slot0, int kind) {
            const int s = acquire();
            if (!ok) return;
            int absent = 0, partial = 0;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = lane + 32 * u;
                const int q = slot_pos(slot0 + r, kind == kTileSink, READ && kind == kTileSlot);
                meta[s].pos[r] = q;
                absent |= q < 0;
                // seen by every row of the CTA: a sink, or in the window of its
                // latest token (every key here is below the chunk's first position)
                partial |= q >= p.sinks && q <= t_hi - p.window;
            }
            absent = __any_sync(0xffffffffu, absent);
            partial = __any_sync(0xffffffffu, partial);
            __syncwarp();
            if (lane == 0) {
                meta[s].kind = kind;
                meta[s].any_absent = absent;
                meta[s].mask = (absent || partial) ? kMaskKeys : kMaskNone;
                unsigned char* dst = sm + S::OffStage + s * S::StageBytes;
                if constexpr (Q8) {
                    // codes by 128-column boxes; scales of the rows inside the half
                    // (a multiple of 4: whole 16-byte copies)
                    const long long urow = unit_base() + slot0, base4 = urow & ~3LL;
                    const int nsc = (int)min((long long)S::ScRows, p.half_rows - base4);   // a multiple of 4
                    meta[s].sc_off = (int)(urow - base4);
                    mbar_expect_tx(&bars->full[s], (uint32_t)(2 * (D / 128) * kWsKeys * 128 + 2 * nsc * 4));
#pragma unroll
                    for (int hh = 0; hh < D / 128; ++hh)
#pragma unroll
                        for (int kv = 0; kv < 2; ++kv)
                            tma_load_4d(code_at(s, hh, kv), &maps.slot, 128 * hh, (int)urow, kv, p.layer, &bars->full[s]);
#pragma unroll
                    for (int kv = 0; kv < 2; ++kv)
                        bulk_load(sc_area + (s * 2 + kv) * S::ScRows, p.scales + p.sc_layer_off + kv * p.sc_kv_off + base4,
                                  (uint32_t)(nsc * 4), &bars->full[s]);
                } else if (maps.slot_whole) {
                    mbar_expect_tx(&bars->full[s], (uint32_t)S::StageBytes);
                    tma_load_5d(dst, &maps.slot, 0, (int)(unit_base() + slot0), 0, p.layer, 0, &bars->full[s]);
                } else {
                    mbar_expect_tx(&bars->full[s], (uint32_t)S::StageBytes);
#pragma unroll
                    for (int cb = 0; cb < CB; ++cb)
                        tma_load_4d(dst + cb * S::KVBlock, &maps.slot, cb * 64, (int)(unit_base() + slot0), 0, p.layer,
                                    &bars->full[s]);
                }
                mbar_arrive(&bars->full[s]);
            }
            ++idx;
        };
        if (t_hi >= 0) {
            if (!paged) {
                if (sink_tile) issue_slot_tile(0, kTileSink);
                // slot tiles with at least one key the CTA can see
                const int nslot = (C + kWsKeys - 1) / kWsKeys;
                for (int k = 0; k < nslot && ok; ++k) {
                    bool any = false;
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        any |= slot_pos(k * kWsKeys + lane + 32 * u, false, READ) >= 0;
                    if (__any_sync(0xffffffffu, any)) issue_slot_tile(k * kWsKeys, kTileSlot);
                }
            } else if (t0 >= 0) {
                // paged: mapped and valid blocks holding positions <= t0, packed
                const int bs = p.bs, per = kWsKeys / bs;
                const int nlb = t0 / bs + 1;
                const int32_t* trow = p.table + (long long)b * p.maxb;
                int fill = 0, s = 0;
                for (int base = 0; base < nlb && ok; base += 32) {
                    const int lb = base + lane;
                    int phys = lb < nlb ? __ldcg(trow + lb) : -1;
                    if (phys >= p.num_blocks) {
                        set_error(p.err, 0x1u /* KVC_DEV_BAD_BLOCK */);
                        phys = -1;
                    }
                    bool att = phys >= 0;
                    if (att && p.valid) att = (__ldcg(p.valid + (phys >> 5)) >> (phys & 31)) & 1u;
                    unsigned m = __ballot_sync(0xffffffffu, att);
                    while (m && ok) {
                        const int src = __ffs(m) - 1;
                        m &= m - 1;
                        const int ph = __shfl_sync(0xffffffffu, phys, src);
                        const int blb = base + src;
                        if (fill == 0) s = acquire();
                        if (!ok) break;
                        if (Q8 && fill == 0 && lane == 0) meta[s].sc_off = 0;   // block rows: multiples of 8
                        // rows of this block: positions blb * bs + r, keys up to t0
                        for (int r = lane; r < bs; r += 32) {
                            const int q = blb * bs + r;
                            meta[s].pos[fill * bs + r] = q <= t0 ? q : -1;
                        }
                        if (lane == 0) {
                            const int row = (int)(((long long)ph * p.Hkv + h) * bs);
                            if constexpr (Q8) {
                                mbar_expect_tx(&bars->full[s], (uint32_t)(2 * (D / 128) * bs * 128 + 2 * bs * 4));
#pragma unroll
                                for (int hh = 0; hh < D / 128; ++hh)
#pragma unroll
                                    for (int kv = 0; kv < 2; ++kv)
                                        tma_load_4d(code_at(s, hh, kv) + fill * bs * 128, &maps.block, 128 * hh, row, kv,
                                                    p.layer, &bars->full[s]);
#pragma unroll
                                for (int kv = 0; kv < 2; ++kv)
                                    bulk_load(sc_area + (s * 2 + kv) * S::ScRows + fill * bs,
                                              p.scales + p.sc_layer_off + kv * p.sc_kv_off + row, (uint32_t)(bs * 4),
                                              &bars->full[s]);
                            } else {
                                mbar_expect_tx(&bars->full[s], (uint32_t)(bs * D * 4));
                                unsigned char* dst = sm + S::OffStage + s * S::StageBytes + fill * bs * 128;
#pragma unroll
                                for (int cb = 0; cb < CB; ++cb)
#pragma unroll
                                    for (int kv = 0; kv < 2; ++kv)
                                        tma_load_4d(dst + cb * S::KVBlock + kv * kWsKeys * 128, &maps.block, cb * 64, row,
                                                    kv, p.layer, &bars->full[s]);
                            }
                        }
                        if (++fill == per) {
                            __syncwarp();
                            if (lane == 0) {
                                meta[s].kind = kTileBlocks;
                                meta[s].any_absent = t0 < blb * bs + bs - 1;   // the last block's rows past t0
                                // every cached key precedes every token of the chunk
                                meta[s].mask = meta[s].any_absent ? kMaskKeys : kMaskNone;
                                mbar_arrive(&bars->full[s]);
                            }
                            fill = 0;
                            ++idx;
                        }
                    }
                }
                if (ok && fill > 0) {
                    // a partial tile: the rest of its rows hold no key, and no copy lands there
                    for (int r = fill * bs + lane; r < kWsKeys; r += 32) meta[s].pos[r] = -1;
                    __syncwarp();
                    if (lane == 0) {
                        meta[s].kind = kTileBlocks;
                        meta[s].any_absent = 1;
                        meta[s].mask = kMaskKeys;
                        mbar_arrive(&bars->full[s]);
                    }
                    ++idx;
                }
            }
            // the chunk's own rows, tokens 0 .. i_last, 64 to a tile
            for (int i_s = 0; i_s <= i_last && ok; i_s += kWsKeys) {
                const int s = acquire();
                if (!ok) break;
                int absent = 0;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int r = lane + 32 * u;
                    const int i = i_s + r;
                    const int q = (i <= i_last && pos0 + i >= 0) ? pos0 + i : -1;
                    meta[s].pos[r] = q;
                    absent |= q < 0;
                }
                absent = __any_sync(0xffffffffu, absent);
                __syncwarp();
                if (lane == 0) {
                    meta[s].kind = kTileStage;
                    meta[s].any_absent = absent;
                    meta[s].mask = kMaskRange;
                    meta[s].kbase = pos0 + i_s;
                    unsigned char* dst = sm + S::OffStage + s * S::StageBytes;
                    mbar_expect_tx(&bars->full[s], (uint32_t)S::StageBytes);
                    tma_load_5d(dst, &maps.stage, 0, h, b * p.T + i_s, 0, 0, &bars->full[s]);
                    mbar_arrive(&bars->full[s]);
                }
                ++idx;
            }
        }
        // end marker
        if (ok) {
            const int s = acquire();
            if (ok && lane == 0) {
                meta[s].kind = kTileEnd;
                mbar_arrive(&bars->full[s]);
            }
            if (ok) ++idx;
        }
        // never leave with copies landing in shared memory
        if (!ok && lane == 0)
            for (int k = (idx > NST ? idx - NST : 0); k < idx; ++k) mbar_wait(&bars->full[k % NST], (k / NST) & 1);
    } else if (warp == 2 || warp == 3) {
        // ============================ fix-up ===============================
        const int ft = tid - 64;                       // 0 .. 63
        uint32_t fix_phase = 0;
        for (int j = 0;; ++j) {
            const int s = j % NST;
            if (!ws_wait(&bars->full[s], (j / NST) & 1, abort)) {
                give_up();
                break;
            }
            const int kind = meta[s].kind;
            unsigned char* st = sm + S::OffStage + s * S::StageBytes;
            if (kind != kTileEnd) {
                bool wrote = false;
                if constexpr (Q8) {
                    if (kind != kTileStage) {
                        // row ft of the cache tile: code x row scale to bf16, in the
                        // stage's K / V layout.  Column boxes go in order: box hh
                        // overwrites (in blocks 2 hh, 2 hh + 1) only this row's codes
                        // of boxes < hh and its own, each already read.
                        const float* scs = sc_area + s * 2 * S::ScRows + meta[s].sc_off;
                        const float scl[2] = {scs[ft], scs[S::ScRows + ft]};
#pragma unroll
                        for (int hh = 0; hh < D / 128; ++hh) {
#pragma unroll
                            for (int kv = 0; kv < 2; ++kv) {
                                const uint4* src = reinterpret_cast<const uint4*>(code_at(s, hh, kv) + ft * 128);
                                uint4 cw[8];
#pragma unroll
                                for (int q = 0; q < 8; ++q) cw[q] = src[q];
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    const uint32_t w4[4] = {cw[q].x, cw[q].y, cw[q].z, cw[q].w};
                                    const float2 sc2 = make_float2(scl[kv], scl[kv]);
#pragma unroll
                                    for (int hf = 0; hf < 2; ++hf) {
                                        uint32_t o[4];
#pragma unroll
                                        for (int e = 0; e < 2; ++e) {
                                            // code c as the fp32 2^23 + (c + 128) (the byte under
                                            // the exponent of 2^23), less 2^23 + 128: exact
                                            const uint32_t x = w4[2 * hf + e] ^ 0x80808080u;
#pragma unroll
                                            for (int h2 = 0; h2 < 2; ++h2) {
                                                float2 f = make_float2(
                                                    __int_as_float(__byte_perm(x, 0x4B000000u, 0x7540u | (uint32_t)(2 * h2))),
                                                    __int_as_float(__byte_perm(x, 0x4B000000u, 0x7540u | (uint32_t)(2 * h2 + 1))));
                                                f = __fmul2_rn(__fadd2_rn(f, make_float2(-8388736.f, -8388736.f)), sc2);
                                                o[2 * e + h2] = pack_bf16x2(f.x, f.y);
                                            }
                                        }
                                        const int ch = 16 * hh + 2 * q + hf;     // 8-column chunk of the row
                                        *reinterpret_cast<uint4*>(st + ws_off(ft, ch) + kv * (kWsKeys * 128)) =
                                            make_uint4(o[0], o[1], o[2], o[3]);
                                    }
                                }
                            }
                        }
                        wrote = true;
                    }
                }
                if (meta[s].any_absent) {
                    // V rows of absent keys to zero: 64 threads, one row each
                    if (meta[s].pos[ft] < 0) {
#pragma unroll
                        for (int cb = 0; cb < CB; ++cb)
#pragma unroll
                            for (int ch = 0; ch < 8; ++ch)
                                *reinterpret_cast<uint4*>(st + cb * S::KVBlock + kWsKeys * 128 + ft * 128 + ch * 16) =
                                    make_uint4(0u, 0u, 0u, 0u);
                    }
                    wrote = true;
                }
                if constexpr (READ && Q8) {
                    // the rotation below reads rows other threads expanded
                    mbar_arrive(&bars->fixb);
                    if (!ws_wait(&bars->fixb, fix_phase & 1, abort)) {
                        give_up();
                        break;
                    }
                    ++fix_phase;
                }
                if constexpr (READ) {
                    // raw K rows rotated at their positions: thread ft takes the
                    // 16-byte chunk pair c (elements 8c .. 8c + 7 and their
                    // partners at + D/2) of rows r0 .. r0 + RUN - 1, in f32x2
                    // pairs; the angles advance by one step from row to row while
                    // positions are consecutive, else are computed afresh
                    constexpr int CP = D / 16, RG = 64 / CP, RUN = kWsKeys / RG;
                    const int c = ft % CP, r0 = (ft / CP) * RUN;
                    float2 cc[4], ss[4], stc[4], sts[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        rope_cos_sin(1, p.theta[8 * c + 2 * u], &stc[u].x, &sts[u].x);
                        rope_cos_sin(1, p.theta[8 * c + 2 * u + 1], &stc[u].y, &sts[u].y);
                        cc[u] = make_float2(1.f, 1.f);
                        ss[u] = make_float2(0.f, 0.f);
                    }
                    int prev = -2;
#pragma unroll 1
                    for (int r = r0; r < r0 + RUN; ++r) {
                        const int q = meta[s].pos[r];
                        if (q < 0) {
                            prev = -2;
                            continue;
                        }
                        if (q == prev + 1) {
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const float2 c0 = cc[u];
                                cc[u] = __ffma2_rn(c0, stc[u], __fmul2_rn(ss[u], make_float2(-sts[u].x, -sts[u].y)));
                                ss[u] = __ffma2_rn(ss[u], stc[u], __fmul2_rn(c0, sts[u]));
                            }
                        } else {
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                rope_cos_sin((long long)q, p.theta[8 * c + 2 * u], &cc[u].x, &ss[u].x);
                                rope_cos_sin((long long)q, p.theta[8 * c + 2 * u + 1], &cc[u].y, &ss[u].y);
                            }
                        }
                        prev = q;
                        uint4* plo = reinterpret_cast<uint4*>(st + ws_off(r, c));
                        uint4* phi = reinterpret_cast<uint4*>(st + ws_off(r, c + CP));
                        const uint4 wl = *plo, wh = *phi;
                        const uint32_t lw[4] = {wl.x, wl.y, wl.z, wl.w}, hw[4] = {wh.x, wh.y, wh.z, wh.w};
                        uint32_t ol[4], oh[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float2 x1 = make_float2(__uint_as_float(lw[u] << 16), __uint_as_float(lw[u] & 0xffff0000u));
                            const float2 x2 = make_float2(__uint_as_float(hw[u] << 16), __uint_as_float(hw[u] & 0xffff0000u));
                            const float2 y1 = __ffma2_rn(x1, cc[u], __fmul2_rn(x2, make_float2(-ss[u].x, -ss[u].y)));
                            const float2 y2 = __ffma2_rn(x1, ss[u], __fmul2_rn(x2, cc[u]));
                            ol[u] = pack_bf16x2(y1.x, y1.y);
                            oh[u] = pack_bf16x2(y2.x, y2.y);
                        }
                        *plo = make_uint4(ol[0], ol[1], ol[2], ol[3]);
                        *phi = make_uint4(oh[0], oh[1], oh[2], oh[3]);
                    }
                    wrote = true;
                }
                if (wrote) fence_proxy_async_smem();
            }
            mbar_arrive(&bars->ready[s]);
            if (kind == kTileEnd) break;
        }
    } else if (warp == 1) {
        // =========================== MMA issuer =============================
        if (lane == 0) {
            constexpr uint32_t kIdescS = ws_idesc(kWsRows, kWsKeys, 0);
            constexpr uint32_t kIdescO = ws_idesc(kWsRows, D, 1);
            bool ok = true;
            int nt = 0x7fffffff;
            auto stage_u = [&](int j) { return sm_u + S::OffStage + (j % NST) * S::StageBytes; };
            // S_i(j) = Q_i K_j^T
            auto issue_s = [&](int j) {
                for (int i = 0; i < NQ && ok; ++i) {
                    if (j >= 2 && !ws_wait(&bars->s_free[i][j & 1], ((j >> 1) - 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    ws_fence_after();
                    const uint32_t q_u = sm_u + S::OffQ + i * S::QBytes;
                    const uint32_t k_u = stage_u(j);
                    const uint32_t d = tmem + S::SCol0 + (uint32_t)((i * 2 + (j & 1)) * kWsKeys);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t within = (ks & 3) * 32;
                        ws_mma(d, ws_sdesc(q_u + (ks >> 2) * (kWsRows * 128) + within, 16, 1024),
                               ws_sdesc(k_u + (ks >> 2) * S::KVBlock + within, 16, 1024), kIdescS, ks > 0);
                    }
                    ws_commit(&bars->s_full[i][j & 1]);
                }
            };
            // S of tile t for every Q tile, once its keys are in place; false at
            // the end marker (nt = t) or when a wait gave up
            auto try_issue = [&](int t) -> bool {
                if (!ok || t >= nt) return false;
                if (!ws_wait(&bars->ready[t % NST], (t / NST) & 1, abort)) {
                    ok = false;
                    return false;
                }
                if (meta[t % NST].kind == kTileEnd) {
                    nt = t;
                    return false;
                }
                for (int i = 0; i < NQ && ok; ++i) {
                    // q at position 0, and (read-time RoPE) again past the sink tile
                    if (t == 0 && !ws_wait(&bars->q_ready[i], 0, abort)) ok = false;
                    if (READ && sink_tile && t == 1 && !ws_wait(&bars->q_ready[i], 1, abort)) ok = false;
                }
                if (ok) issue_s(t);
                return ok;
            };
            // S runs LA tiles ahead of P V: each Q tile's next scores are queued
            // on the tensor cores while its softmax works on the current ones.
            // LA + 1 tiles are in flight, so the stages must hold them.
            constexpr int LA = NST >= 3 ? 2 : 1;
            int issued = 0;
            while (issued < LA && try_issue(issued)) ++issued;
            int j = 0;
            for (; ok && j < issued; ++j) {
                // O_i += P_i V_j
                for (int i = 0; i < NQ && ok; ++i) {
                    if (!ws_wait(&bars->p_full[i], j & 1, abort)) {
                        ok = false;
                        break;
                    }
                    ws_fence_after();
                    // P_i(j) in the S buffer it came from (bf16 pairs, 32 columns);
                    // S of tile j + 2 reuses that buffer, issued after this P V
                    const uint32_t p_t = tmem + S::SCol0 + (uint32_t)((i * 2 + (j & 1)) * kWsKeys);
                    const uint32_t v_u = stage_u(j) + kWsKeys * 128;
#pragma unroll
                    for (int ks = 0; ks < kWsKeys / 16; ++ks)
                        ws_mma_ts(tmem + (uint32_t)(i * D), p_t + (uint32_t)(ks * 8),
                                  ws_sdesc(v_u + ks * 16 * 128, S::KVBlock, 1024), kIdescO, (j > 0 || ks > 0));
                    ws_commit(&bars->o_done[i]);
                }
                if (!ok) break;
                ws_commit(&bars->empty[j % NST]);       // K and V of tile j are done with
                if (issued == j + LA && try_issue(issued)) ++issued;
            }
            if (*abort) ok = false;
            nt = j;
            if (ok) {
                // the end: the softmax warps learn the tile count at the S slot
                // they wait on next (every S before it has been consumed)
                bars->ntiles = nt;
                for (int i = 0; i < NQ; ++i) mbar_arrive(&bars->s_full[i][nt & 1]);
            } else {
                give_up();
            }
            // every product this thread issued is done before TMEM is freed
            ws_commit(&bars->fin);
            if (!mbar_wait(&bars->fin, 0)) set_error(p.err, 0x8u /* KVC_DEV_TIMEOUT */);
        }
        __syncwarp();
    } else if (warp >= kWsSoftmax0 && warp < kWsSoftmax0 + 4 * NQ) {
        // ============================ softmax ==============================
        const int qi = (warp - kWsSoftmax0) >> 2;     // Q tile
        const int r = tid - (kWsSoftmax0 + 4 * qi) * 32;   // row = TMEM lane
        const int tl = r / G;
        const int row_i = i0 + qi * tq + tl;
        const int row_h = h * G + r % G;
        const int row_t = pos0 + row_i;
        const bool row_ok = tl < tq && row_i < p.T && row_t >= 0;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        unsigned char* Qs = sm + S::OffQ + qi * S::QBytes;

        // Q row: rotated at qpos, scaled by q_scale (softmax scale * log2 e), bf16
        auto write_q = [&](long long qpos) {
            const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) +
                                        (((long long)b * p.T + (row_ok ? row_i : 0)) * p.Hq + row_h) * D;
            const bool rot = p.rope != kRopeNone && row_ok;
#pragma unroll 1
            for (int cbk = 0; cbk < D / 16; ++cbk) {
                uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
                if (row_ok) {
                    lo = *reinterpret_cast<const uint4*>(qrow + 8 * cbk);
                    hi = *reinterpret_cast<const uint4*>(qrow + D / 2 + 8 * cbk);
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
                            rope_cos_sin(qpos, p.theta[8 * cbk + 2 * e + u], &cs, &sn);
                            const float x1 = x[u], x2 = y[u];
                            x[u] = x1 * cs - x2 * sn;
                            y[u] = x1 * sn + x2 * cs;
                        }
                    }
                    lo2[e] = pack_bf16x2(x[0] * p.q_scale, x[1] * p.q_scale);
                    hi2[e] = pack_bf16x2(y[0] * p.q_scale, y[1] * p.q_scale);
                }
                // Q tile: [column block][128 rows][128 B], 128-byte swizzle
                const int c1 = cbk, c2 = cbk + D / 16;
                *reinterpret_cast<uint4*>(Qs + (c1 >> 3) * (kWsRows * 128) + r * 128 + (((c1 ^ r) & 7) << 4)) =
                    make_uint4(lo2[0], lo2[1], lo2[2], lo2[3]);
                *reinterpret_cast<uint4*>(Qs + (c2 >> 3) * (kWsRows * 128) + r * 128 + (((c2 ^ r) & 7) << 4)) =
                    make_uint4(hi2[0], hi2[1], hi2[2], hi2[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars->q_ready[qi]);
        };
        write_q(sink_tile ? min(row_t, C - 1) : row_t);

        float m_run = -INFINITY, l_run = 0.f;
        int j = 0;
        bool ok = true;
        for (;; ++j) {
            if (!ws_wait(&bars->s_full[qi][j & 1], (j >> 1) & 1, abort)) {
                ok = false;
                break;
            }
            if (j == *reinterpret_cast<volatile int*>(&bars->ntiles)) break;
            ws_fence_after();
            float sv[kWsKeys];
            const uint32_t scol = S::SCol0 + (uint32_t)((qi * 2 + (j & 1)) * kWsKeys);
            ws_ld32(lane_base + scol, sv);
            ws_ld32(lane_base + scol + 32, sv + 32);
            ws_wait_ld();
            ws_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->s_free[qi][j & 1]);
            if (READ && sink_tile && j == 0) write_q(row_t);     // S of the sink tile is out of TMEM
            const int s = j % NST;
            if (!ws_wait(&bars->ready[s], (j / NST) & 1, abort)) {    // the stage's meta
                ok = false;
                break;
            }
            // masks: a key at position q is seen by the row at t iff q <= t and
            // (paged, or a sink q < S, or q in the window t - W + 1 .. t)
            const int mode = meta[s].mask;
            if (!row_ok) {
#pragma unroll
                for (int k = 0; k < kWsKeys; ++k) sv[k] = -INFINITY;
            } else if (mode == kMaskRange) {
                // the chunk's own rows: key k at kbase + k is seen iff 0 <= kbase + k <= t
                // (the window holds every chunk token, the chunk being no longer than it)
                const int kb = meta[s].kbase;
                const int klo = -kb, khi = row_t - kb;
#pragma unroll
                for (int k = 0; k < kWsKeys; ++k) sv[k] = (k >= klo && k <= khi) ? sv[k] : -INFINITY;
            } else if (mode == kMaskKeys) {
#pragma unroll
                for (int k = 0; k < kWsKeys; ++k) {
                    const int q = meta[s].pos[k];
                    bool allowed = q >= 0 && q <= row_t;
                    if (!paged) allowed = allowed && (q < p.sinks || q > row_t - p.window);
                    sv[k] = allowed ? sv[k] : -INFINITY;
                }
            }
            // four independent chains (latency, not issue slots, is what the
            // softmax warps wait on)
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int k = 0; k < kWsKeys; k += 4)
#pragma unroll
                for (int u = 0; u < 4; ++u) mq[u] = fmaxf(mq[u], sv[k + u]);
            const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            float mn = m_run, alpha = 1.f;
            if (mx > m_run + kWsLazy) {
                mn = mx;
                alpha = m_run == -INFINITY ? 1.f : exp2f(m_run - mn);
            }
            // p = 2^(s - m) (exactly 0 for a masked key: 2^-inf), summed in pairs
            const float nmn = mn == -INFINITY ? 0.f : -mn;
            float2 ls2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int k = 0; k < kWsKeys; k += 2) {
                const float2 d2 = __fadd2_rn(make_float2(sv[k], sv[k + 1]), make_float2(nmn, nmn));
                const float2 e2 = ws_ex2_pair(d2.x, d2.y);
                sv[k] = e2.x;
                sv[k + 1] = e2.y;
                ls2[(k >> 1) & 3] = __fadd2_rn(ls2[(k >> 1) & 3], e2);
            }
            const float2 lsa = __fadd2_rn(__fadd2_rn(ls2[0], ls2[1]), __fadd2_rn(ls2[2], ls2[3]));
            l_run = l_run * alpha + (lsa.x + lsa.y);
            m_run = mn;
            // P V of the previous tile is done: P's buffer and O are free
            if (j > 0 && !ws_wait(&bars->o_done[qi], (j - 1) & 1, abort)) {
                ok = false;
                break;
            }
            ws_fence_after();
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    float ov[32];
                    ws_ld32(lane_base + (uint32_t)(qi * D + 32 * c4), ov);
                    ws_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) ov[k] *= alpha;
                    ws_st32(lane_base + (uint32_t)(qi * D + 32 * c4), ov);
                }
                ws_wait_st();
            }
            // P row r (bf16 pairs of the 64 keys) into the S buffer just read:
            // the A operand of P V, in tensor memory
            {
                float pw[kWsKeys / 2];
#pragma unroll
                for (int k2 = 0; k2 < kWsKeys / 2; ++k2) pw[k2] = __uint_as_float(pack_bf16x2(sv[2 * k2], sv[2 * k2 + 1]));
                ws_st32(lane_base + scol, pw);
            }
            ws_wait_st();
            ws_fence_before();
            mbar_arrive(&bars->p_full[qi]);
        }
        if (!ok) give_up();
        // the last P V, then O / l to the output
        const int nt = j;
        bool have_o = false;
        if (ok && nt > 0) {
            if (ws_wait(&bars->o_done[qi], (nt - 1) & 1, abort))
                have_o = true;
            else
                give_up();
        }
        ws_fence_after();
        if (!*abort) {
            const float inv = (have_o && l_run > 0.f) ? 1.f / l_run : 0.f;
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + (((long long)b * p.T + row_i) * p.Hq + row_h) * D;
            const bool store = tl < tq && row_i < p.T;
#pragma unroll 1
            for (int c4 = 0; c4 < D / 32; ++c4) {
                float ov[32];
                if (have_o) {
                    ws_ld32(lane_base + (uint32_t)(qi * D + 32 * c4), ov);
                    ws_wait_ld();
                }
                if (store) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = (have_o && row_ok) ? pack_bf16x2(ov[8 * q4 + 2 * e] * inv, ov[8 * q4 + 2 * e + 1] * inv)
                                                      : 0u;
                        *reinterpret_cast<uint4*>(dst + 32 * c4 + 8 * q4) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        }
    }

    // the MMA thread has waited for all of its products (its last commit)
    ws_fence_before();
    __syncthreads();
    ws_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(S::TmemCols) : "memory");
}

template <int D, bool READ, bool Q8>
static cudaError_t launch_prefill_ws_t(const PrefillParams& p, const PrefillMaps& maps, cudaStream_t stream) {
    constexpr int kSmem = ws_smem_bytes<D>();
    static_assert(kSmem <= 227 * 1024, "shared memory of one CTA");
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_relaxed) & bit)) {
        e = cudaFuncSetAttribute(prefill_ws_kernel<D, READ, Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_relaxed);
    }
    const int tok = kWsRows / p.G * WsShape<D>::NQ;
    dim3 grid((p.T + tok - 1) / tok, p.Hkv, p.B);
    prefill_ws_kernel<D, READ, Q8><<<grid, WsShape<D>::Threads, kSmem, stream>>>(p, maps);
    return cudaGetLastError();
}

cudaError_t launch_prefill_ws(int head_dim, bool q8, const PrefillParams& p, const PrefillMaps& maps,
                              cudaStream_t stream) {
    if (p.G < 1 || kWsRows % p.G) return cudaErrorInvalidValue;
    const bool rd = p.rope == kRopeRead;
#define KVC_WS(DD, RD, Q) \
    if (head_dim == DD && rd == RD && q8 == Q) return launch_prefill_ws_t<DD, RD, Q>(p, maps, stream);
    KVC_WS(64, false, false) KVC_WS(64, true, false)
    KVC_WS(128, false, false) KVC_WS(128, true, false) KVC_WS(128, false, true) KVC_WS(128, true, true)
    KVC_WS(256, false, false) KVC_WS(256, true, false) KVC_WS(256, false, true) KVC_WS(256, true, true)
#undef KVC_WS
    return cudaErrorInvalidValue;
}

}  // namespace kvc
