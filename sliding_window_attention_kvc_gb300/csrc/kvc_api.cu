// Host side of the C ABI declared in include/kvc.h: descriptor checks,
// workspace carve-up, launch configuration and dispatch to the kernels.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>

#include "kvc.h"
#include "kvc_params.h"

namespace kvc {

template <typename Elt, int D, int GH, bool PAGED, bool READ>
cudaError_t launch_decode_t(const DecodeParams& p, dim3 grid, cudaStream_t stream);
template <int D, int GH, bool PAGED, bool READ, bool Q8>
cudaError_t launch_decode_mma_t(const DecodeParams& p, const KvTensorMaps& maps, dim3 grid, cudaStream_t stream);

namespace {

struct Geo {
    int elt;        // bytes per cache element (INT8: the codes)
    int act_elt;    // bytes per element of q, out, k_new, v_new
    int C;          // window layouts: slots per (sequence, kv head)
    int G, GH, nsub;
    long long half_elems;   // elements of one K (or V) half of one layer
};

// rows of K/V one pipeline stage holds: fp32 kernel 8 KiB per K stage;
// bf16 tensor-core kernel 4 (2 for head_dim 256) sub-tiles of 16 rows
int rows_per_stage(int elt, int D) { return elt == 4 ? 8192 / (D * elt) : (D == 256 ? 32 : 64); }

int check_desc(const kvc_desc* d, Geo* g) {
    if (!d) return KVC_ERR_NULL;
    if (d->layout < 0 || d->layout > 2 || d->rope < 0 || d->rope > 2 || d->dtype < 0 || d->dtype > 2)
        return KVC_ERR_DESC;
    if (d->layers < 1 || d->batch < 1 || d->kv_heads < 1 || d->q_heads < 1 || d->q_heads % d->kv_heads)
        return KVC_ERR_DESC;
    if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256) return KVC_ERR_UNSUPPORTED;
    if (d->num_splits < 0) return KVC_ERR_DESC;
    if (d->rope != KVC_ROPE_NONE && !(d->rope_base > 0.f)) return KVC_ERR_DESC;
    if (d->softmax_scale < 0.f) return KVC_ERR_DESC;
    g->elt = d->dtype == KVC_F32 ? 4 : (d->dtype == KVC_BF16 ? 2 : 1);
    g->act_elt = d->dtype == KVC_F32 ? 4 : 2;
    if (d->dtype == KVC_I8 && d->head_dim < 128) return KVC_ERR_UNSUPPORTED;
    g->G = d->q_heads / d->kv_heads;
    g->GH = (g->G % 4 == 0) ? 4 : ((g->G % 2 == 0) ? 2 : 1);
    g->nsub = g->G / g->GH;
    // launch-grid limits: sequences on x, (kv head, q-head group) pairs on y,
    // and a 32-bit count of (sequence, pair) units
    const long long pairs = (long long)d->kv_heads * g->nsub;
    if (d->batch > 65535 || pairs > 65535 || d->batch * pairs > 0x7fffffffLL) return KVC_ERR_DESC;
    if (d->layout == KVC_LAYOUT_PAGED) {
        if (d->block_size < 1 || d->num_blocks < 1 || d->max_blocks_per_seq < 1) return KVC_ERR_DESC;
        if ((long long)d->block_size * d->max_blocks_per_seq > 0x7fffffffLL) return KVC_ERR_DESC;
        if (d->rope == KVC_ROPE_READ_INCACHE) return KVC_ERR_UNSUPPORTED;
        g->C = 0;
        g->half_elems = (long long)d->num_blocks * d->kv_heads * d->block_size * d->head_dim;
    } else {
        if (d->window < 1) return KVC_ERR_DESC;
        if (d->layout == KVC_LAYOUT_RING && d->sinks != 0) return KVC_ERR_DESC;
        if (d->layout == KVC_LAYOUT_SINK_RING && d->sinks < 1) return KVC_ERR_DESC;
        if ((long long)d->window + d->sinks > 0x3fffffffLL) return KVC_ERR_DESC;
        g->C = d->window + d->sinks;
        g->half_elems = (long long)d->batch * d->kv_heads * g->C * d->head_dim;
    }
    // INT8 scale tensor maps: rows of a half in multiples of 4 (16-byte strides)
    if (d->dtype == KVC_I8 && (g->half_elems / d->head_dim) % 4) return KVC_ERR_UNSUPPORTED;
    return KVC_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WorkspaceLayout ws_layout(const kvc_desc* d, const Geo& g) {
    WorkspaceLayout w{};
    const int units = d->batch * d->kv_heads * g.nsub;
    const int groups = d->kv_heads * g.nsub;
    // stream-K shares per (kv head, q-head group): bf16 kernels, and the paged
    // plan.  bf16: a persistent grid of about two CTAs per SM claims them in turn.
    // the persistent grid: 152 SMs times the decode kernel's resident CTAs
    // (at least two: kernels held to one CTA per SM keep two shares per SM)
    const int per_sm = decode_ctas_per_sm(d->dtype == KVC_I8, d->layout == KVC_LAYOUT_PAGED,
                                          d->rope == KVC_ROPE_READ_INCACHE, d->head_dim);
    const int stream_ctas = kStreamCtas / 2 * (per_sm > 2 ? per_sm : 2);
    const int persist = (stream_ctas + groups - 1) / groups;
    if (d->layout == KVC_LAYOUT_PAGED || d->dtype != KVC_F32) {
        const bool bf16 = d->dtype != KVC_F32;     // tensor-core kernel (bf16 or INT8 cache)
        const int factor = (bf16 && d->layout == KVC_LAYOUT_PAGED && d->batch >= kPagedShareBatch)
                               ? kPagedShareFactor : 1;
        w.shares = d->num_splits > 0 ? d->num_splits : factor * persist;
        w.ctas = bf16 ? (persist < w.shares ? persist : w.shares) : w.shares;
        w.items = w.shares + d->batch;     // slot x + b of segment (share x, sequence b)
        w.nsplit = 0;
    } else {
        const int T = rows_per_stage(g.elt, d->head_dim);
        int maxs = g.C / (2 * T);
        if (maxs < 1) maxs = 1;
        int ns = d->num_splits > 0 ? d->num_splits : (kTargetCtas + units - 1) / units;
        if (d->num_splits <= 0 && ns > maxs) ns = maxs;
        if (ns < 1) ns = 1;
        w.nsplit = ns;
        w.items = d->batch * ns;
    }
    size_t off = 0;
    w.err = off;
    off += 256;
    w.counters = off;
    off = align_up(off + (size_t)(units + 1) * 4, 256);
    w.part_ml = off;
    off = align_up(off + (size_t)w.items * d->q_heads * 8, 256);
    w.part_o = off;
    off = align_up(off + (size_t)w.items * d->q_heads * d->head_dim * 4, 256);
    w.plan_seq = w.plan_acc = w.plan_items = w.plan_info = w.plan_total = w.plan_cta = w.plan_dir = w.plan_refs = w.blocks = off;
    if (d->layout == KVC_LAYOUT_PAGED) {
        w.plan_seq = off;
        off = align_up(off + (size_t)d->batch * 8, 256);
        w.plan_acc = off;
        off = align_up(off + (size_t)d->batch * 12, 256);
        w.plan_items = off;
        off = align_up(off + (size_t)w.items * 16, 256);
        w.plan_info = off;
        off = align_up(off + (size_t)w.items * 16, 256);
        w.plan_cta = off;
        off = align_up(off + (size_t)w.shares * 8, 256);
        w.plan_dir = off;
        off = align_up(off + (size_t)d->batch * ((d->max_blocks_per_seq + 31) / 32) * 8, 256);
        w.plan_refs = off;
        off = align_up(off + (size_t)d->num_blocks * 4, 256);
        w.blocks = off;
        off = align_up(off + align_up((size_t)d->batch * 5 * 4, 16) + (size_t)d->batch * 16 + 16 +
                           (size_t)d->num_blocks * 4, 256);
        w.plan_total = off;
        off += 256;
    }
    w.total = off;
    return w;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// theta_i = base^(-2i/D); passed as fp32 (small in-tile angles) and as the
// 64-bit fixed-point fraction of a turn theta_i / (2 pi) * 2^64 used for
// exact reduction of pos * theta_i on the device.
void fill_theta(int D, float base, unsigned long long* turns, float* theta_f) {
    const double two_pi = 6.283185307179586476925286766559;
    for (int i = 0; i < D / 2; ++i) {
        const double th = std::pow((double)base, -2.0 * i / D);
        turns[i] = (unsigned long long)std::ldexp(th / two_pi, 64);
        if (theta_f) theta_f[i] = (float)th;
    }
}

}  // namespace

cudaError_t launch_decode(int dtype, int D, int gh, bool paged, bool rd, const DecodeParams& p, dim3 grid,
                          cudaStream_t s) {
#define KVC_CASE(E, DD, GG, PG, RD) \
    if (D == DD && gh == GG && paged == PG && rd == RD) return launch_decode_t<E, DD, GG, PG, RD>(p, grid, s);
#define KVC_CASES(E, PG, RD)                                                         \
    KVC_CASE(E, 64, 1, PG, RD) KVC_CASE(E, 64, 2, PG, RD) KVC_CASE(E, 64, 4, PG, RD)    \
    KVC_CASE(E, 128, 1, PG, RD) KVC_CASE(E, 128, 2, PG, RD) KVC_CASE(E, 128, 4, PG, RD) \
    KVC_CASE(E, 256, 1, PG, RD) KVC_CASE(E, 256, 2, PG, RD) KVC_CASE(E, 256, 4, PG, RD)
    if (dtype == KVC_F32) {
        KVC_CASES(float, false, false)
        KVC_CASES(float, false, true)
        KVC_CASES(float, true, false)
    }
#undef KVC_CASES
#undef KVC_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_mma(int D, int gh, bool paged, bool rd, bool q8, const DecodeParams& p,
                              const KvTensorMaps& maps, dim3 grid, cudaStream_t s) {
#define KVC_CASE(DD, GG, PG, RD, Q)                                       \
    if (D == DD && gh == GG && paged == PG && rd == RD && q8 == Q)        \
        return launch_decode_mma_t<DD, GG, PG, RD, Q>(p, maps, grid, s);
#define KVC_CASES(PG, RD)                                                                        \
    KVC_CASE(64, 1, PG, RD, false) KVC_CASE(64, 2, PG, RD, false) KVC_CASE(64, 4, PG, RD, false)    \
    KVC_CASE(128, 1, PG, RD, false) KVC_CASE(128, 2, PG, RD, false) KVC_CASE(128, 4, PG, RD, false) \
    KVC_CASE(256, 1, PG, RD, false) KVC_CASE(256, 2, PG, RD, false) KVC_CASE(256, 4, PG, RD, false)
#define KVC_CASES_Q8(PG, RD)                                                                    \
    KVC_CASE(128, 1, PG, RD, true) KVC_CASE(128, 2, PG, RD, true) KVC_CASE(128, 4, PG, RD, true) \
    KVC_CASE(256, 1, PG, RD, true) KVC_CASE(256, 2, PG, RD, true) KVC_CASE(256, 4, PG, RD, true)
    KVC_CASES(false, false)
    KVC_CASES(false, true)
    KVC_CASES(true, false)
    KVC_CASES_Q8(false, false)
    KVC_CASES_Q8(false, true)
    KVC_CASES_Q8(true, false)
#undef KVC_CASES_Q8
#undef KVC_CASES
#undef KVC_CASE
    return cudaErrorInvalidValue;
}

namespace {

// cuTensorMapEncodeTiled, looked up once through the runtime's driver entry
// point (no link against the driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Tensor maps over a bf16 cache for copies of runs of 16 r consecutive rows of
// one K half together with the same rows of its V half (r = 1..kRunMaps).
// The cache [layers][K|V][rows per half][head_dim] is viewed as the 5-D tensor
// {64 columns, row, K|V, layer, 64-column block} (byte strides: row, half,
// 2 halves, 128), which brings every column block in one copy; if the driver
// refuses it, the 4-D tensor {column, row, K|V, layer} takes one copy per
// 64-column block.  Both land as [column block][K|V][rows][128 bytes] with the
// 128-byte swizzle.  Rows past the end of a half read as zeros.
int encode_kv_maps(const kvc_desc* d, const Geo& g, const void* cache, KvTensorMaps* maps, int* whole) {
    const unsigned long long half_rows = (unsigned long long)g.half_elems / d->head_dim;
    if (half_rows >= (1ull << 31)) return KVC_ERR_UNSUPPORTED;
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return KVC_ERR_CUDA;
    const bool q8 = d->dtype == KVC_I8;
    const CUtensorMapDataType type = q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t row_bytes = (cuuint64_t)d->head_dim * g.elt, half_bytes = half_rows * row_bytes;
    const cuuint32_t bcols = 128u / (cuuint32_t)g.elt;                 // columns of a 128-byte box row
    const cuuint32_t boxes = (cuuint32_t)(d->head_dim / bcols);
    if (q8) {
        // row scales: {row, K|V, layer} fp32 after the codes of every layer
        void* scales = static_cast<char*>(const_cast<void*>(cache)) + (size_t)d->layers * 2 * half_bytes;
        const cuuint64_t dims[3] = {half_rows, 2, (cuuint64_t)d->layers};
        const cuuint64_t strides[2] = {half_rows * 4, 2 * half_rows * 4};
        const cuuint32_t estr[3] = {1, 1, 1};
        const cuuint32_t box_run[3] = {(cuuint32_t)kScRunRows, 2, 1}, box_sub[3] = {(cuuint32_t)kScSubRows, 2, 1};
        if (fn(&maps->sc_run, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, scales, dims, strides, box_run, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
            fn(&maps->sc_sub, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, scales, dims, strides, box_sub, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return KVC_ERR_CUDA;
    }
    for (int pass = boxes > 1 ? 0 : 1; pass < 2; ++pass) {
        const bool five = pass == 0;
        bool ok = true;
        for (int r = 0; r < kRunMaps && ok; ++r) {
            const cuuint32_t R = 16u * (cuuint32_t)(r + 1);
            CUresult e;
            if (five) {
                const cuuint64_t dims[5] = {bcols, half_rows, 2, (cuuint64_t)d->layers, boxes};
                const cuuint64_t strides[4] = {row_bytes, half_bytes, 2 * half_bytes, 128};
                const cuuint32_t box[5] = {bcols, R, 2, 1, boxes};
                const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
                e = fn(&maps->run[r], type, 5, const_cast<void*>(cache), dims, strides,
                       box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            } else {
                const cuuint64_t dims[4] = {(cuuint64_t)d->head_dim, half_rows, 2, (cuuint64_t)d->layers};
                const cuuint64_t strides[3] = {row_bytes, half_bytes, 2 * half_bytes};
                const cuuint32_t box[4] = {bcols, R, 2, 1};
                const cuuint32_t estr[4] = {1, 1, 1, 1};
                e = fn(&maps->run[r], type, 4, const_cast<void*>(cache), dims, strides,
                       box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            }
            ok = e == CUDA_SUCCESS;
        }
        if (ok) {
            *whole = five ? 1 : 0;
            return KVC_OK;
        }
    }
    return KVC_ERR_CUDA;
}

// The maps depend only on the cache's address and shape: the last few are
// kept, so that a decode step does not pay for encoding them.
int kv_maps_for(const kvc_desc* d, const Geo& g, const void* cache, KvTensorMaps* maps, int* whole) {
    struct Entry {
        const void* cache;
        long long half_elems;
        int layers, head_dim, dtype, device, whole;
        KvTensorMaps maps;
    };
    constexpr int kEntries = 8;
    static Entry entries[kEntries];
    static int used = 0, next = 0;
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVC_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i) {
            const Entry& e = entries[i];
            if (e.cache == cache && e.half_elems == g.half_elems && e.layers == d->layers &&
                e.head_dim == d->head_dim && e.dtype == d->dtype && e.device == dev) {
                *maps = e.maps;
                *whole = e.whole;
                return KVC_OK;
            }
        }
    }
    const int rc = encode_kv_maps(d, g, cache, maps, whole);
    if (rc) return rc;
    std::lock_guard<std::mutex> lock(mu);
    Entry& e = entries[next];
    e.cache = cache;
    e.half_elems = g.half_elems;
    e.layers = d->layers;
    e.head_dim = d->head_dim;
    e.dtype = d->dtype;
    e.device = dev;
    e.whole = *whole;
    e.maps = *maps;
    next = (next + 1) % kEntries;
    if (used < kEntries) ++used;
    return KVC_OK;
}

// INT8 caches, for the warp-specialised prefill: the codes as {D bytes, row,
// K|V, layer}, boxes of 128 codes of `rows` rows (64 for slot tiles, a block
// for paged tiles), no swizzle (rows land as 128 contiguous bytes).
int encode_q8_code_map(const kvc_desc* d, const Geo& g, const void* cache, int rows, CUtensorMap* map) {
    const unsigned long long half_rows = (unsigned long long)g.half_elems / d->head_dim;
    if (half_rows >= (1ull << 31)) return KVC_ERR_UNSUPPORTED;
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return KVC_ERR_CUDA;
    const cuuint64_t row_bytes = (cuuint64_t)d->head_dim, half_bytes = half_rows * row_bytes;
    const cuuint64_t dims[4] = {(cuuint64_t)d->head_dim, half_rows, 2, (cuuint64_t)d->layers};
    const cuuint64_t strides[3] = {row_bytes, half_bytes, 2 * half_bytes};
    const cuuint32_t box[4] = {128, (cuuint32_t)rows, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(cache), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? KVC_OK
               : KVC_ERR_CUDA;
}

// Paged caches, for the warp-specialised prefill: {column, row, K|V, layer}
// with boxes of one block (bs rows) of K or of V, 64 columns.
int encode_block_map(const kvc_desc* d, const Geo& g, const void* cache, CUtensorMap* map) {
    const unsigned long long half_rows = (unsigned long long)g.half_elems / d->head_dim;
    if (half_rows >= (1ull << 31)) return KVC_ERR_UNSUPPORTED;
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return KVC_ERR_CUDA;
    const cuuint64_t row_bytes = (cuuint64_t)d->head_dim * 2, half_bytes = half_rows * row_bytes;
    const cuuint64_t dims[4] = {(cuuint64_t)d->head_dim, half_rows, 2, (cuuint64_t)d->layers};
    const cuuint64_t strides[3] = {row_bytes, half_bytes, 2 * half_bytes};
    const cuuint32_t box[4] = {64, (cuuint32_t)d->block_size, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(cache), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? KVC_OK
               : KVC_ERR_CUDA;
}

// The chunk's staged rows, K [batch][T][kv head][D] then V at kv_bytes past
// it: {64 columns, kv head, batch * T, K|V, column block}, boxes of 64 tokens
// of one kv head, K and V, every column.
int encode_stage_map(const kvc_desc* d, const void* kst, long long T, size_t kv_bytes, CUtensorMap* map) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return KVC_ERR_CUDA;
    const cuuint64_t D = (cuuint64_t)d->head_dim;
    const cuuint64_t dims[5] = {64, (cuuint64_t)d->kv_heads, (cuuint64_t)(d->batch * T), 2, D / 64};
    const cuuint64_t strides[4] = {D * 2, (cuuint64_t)d->kv_heads * D * 2, (cuuint64_t)kv_bytes, 128};
    const cuuint32_t box[5] = {64, 1, 64, 2, (cuuint32_t)(D / 64)};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(kst), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? KVC_OK
               : KVC_ERR_CUDA;
}

}  // namespace

}  // namespace kvc

using namespace kvc;

extern "C" KVC_API int kvc_append(const kvc_desc* d, void* cache, int32_t layer, const void* k_new, const void* v_new,
                                  int32_t n_new, const int32_t* pos, const int32_t* block_table, void* workspace,
                                  size_t workspace_bytes, void* stream);

// The attention's pointer, alignment and layer checks (kvc_decode_attention,
// kvc_decode_step, kvc_decode_attention_noalloc), made before anything is issued.
static int decode_args(const kvc_desc* d, const void* cache, int32_t layer, const void* q, const int32_t* pos,
                       const int32_t* block_table, const void* out) {
    if (!cache || !q || !pos || !out) return KVC_ERR_NULL;
    if (d->layout == KVC_LAYOUT_PAGED && !block_table) return KVC_ERR_NULL;
    if (!aligned16(cache) || !aligned16(q) || !aligned16(out)) return KVC_ERR_ALIGN;
    if (layer < 0 || layer >= d->layers) return KVC_ERR_ARG;
    return KVC_OK;
}

static int decode_impl(const kvc_desc* d, const void* cache, int32_t layer, const void* q, const void* k_new,
                       const void* v_new, const int32_t* pos, const int32_t* block_table,
                       const uint32_t* valid_bits, void* out, void* workspace, size_t workspace_bytes,
                       void* stream) {
    Geo g;
    int rc = check_desc(d, &g);
    if (rc) return rc;
    if ((rc = decode_args(d, cache, layer, q, pos, block_table, out))) return rc;
    if (!workspace) return KVC_ERR_NULL;
    if (!aligned16(workspace)) return KVC_ERR_ALIGN;
    const bool paged = d->layout == KVC_LAYOUT_PAGED;
    const WorkspaceLayout w = ws_layout(d, g);
    if (workspace_bytes < w.total) return KVC_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    cudaStream_t s = (cudaStream_t)stream;

    DecodeParams p{};
    p.cache = cache;
    p.q = q;
    p.pos = pos;
    p.table = block_table;
    p.valid = valid_bits;
    p.out = out;
    p.k_new = k_new;
    p.v_new = v_new;
    p.err = reinterpret_cast<uint32_t*>(ws + w.err);
    p.counters = reinterpret_cast<uint32_t*>(ws + w.counters);
    p.part_ml = reinterpret_cast<float2*>(ws + w.part_ml);
    p.part_o = reinterpret_cast<float*>(ws + w.part_o);
    p.layer_off = (long long)layer * 2 * g.half_elems;
    p.layer = layer;
    p.kv_off = g.half_elems;
    if (d->dtype == KVC_I8) {
        const long long half_rows = g.half_elems / d->head_dim;
        p.scales = reinterpret_cast<float*>(static_cast<char*>(const_cast<void*>(cache)) +
                                            (size_t)d->layers * 2 * (size_t)g.half_elems);
        p.sc_layer_off = (long long)layer * 2 * half_rows;
        p.sc_kv_off = half_rows;
    }
    p.B = d->batch;
    p.Hq = d->q_heads;
    p.Hkv = d->kv_heads;
    p.G = g.G;
    p.nsub = g.nsub;
    p.window = d->window;
    p.sinks = d->layout == KVC_LAYOUT_SINK_RING ? d->sinks : 0;
    p.capacity = g.C;
    p.bs = d->block_size;
    p.num_blocks = d->num_blocks;
    p.maxb = d->max_blocks_per_seq;
    p.nsplit = d->dtype != KVC_F32 ? w.shares : w.nsplit;   // bf16 / INT8: stream-K shares per (kv head, group)
    p.max_items = w.items;
    p.rope = d->rope;
    const float scale = d->softmax_scale > 0.f ? d->softmax_scale : 1.0f / std::sqrt((float)d->head_dim);
    p.q_scale = scale * 1.4426950408889634f;   // log2(e): softmax in base 2
    if (d->rope != KVC_ROPE_NONE) fill_theta(d->head_dim, d->rope_base, p.theta, p.theta_f);

    dim3 grid(d->dtype != KVC_F32 ? w.ctas : w.items, d->kv_heads, g.nsub);
    // the tensor-core kernel's maps, encoded before anything is launched (a
    // failure leaves the cache and the workspace untouched)
    KvTensorMaps maps;
    if (d->dtype != KVC_F32 && (rc = kv_maps_for(d, g, cache, &maps, &p.tma_whole))) return rc;
    // one paged sequence on the tensor-core kernel: its CTAs plan their own
    // shares from the block table and write the step's token themselves
    // (the CTAs bulk-copy the table and the valid words: 16-byte aligned buffers)
    p.self_plan = (paged && d->dtype != KVC_F32 && d->batch == 1 && d->max_blocks_per_seq <= kSelfPlanMax &&
                   (d->num_blocks + 31) / 32 <= kSelfPlanValidWords && aligned16(block_table) &&
                   (!valid_bits || aligned16(valid_bits))) ? 1 : 0;
    if (p.self_plan) {
        p.seq_items = reinterpret_cast<int2*>(ws + w.plan_seq);
        p.n_items = reinterpret_cast<int32_t*>(ws + w.plan_total);
        p.items = reinterpret_cast<int4*>(ws + w.plan_items);
        p.item_info = reinterpret_cast<int4*>(ws + w.plan_info);
        p.cta_items = reinterpret_cast<int2*>(ws + w.plan_cta);
    } else if (paged) {
        PlanParams pp{};
        pp.pos = pos;
        pp.table = block_table;
        pp.valid = valid_bits;
        pp.err = p.err;
        pp.seq_off = reinterpret_cast<long long*>(ws + w.plan_acc);
        pp.seq_rows = reinterpret_cast<int32_t*>(ws + w.plan_acc + (size_t)d->batch * 8);
        pp.ticket = reinterpret_cast<uint32_t*>(ws + w.counters) + (size_t)d->batch * d->kv_heads * g.nsub;
        pp.seq_items = reinterpret_cast<int2*>(ws + w.plan_seq);
        pp.items = reinterpret_cast<int4*>(ws + w.plan_items);
        pp.item_info = reinterpret_cast<int4*>(ws + w.plan_info);
        pp.n_items = reinterpret_cast<int32_t*>(ws + w.plan_total);
        pp.cta_items = reinterpret_cast<int2*>(ws + w.plan_cta);
        pp.ctas = w.shares;
        pp.B = d->batch;
        pp.bs = d->block_size;
        pp.num_blocks = d->num_blocks;
        pp.maxb = d->max_blocks_per_seq;
        pp.max_items = w.items;
        if (k_new) {             // kvc_decode_step: the plan kernel writes the new token first
            pp.cache = const_cast<void*>(cache);
            pp.k_new = k_new;
            pp.v_new = v_new;
            pp.layer_off = p.layer_off;
            pp.kv_off = p.kv_off;
            pp.Hkv = d->kv_heads;
            pp.D = d->head_dim;
            pp.rope = d->rope;
            pp.elt = g.elt;
            pp.scales = p.scales;
            pp.sc_layer_off = p.sc_layer_off;
            pp.sc_kv_off = p.sc_kv_off;
            if (d->rope == KVC_ROPE_BAKED) fill_theta(d->head_dim, d->rope_base, pp.theta, nullptr);
        }
        if (d->dtype != KVC_F32) {
            // the tensor-core kernel cuts its own shares from the rows and the
            // directory of each sequence
            pp.dir = reinterpret_cast<int2*>(ws + w.plan_dir);
            pp.dir_groups = (d->max_blocks_per_seq + 31) / 32;
            pp.refs = reinterpret_cast<uint32_t*>(ws + w.plan_refs);
            if (launch_plan_rows(pp, s) != cudaSuccess) return KVC_ERR_CUDA;
            p.seq_rows = pp.seq_rows;
            p.dir = pp.dir;
            p.dir_groups = pp.dir_groups;
            p.refs = pp.refs;
        } else if (launch_plan(pp, s) != cudaSuccess) {
            return KVC_ERR_CUDA;
        }
        p.items = pp.items;
        p.item_info = pp.item_info;
        p.seq_items = pp.seq_items;
        p.n_items = pp.n_items;
        p.cta_items = pp.cta_items;
    }
    const bool rd = d->rope == KVC_ROPE_READ_INCACHE;
    if (d->dtype != KVC_F32) {
        if (launch_decode_mma(d->head_dim, g.GH, paged, rd, d->dtype == KVC_I8, p, maps, grid, s) != cudaSuccess)
            return KVC_ERR_CUDA;
        return KVC_OK;
    }
    if (launch_decode(d->dtype, d->head_dim, g.GH, paged, rd, p, grid, s) != cudaSuccess) return KVC_ERR_CUDA;
    return KVC_OK;
}


namespace {
// Block manager parameters over the workspace's block region.
int block_params(const kvc_desc* d, const Geo& g, void* workspace, size_t workspace_bytes, kvc::BlockParams* p) {
    if (d->layout != KVC_LAYOUT_PAGED) return KVC_ERR_DESC;
    if (!workspace) return KVC_ERR_NULL;
    if (!aligned16(workspace)) return KVC_ERR_ALIGN;
    const WorkspaceLayout w = ws_layout(d, g);
    if (workspace_bytes < w.total) return KVC_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    char* r = ws + w.blocks;
    const size_t B = (size_t)d->batch;
    *p = kvc::BlockParams{};
    p->err = reinterpret_cast<uint32_t*>(ws + w.err);
    p->tgt = reinterpret_cast<int32_t*>(r);
    p->rcnt = p->tgt + B;
    p->need = p->rcnt + B;
    p->aidx = p->need + B;
    p->prev = p->aidx + B;
    p->copies = reinterpret_cast<int4*>(r + align_up(5 * 4 * B, 16));
    p->ncopies = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(p->copies) + 16 * B);
    p->flags = p->ncopies + 4;
    p->B = d->batch;
    p->bs = d->block_size;
    p->num_blocks = d->num_blocks;
    p->maxb = d->max_blocks_per_seq;
    p->layers = d->layers;
    p->Hkv = d->kv_heads;
    p->D = d->head_dim;
    return KVC_OK;
}
}  // namespace

extern "C" {

KVC_API size_t kvc_cache_bytes(const kvc_desc* d) {
    Geo g;
    if (check_desc(d, &g) != KVC_OK) return 0;
    const size_t rows = (size_t)d->layers * 2 * (size_t)(g.half_elems / d->head_dim);
    // INT8: the codes, then one fp32 scale per row
    return rows * d->head_dim * g.elt + (d->dtype == KVC_I8 ? rows * 4 : 0);
}

KVC_API size_t kvc_workspace_bytes(const kvc_desc* d) {
    Geo g;
    if (check_desc(d, &g) != KVC_OK) return 0;
    return ws_layout(d, g).total;
}

KVC_API int kvc_workspace_init(const kvc_desc* d, void* workspace, size_t workspace_bytes, void* stream) {
    Geo g;
    int rc = check_desc(d, &g);
    if (rc) return rc;
    if (!workspace) return KVC_ERR_NULL;
    const size_t need = ws_layout(d, g).total;
    if (workspace_bytes < need) return KVC_ERR_WORKSPACE;
    if (cudaMemsetAsync(workspace, 0, need, (cudaStream_t)stream) != cudaSuccess) return KVC_ERR_CUDA;
    return KVC_OK;
}

KVC_API int kvc_append(const kvc_desc* d, void* cache, int32_t layer, const void* k_new, const void* v_new,
                       int32_t n_new, const int32_t* pos, const int32_t* block_table, void* workspace,
                       size_t workspace_bytes, void* stream) {
    Geo g;
    int rc = check_desc(d, &g);
    if (rc) return rc;
    if (!cache || !k_new || !v_new || !pos || !workspace) return KVC_ERR_NULL;
    if (d->layout == KVC_LAYOUT_PAGED && !block_table) return KVC_ERR_NULL;
    if (!aligned16(cache) || !aligned16(workspace)) return KVC_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & (uintptr_t)(g.act_elt - 1))
        return KVC_ERR_ALIGN;
    if (layer < 0 || layer >= d->layers || n_new < 1 || n_new > 0x7fffffff / 2) return KVC_ERR_ARG;
    const WorkspaceLayout w = ws_layout(d, g);
    if (workspace_bytes < w.total) return KVC_ERR_WORKSPACE;
    AppendParams p{};
    p.cache = cache;
    p.k_new = k_new;
    p.v_new = v_new;
    p.pos = pos;
    p.table = block_table;
    p.err = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + w.err);
    p.layer_off = (long long)layer * 2 * g.half_elems;
    p.kv_off = g.half_elems;
    if (d->dtype == KVC_I8) {
        const long long half_rows = g.half_elems / d->head_dim;
        p.scales = reinterpret_cast<float*>(static_cast<char*>(cache) + (size_t)d->layers * 2 * (size_t)g.half_elems);
        p.sc_layer_off = (long long)layer * 2 * half_rows;
        p.sc_kv_off = half_rows;
    }
    p.B = d->batch;
    p.Hkv = d->kv_heads;
    p.D = d->head_dim;
    p.n_new = n_new;
    p.layout = d->layout;
    p.window = d->window;
    p.sinks = d->layout == KVC_LAYOUT_SINK_RING ? d->sinks : 0;
    p.capacity = g.C;
    p.bs = d->block_size;
    p.num_blocks = d->num_blocks;
    p.maxb = d->max_blocks_per_seq;
    p.rope = d->rope;
    if (d->rope == KVC_ROPE_BAKED) fill_theta(d->head_dim, d->rope_base, p.theta, nullptr);
    if (launch_append(d->dtype, p, (cudaStream_t)stream) != cudaSuccess) return KVC_ERR_CUDA;
    return KVC_OK;
}

namespace {
// Staging area of kvc_prefill (the chunk's K and V rows, bf16), after the
// decode workspace.
size_t prefill_stage_offset(const kvc_desc* d, const Geo& g) { return align_up(ws_layout(d, g).total, 256); }
size_t prefill_stage_bytes(const kvc_desc* d, long long T) {
    return 2 * (size_t)d->batch * (size_t)T * (size_t)d->kv_heads * (size_t)d->head_dim * 2;
}
}  // namespace

KVC_API size_t kvc_prefill_workspace_bytes(const kvc_desc* d, int32_t T) {
    Geo g;
    if (check_desc(d, &g) != KVC_OK || T < 1) return 0;
    return prefill_stage_offset(d, g) + prefill_stage_bytes(d, T);
}

KVC_API int kvc_prefill(const kvc_desc* d, void* cache, int32_t layer, const void* q, const void* k_new,
                        const void* v_new, int32_t T, const int32_t* pos0, const int32_t* block_table,
                        const uint32_t* valid_bits, void* out, void* workspace, size_t workspace_bytes,
                        void* stream) {
    Geo g;
    int rc = check_desc(d, &g);
    if (rc) return rc;
    if (d->dtype == KVC_F32) return KVC_ERR_UNSUPPORTED;
    const bool q8 = d->dtype == KVC_I8;
    const bool paged_l = d->layout == KVC_LAYOUT_PAGED;
    // the warp-specialised kernel: 128-row Q tiles of whole GQA groups, paged
    // blocks that pack a 64-key tile, chunks no longer than the window
    const bool ws_kernel = 128 % g.G == 0 &&
                           (paged_l ? (d->block_size % 8 == 0 && 64 % d->block_size == 0) : T <= d->window);
    if (!ws_kernel && (q8 || (d->head_dim != 64 && d->head_dim != 128) || g.G > 64)) return KVC_ERR_UNSUPPORTED;
    if (!cache || !q || !k_new || !v_new || !pos0 || !out || !workspace) return KVC_ERR_NULL;
    const bool paged = d->layout == KVC_LAYOUT_PAGED;
    if (paged && !block_table) return KVC_ERR_NULL;
    if (!aligned16(cache) || !aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out) ||
        !aligned16(workspace))
        return KVC_ERR_ALIGN;
    if (layer < 0 || layer >= d->layers || T < 1 || T > 0x7fffffff / 2) return KVC_ERR_ARG;
    if (workspace_bytes < kvc_prefill_workspace_bytes(d, T)) return KVC_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    const WorkspaceLayout w = ws_layout(d, g);
    cudaStream_t s = (cudaStream_t)stream;
    void* kst = ws + prefill_stage_offset(d, g);
    void* vst = static_cast<char*>(kst) + prefill_stage_bytes(d, T) / 2;

    AppendParams ap{};
    ap.cache = cache;
    ap.k_new = k_new;
    ap.v_new = v_new;
    ap.pos = pos0;
    ap.table = block_table;
    ap.err = reinterpret_cast<uint32_t*>(ws + w.err);
    ap.layer_off = (long long)layer * 2 * g.half_elems;
    ap.kv_off = g.half_elems;
    ap.B = d->batch;
    ap.Hkv = d->kv_heads;
    ap.D = d->head_dim;
    ap.n_new = T;
    ap.layout = d->layout;
    ap.window = d->window;
    ap.sinks = d->layout == KVC_LAYOUT_SINK_RING ? d->sinks : 0;
    ap.capacity = g.C;
    ap.bs = d->block_size;
    ap.num_blocks = d->num_blocks;
    ap.maxb = d->max_blocks_per_seq;
    ap.rope = d->rope;
    if (d->rope == KVC_ROPE_BAKED) fill_theta(d->head_dim, d->rope_base, ap.theta, nullptr);
    const long long half_rows = g.half_elems / d->head_dim;
    if (q8) {
        ap.scales = reinterpret_cast<float*>(static_cast<char*>(cache) + (size_t)d->layers * 2 * (size_t)g.half_elems);
        ap.sc_layer_off = (long long)layer * 2 * half_rows;
        ap.sc_kv_off = half_rows;
    }
    // the warp-specialised kernel's maps, encoded before anything is launched
    PrefillMaps pm;
    std::memset(&pm, 0, sizeof(pm));
    if (ws_kernel) {
        if (q8) {
            if ((rc = encode_q8_code_map(d, g, cache, paged_l ? d->block_size : 64, paged_l ? &pm.block : &pm.slot)))
                return rc;
        } else if (paged_l) {
            if ((rc = encode_block_map(d, g, cache, &pm.block))) return rc;
        } else {
            KvTensorMaps km;
            if ((rc = kv_maps_for(d, g, cache, &km, &pm.slot_whole))) return rc;
            pm.slot = km.run[kRunMaps - 1];                 // 64-row runs
        }
        if ((rc = encode_stage_map(d, kst, T, prefill_stage_bytes(d, T) / 2, &pm.stage))) return rc;
    }
    // 1. the chunk's rows as the cache will hold them (INT8: as it reads them back)
    if (launch_prefill_stage(ap, kst, vst, s) != cudaSuccess) return KVC_ERR_CUDA;
    // 2. attention: earlier keys from the cache as it stands, the chunk's from the stage
    PrefillParams pp{};
    pp.cache = cache;
    pp.q = q;
    pp.kst = kst;
    pp.vst = vst;
    pp.pos0 = pos0;
    pp.table = block_table;
    pp.valid = valid_bits;
    pp.out = out;
    pp.err = ap.err;
    pp.layer_off = ap.layer_off;
    pp.kv_off = ap.kv_off;
    pp.B = d->batch;
    pp.T = T;
    pp.Hq = d->q_heads;
    pp.Hkv = d->kv_heads;
    pp.G = g.G;
    pp.layout = d->layout;
    pp.window = d->window;
    pp.sinks = ap.sinks;
    pp.capacity = g.C;
    pp.bs = d->block_size;
    pp.num_blocks = d->num_blocks;
    pp.maxb = d->max_blocks_per_seq;
    pp.rope = d->rope;
    pp.layer = layer;
    const float scale = d->softmax_scale > 0.f ? d->softmax_scale : 1.0f / std::sqrt((float)d->head_dim);
    pp.q_scale = scale * 1.4426950408889634f;
    pp.scales = ap.scales;
    pp.sc_layer_off = ap.sc_layer_off;
    pp.sc_kv_off = ap.sc_kv_off;
    pp.half_rows = half_rows;
    if (d->rope != KVC_ROPE_NONE) fill_theta(d->head_dim, d->rope_base, pp.theta, nullptr);
    if (ws_kernel) {
        if (launch_prefill_ws(d->head_dim, q8, pp, pm, s) != cudaSuccess) return KVC_ERR_CUDA;
    } else if (launch_prefill(d->head_dim, g.G, pp, s) != cudaSuccess) {
        return KVC_ERR_CUDA;
    }
    // 3. the chunk appended
    if (launch_append(d->dtype, ap, s) != cudaSuccess) return KVC_ERR_CUDA;
    return KVC_OK;
}

KVC_API int kvc_decode_attention(const kvc_desc* d, const void* cache, int32_t layer, const void* q,
                                 const int32_t* pos, const int32_t* block_table, const uint32_t* valid_bits,
                                 void* out, void* workspace, size_t workspace_bytes, void* stream) {
    return decode_impl(d, cache, layer, q, nullptr, nullptr, pos, block_table, valid_bits, out, workspace,
                       workspace_bytes, stream);
}

KVC_API int kvc_decode_step(const kvc_desc* d, void* cache, int32_t layer, const void* q, const void* k_new,
                            const void* v_new, const int32_t* pos, const int32_t* block_table,
                            const uint32_t* valid_bits, void* out, void* workspace, size_t workspace_bytes,
                            void* stream) {
    Geo g;
    int rc = check_desc(d, &g);
    if (rc) return rc;
    if (!k_new || !v_new) return KVC_ERR_NULL;
    if (!aligned16(k_new) || !aligned16(v_new)) return KVC_ERR_ALIGN;
    if (d->dtype != KVC_F32 || d->layout == KVC_LAYOUT_PAGED) {
        // no separate append launch: the decode kernel (bf16 / INT8 ring / sink+ring)
        // or the paged plan kernel writes the new token itself
        return decode_impl(d, cache, layer, q, k_new, v_new, pos, block_table, valid_bits, out, workspace,
                           workspace_bytes, stream);
    }
    // the attention's own arguments are checked before the append launches
    if ((rc = decode_args(d, cache, layer, q, pos, block_table, out))) return rc;
    if (!workspace) return KVC_ERR_NULL;
    if (!aligned16(workspace)) return KVC_ERR_ALIGN;
    if (workspace_bytes < ws_layout(d, g).total) return KVC_ERR_WORKSPACE;
    rc = kvc_append(d, cache, layer, k_new, v_new, 1, pos, block_table, workspace, workspace_bytes, stream);
    if (rc) return rc;
    return decode_impl(d, cache, layer, q, nullptr, nullptr, pos, block_table, valid_bits, out, workspace,
                       workspace_bytes, stream);
}

KVC_API int kvc_block_table_write(const kvc_desc* d, int32_t* block_table, uint32_t* valid_bits, int32_t n,
                                  const int32_t* seq, const int32_t* logical_block, const int32_t* physical_block,
                                  void* workspace, size_t workspace_bytes, void* stream) {
    Geo g;
    int rc = check_desc(d, &g);
    if (rc) return rc;
    if (d->layout != KVC_LAYOUT_PAGED) return KVC_ERR_DESC;
    if (n < 0) return KVC_ERR_ARG;
    if (n == 0) return KVC_OK;
    if (!block_table || !seq || !logical_block || !physical_block || !workspace) return KVC_ERR_NULL;
    if (!aligned16(workspace)) return KVC_ERR_ALIGN;
    const WorkspaceLayout w = ws_layout(d, g);
    if (workspace_bytes < w.total) return KVC_ERR_WORKSPACE;
    TableParams p{};
    p.table = block_table;
    p.valid = valid_bits;
    p.seq = seq;
    p.lb = logical_block;
    p.phys = physical_block;
    p.err = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + w.err);
    p.n = n;
    p.B = d->batch;
    p.maxb = d->max_blocks_per_seq;
    p.num_blocks = d->num_blocks;
    if (launch_table_write(p, (cudaStream_t)stream) != cudaSuccess) return KVC_ERR_CUDA;
    return KVC_OK;
}

KVC_API int kvc_valid_write(const kvc_desc* d, uint32_t* valid_bits, int32_t n, const int32_t* slot,
                            const int32_t* value, void* workspace, size_t workspace_bytes, void* stream) {
    Geo g;
    int rc = check_desc(d, &g);
    if (rc) return rc;
    if (d->layout != KVC_LAYOUT_PAGED) return KVC_ERR_DESC;
    if (n < 0) return KVC_ERR_ARG;
    if (n == 0) return KVC_OK;
    if (!valid_bits || !slot || !value || !workspace) return KVC_ERR_NULL;
    if (!aligned16(workspace)) return KVC_ERR_ALIGN;
    const WorkspaceLayout w = ws_layout(d, g);
    if (workspace_bytes < w.total) return KVC_ERR_WORKSPACE;
    TableParams p{};
    p.valid = valid_bits;
    p.phys = slot;
    p.value = value;
    p.err = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + w.err);
    p.n = n;
    p.num_blocks = d->num_blocks;
    if (launch_valid_write(p, (cudaStream_t)stream) != cudaSuccess) return KVC_ERR_CUDA;
    return KVC_OK;
}

KVC_API int kvc_block_prepare(const kvc_desc* d, void* cache, const int32_t* pos, int32_t* block_table,
                              uint32_t* valid_bits, int32_t* refcount, int32_t* free_list, int32_t* free_count,
                              void* workspace, size_t workspace_bytes, void* stream) {
    Geo g;
    int rc = check_desc(d, &g);
    if (rc) return rc;
    if (!cache || !pos || !block_table || !refcount || !free_list || !free_count) return KVC_ERR_NULL;
    if (!aligned16(cache)) return KVC_ERR_ALIGN;
    // the copy kernel's grid carries (layer, K|V, kv head) on y
    if ((long long)d->layers * 2 * d->kv_heads > 65535) return KVC_ERR_UNSUPPORTED;
    kvc::BlockParams p;
    if ((rc = block_params(d, g, workspace, workspace_bytes, &p))) return rc;
    p.cache = cache;
    if (d->dtype == KVC_I8)
        p.scales = reinterpret_cast<float*>(static_cast<char*>(cache) + (size_t)d->layers * 2 * (size_t)g.half_elems);
    p.pos = pos;
    p.table = block_table;
    p.valid = valid_bits;
    p.refcount = refcount;
    p.free_list = free_list;
    p.free_count = free_count;
    return launch_block_prepare(g.elt, p, (cudaStream_t)stream) == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

KVC_API int kvc_block_share(const kvc_desc* d, int32_t* block_table, int32_t* refcount, int32_t n,
                            const int32_t* src_seq, const int32_t* dst_seq, const int32_t* nblocks, void* workspace,
                            size_t workspace_bytes, void* stream) {
    Geo g;
    int rc = check_desc(d, &g);
    if (rc) return rc;
    if (n < 0) return KVC_ERR_ARG;
    if (n == 0) return KVC_OK;
    if (!block_table || !refcount || !src_seq || !dst_seq || !nblocks) return KVC_ERR_NULL;
    kvc::BlockParams p;
    if ((rc = block_params(d, g, workspace, workspace_bytes, &p))) return rc;
    p.table = block_table;
    p.refcount = refcount;
    p.src_seq = src_seq;
    p.dst_seq = dst_seq;
    p.nblocks = nblocks;
    return launch_block_share(p, n, (cudaStream_t)stream) == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

KVC_API int kvc_block_release(const kvc_desc* d, int32_t* block_table, uint32_t* valid_bits, int32_t* refcount,
                              int32_t* free_list, int32_t* free_count, int32_t n, const int32_t* seq,
                              void* workspace, size_t workspace_bytes, void* stream) {
    Geo g;
    int rc = check_desc(d, &g);
    if (rc) return rc;
    if (n < 0) return KVC_ERR_ARG;
    if (n == 0) return KVC_OK;
    if (!block_table || !refcount || !free_list || !free_count || !seq) return KVC_ERR_NULL;
    kvc::BlockParams p;
    if ((rc = block_params(d, g, workspace, workspace_bytes, &p))) return rc;
    p.table = block_table;
    p.valid = valid_bits;
    p.refcount = refcount;
    p.free_list = free_list;
    p.free_count = free_count;
    p.src_seq = seq;
    return launch_block_release(p, n, (cudaStream_t)stream) == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

KVC_API int kvc_get_error(void* workspace, void* stream) {
    if (!workspace) return KVC_ERR_NULL;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t bits = 0;
    if (cudaMemcpyAsync(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost, s) != cudaSuccess) return KVC_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVC_ERR_CUDA;
    if (bits && cudaMemsetAsync(workspace, 0, sizeof(bits), s) != cudaSuccess) return KVC_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVC_ERR_CUDA;
    return (int)(bits & 0x7fffffffu);
}

KVC_API const char* kvc_strerror(int code) {
    switch (code) {
        case KVC_OK: return "ok";
        case KVC_ERR_NULL: return "a required pointer is NULL";
        case KVC_ERR_DESC: return "inconsistent cache descriptor";
        case KVC_ERR_UNSUPPORTED:
            return "unsupported combination of head_dim, cache dtype, layout and RoPE mode for this call, "
                   "or past one of its launch limits";
        case KVC_ERR_ALIGN: return "pointer not 16-byte aligned";
        case KVC_ERR_WORKSPACE: return "workspace smaller than kvc_workspace_bytes()";
        case KVC_ERR_ARG: return "argument out of range";
        case KVC_ERR_CUDA: return "CUDA launch or runtime call failed";
        case KVC_ERR_TOO_LARGE: return "problem needs more scratch than KVC_NOALLOC_SCRATCH_BYTES";
        case (int)KVC_DEV_BAD_BLOCK: return "device: block table entry >= num_blocks";
        case (int)KVC_DEV_UNMAPPED_APPEND: return "device: append into an unmapped block";
        case (int)KVC_DEV_BAD_POSITION: return "device: position < 0 or beyond the block table";
        case (int)KVC_DEV_TIMEOUT: return "device: a bounded wait timed out";
        case (int)KVC_DEV_BAD_ENTRY: return "device: table/valid update entry out of range";
        case (int)KVC_DEV_INTERNAL: return "device: an internal index check failed (access skipped)";
        case (int)KVC_DEV_NO_FREE_BLOCK: return "device: no free block left for a new or copied block";
        default: return "unknown code";
    }
}

}  // extern "C"

// ---------------------------------------------------------------------------
// kvc_decode_attention_noalloc: kvc_decode_attention with the library's own
// fixed scratch array in place of a caller workspace, for callers that cannot
// allocate device memory.
// ---------------------------------------------------------------------------
namespace {

// Device scratch shared by every kvc_decode_attention_noalloc call on a GPU.
static __device__ __align__(256) unsigned char kvc_noalloc_scratch[KVC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
    unsigned long long ctx_id;   // unique id of the context the address belongs to
    void* ptr;
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Unique id of the calling thread's current context (0 when none is current
// yet), through the runtime's driver entry points.
unsigned long long current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext*);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<GetCurrentFn>(a);
            get_id = reinterpret_cast<GetIdFn>(b);
        }
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with that device current, once per device and context: a context that was
// torn down and created again (cudaDeviceReset) may hold the array at another
// address, and is looked up afresh.
int scratch_on_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchAddr& a = g_scratch_addr[dev];
    unsigned long long id = current_context_id();
    if (!a.ptr || id == 0 || id != a.ctx_id) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, kvc_noalloc_scratch) != cudaSuccess || !ptr) return KVC_ERR_CUDA;
        if (id == 0) id = current_context_id();   // the lookup made the context current
        a.ptr = ptr;
        a.ctx_id = id;
    }
    *out = a.ptr;
    return KVC_OK;
}

}  // namespace

extern "C" KVC_API int kvc_decode_attention_noalloc(const kvc_desc* d, const void* cache, int32_t layer,
                                                    const void* q, const int32_t* pos,
                                                    const int32_t* block_table, const uint32_t* valid_bits,
                                                    void* out, void* stream) {
    Geo g;
    int rc = check_desc(d, &g);
    if (rc) return rc;
    if ((rc = decode_args(d, cache, layer, q, pos, block_table, out))) return rc;
    const WorkspaceLayout w = ws_layout(d, g);
    if (w.total > (size_t)KVC_NOALLOC_SCRATCH_BYTES) return KVC_ERR_TOO_LARGE;
    void* scratch = nullptr;
    rc = scratch_on_current_device(&scratch);
    if (rc) return rc;
    // error word and completion counters must start at zero
    if (cudaMemsetAsync(scratch, 0, w.part_ml, (cudaStream_t)stream) != cudaSuccess) return KVC_ERR_CUDA;
    return kvc_decode_attention(d, cache, layer, q, pos, block_table, valid_bits, out, scratch,
                                (size_t)KVC_NOALLOC_SCRATCH_BYTES, stream);
}
