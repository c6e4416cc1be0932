// Device-side building blocks shared by the kvc kernels: element
// conversion, RoPE angles, mbarrier / bulk-copy (TMA) wrappers with bounded
// waits, and the error word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvc_params.h"

namespace kvc {

// ---------------------------------------------------------------------------
// element types
// ---------------------------------------------------------------------------
template <typename Elt> struct EltTraits;
template <> struct EltTraits<float> {
    static constexpr int kBytes = 4;
    __device__ static __forceinline__ float to_f32(float x) { return x; }
    __device__ static __forceinline__ float from_f32(float x) { return x; }
    // unpack one 16-byte chunk (4 values)
    __device__ static __forceinline__ void unpack(const uint4& w, float* f) {
        f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y);
        f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
    }
};
template <> struct EltTraits<__nv_bfloat16> {
    static constexpr int kBytes = 2;
    __device__ static __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ static __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
    // bf16 is the high half of an fp32: a shift or a mask widens it exactly.
    __device__ static __forceinline__ void unpack(const uint4& w, float* f) {
        f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xffff0000u);
        f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xffff0000u);
        f[4] = __uint_as_float(w.z << 16); f[5] = __uint_as_float(w.z & 0xffff0000u);
        f[6] = __uint_as_float(w.w << 16); f[7] = __uint_as_float(w.w & 0xffff0000u);
    }
};

// ---------------------------------------------------------------------------
// errors
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bits) {
    if (err) atomicOr(err, bits);
}

// An index computed in a kernel failed its bounds check: KVC_DEV_INTERNAL,
// and the first failure's (site, value) kept in err[1], err[2].  The caller
// skips the access.
__device__ __forceinline__ void index_fault(uint32_t* err, uint32_t site, long long value) {
    if (!err) return;
    if ((atomicOr(err, 0x20u) & 0x20u) == 0u) {
        err[1] = site;
        err[2] = (uint32_t)value;
    }
}

// ---------------------------------------------------------------------------
// RoPE angle pos * theta_i, reduced exactly: the host passes
// F_i = theta_i / (2 pi) * 2^64 as an unsigned 64-bit fixed-point fraction of a
// turn; pos * F_i mod 2^64 (integer multiply, wraps) is the angle's fraction
// of a turn, whose top 32 bits, read as a signed number, place it in
// [-1/2, 1/2) turn.  Error: the rounding of F_i (2^-53 relative, ~1e-11 rad at
// pos = 2^20) plus one fp32 rounding (~2e-7 rad); fp32 pos * theta would be
// off by ~1e-2 rad at pos ~ 2.6e5, fp64 is slow on this part.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void rope_cos_sin(long long pos, unsigned long long turn_frac, float* c, float* s) {
    const unsigned long long ph = (unsigned long long)pos * turn_frac;     // mod 2^64
    const float turns = (float)(int)(unsigned)(ph >> 32) * 2.3283064365386963e-10f;   // 2^-32
    sincosf(turns * 6.283185307179586f, s, c);
}

// ---------------------------------------------------------------------------
// shared-memory mbarriers and 1-D bulk copies (cp.async.bulk, TMA engine)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// kWaitCycles SM clocks (about a second) and returns false; the caller sets
// KVC_DEV_TIMEOUT and stops using the pipeline.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitCycles) return false;
    }
    return true;
}

// Global -> shared bulk copy of `bytes` (multiple of 16, both ends 16-byte
// aligned); completion is counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Named barrier over the first `threads` threads of the block (id 1..15).
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}


}  // namespace kvc

namespace kvc {

// ---------------------------------------------------------------------------
// 2-D tensor copies (TMA) and tensor-core fragments for the bf16 kernel
// ---------------------------------------------------------------------------

// Box loads of a 4-D / 5-D tensor map at element coordinates (x, y, z, w[, v]).
__device__ __forceinline__ void tma_load_4d(void* dst_smem, const void* tmap, int x, int y, int z, int w,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];"
        ::"r"(smem_u32(dst_smem)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(w),
        "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_5d(void* dst_smem, const void* tmap, int x, int y, int z, int w, int v,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
        ::"r"(smem_u32(dst_smem)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(v),
        "r"(smem_u32(bar))
        : "memory");
}

// The same copies with an L2 cache policy (createpolicy): data read once per
// call is marked evict-first, so that streaming it does not push out what
// every call reads again (the kernels' code, block tables, partials, q).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_load_4d_hint(void* dst_smem, const void* tmap, int x, int y, int z, int w,
                                                 uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
        ::"r"(smem_u32(dst_smem)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(w),
        "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void tma_load_5d_hint(void* dst_smem, const void* tmap, int x, int y, int z, int w, int v,
                                                 uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;"
        ::"r"(smem_u32(dst_smem)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(v),
        "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) into L2: a
// hint, with no effect on what any load returns.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}

// D = A * B + D, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two floats -> one 32-bit register of two bf16 (lo = first), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// ---------------------------------------------------------------------------
// INT8 cache rows ([primer] 5.1, quantised cache).  Each stored row (one
// token's K or V for one kv head) keeps an fp32 scale s = max|x| / 127 and
// codes c = rint(x / s) clamped to +-127 (IEEE fp32 quotients, nearest, ties
// to even); it reads back as c * s.  A zero row keeps s = 0 and zero codes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int q8_code(float x, float s) {
    if (!(s > 0.f)) return 0;
    const float r = rintf(__fdiv_rn(x, s));
    return (int)fminf(fmaxf(r, -127.f), 127.f);
}

// Warp-wide quantisation of one row whose N values per lane are x: returns
// the row's scale (to every lane) and the lane's codes.
template <int N>
__device__ __forceinline__ float q8_quantize_lane(const float (&x)[N], int8_t (&c)[N]) {
    float a = 0.f;
#pragma unroll
    for (int k = 0; k < N; ++k) a = fmaxf(a, fabsf(x[k]));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    const float s = __fdiv_rn(a, 127.f);
#pragma unroll
    for (int k = 0; k < N; ++k) c[k] = (int8_t)q8_code(x[k], s);
    return s;
}

// One warp stores one token's K row (rotated at `pos` with baked RoPE) and V
// row of one kv head: bf16 sources kr / vr [D], code rows kc / vc, scales
// *ks / *vs.  Lane l handles the rotation pairs i = l + 32 m (columns i and
// i + D/2, NP = D / 64 pairs); its codes come back in kq / vq as
// [2m] = column i, [2m + 1] = column i + D/2, and the scales in sk / sv.
template <int NP>
__device__ __forceinline__ void q8_store_token_warp(const __nv_bfloat16* kr, const __nv_bfloat16* vr, int8_t* kc,
                                                    int8_t* vc, float* ks, float* vs, int rope, long long pos,
                                                    const unsigned long long* theta, int lane,
                                                    int8_t (&kq)[2 * NP], int8_t (&vq)[2 * NP], float* sk,
                                                    float* sv) {
    constexpr int HALF = 32 * NP;
    float kx[2 * NP], vx[2 * NP];
#pragma unroll
    for (int m = 0; m < NP; ++m) {
        const int i = lane + 32 * m;
        float x1 = __bfloat162float(kr[i]), x2 = __bfloat162float(kr[i + HALF]);
        if (rope == 1 /* baked */) {
            float c, s;
            rope_cos_sin(pos, theta[i], &c, &s);
            const float y1 = x1 * c - x2 * s, y2 = x1 * s + x2 * c;
            x1 = y1;
            x2 = y2;
        }
        kx[2 * m] = x1;
        kx[2 * m + 1] = x2;
        vx[2 * m] = __bfloat162float(vr[i]);
        vx[2 * m + 1] = __bfloat162float(vr[i + HALF]);
    }
    *sk = q8_quantize_lane<2 * NP>(kx, kq);
    *sv = q8_quantize_lane<2 * NP>(vx, vq);
#pragma unroll
    for (int m = 0; m < NP; ++m) {
        const int i = lane + 32 * m;
        kc[i] = kq[2 * m];
        kc[i + HALF] = kq[2 * m + 1];
        vc[i] = vq[2 * m];
        vc[i + HALF] = vq[2 * m + 1];
    }
    if (lane == 0) {
        *ks = *sk;
        *vs = *sv;
    }
}

// Two codes -> one register of two bf16 (lo: byte ka of a, hi: byte kb of
// b), exact.  a and b are code words with 0x80 xor-ed into every byte, so a
// byte holds c + 128; placed under the exponent of 2^23 it reads as the fp32
// 2^23 + 128 + c, from which 2^23 + 128 is subtracted.
__device__ __forceinline__ uint32_t q8_pair_bf16x2(uint32_t a, int ka, uint32_t b, int kb) {
    const float fa = __int_as_float(__byte_perm(a, 0x4B000000u, 0x7540u | (uint32_t)ka));
    const float fb = __int_as_float(__byte_perm(b, 0x4B000000u, 0x7540u | (uint32_t)kb));
    const float2 f = __fadd2_rn(make_float2(fa, fb), make_float2(-8388736.f, -8388736.f));
    return pack_bf16x2(f.x, f.y);
}

// D = A * B + D, m16n8k16, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two floats -> one register of two fp16 (lo = first), round to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Two codes -> one register of two fp16, exact.  w holds codes with 0x80
// xor-ed into every byte (a byte is c + 128); sel picks the bytes for the
// low and high halves into byte positions 0 and 2 and 0x64 into 1 and 3
// (0x4140: bytes 0 and 1 of w; 0x4342: bytes 2 and 3).  0x64uu is the fp16
// 1024 + uu, from which 1024 + 128 is subtracted.
__device__ __forceinline__ uint32_t q8_f16x2(uint32_t w, uint32_t sel) {
    uint32_t x = __byte_perm(w, 0x64646464u, sel);
    __half2 h = *reinterpret_cast<const __half2*>(&x);
    h = __hsub2(h, __half2half2(__ushort_as_half((unsigned short)0x6480u)));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// 3-D box load (TMA) at element coordinates (x, y, z).
__device__ __forceinline__ void tma_load_3d(void* dst_smem, const void* tmap, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];"
        ::"r"(smem_u32(dst_smem)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace kvc
