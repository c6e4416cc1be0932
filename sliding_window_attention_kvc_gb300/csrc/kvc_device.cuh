// Device-side building blocks shared by the kvc kernels: element
// conversion, RoPE angles, mbarrier / bulk-copy (TMA) wrappers with bounded
// waits, and the error word.
#pragma once

#include <cuda_bf16.h>
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

// ---------------------------------------------------------------------------
// RoPE angle: pos * theta reduced to [-pi, pi] in fp64 (two-constant
// Cody-Waite reduction), then sin/cos in fp32.  Keeps the rotation accurate at
// positions of 10^5 - 10^6, where an fp32 product pos * theta would already
// be off by ~1e-2 rad.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void rope_cos_sin(double pos, double theta, float* c, float* s) {
    const double kInv2Pi = 0.15915494309189535;      // 1 / (2 pi)
    const double k2PiHi = 6.283185307179586;         // 2 pi rounded to fp64
    const double k2PiLo = 2.4492935982947064e-16;    // 2 pi - k2PiHi
    double a = pos * theta;
    double k = rint(a * kInv2Pi);
    double r = fma(-k, k2PiHi, a);
    r = fma(-k, k2PiLo, r);
    sincosf((float)r, s, c);
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

__device__ __forceinline__ float exp2_approx(float x) { return exp2f(x); }

}  // namespace kvc
