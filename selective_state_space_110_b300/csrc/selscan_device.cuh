// Device-side building blocks shared by the scan and state-update kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace selscan {

constexpr int kN = 16;  // state numbers per channel (Mamba's default state size)

constexpr float kLog2e = 1.4426950408889634f;

// 2^x on the SFU (MUFU.EX2), flush-to-zero. Max relative error about 2^-22.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// softplus(x) = log(1 + e^x). Above 20 the correction log1p(e^-x) < 2.1e-9 is below fp32
// resolution of x, so x is returned. kPrecise uses the accurate library exp; otherwise the
// SFU exp (relative error ~1e-7 in e^x, which log1p passes through unchanged).
template <bool kPrecise>
__device__ __forceinline__ float softplus_f(float x) {
    if (x > 20.f) return x;
    return kPrecise ? log1pf(expf(x)) : log1pf(__expf(x));
}

// silu(z) = z * sigmoid(z) = z / (1 + e^-z). For z -> -inf the denominator overflows to
// +inf and the fast divide returns 0, the correct limit.
template <bool kPrecise>
__device__ __forceinline__ float silu_f(float z) {
    return kPrecise ? z / (1.f + expf(-z)) : __fdividef(z, 1.f + __expf(-z));
}

// ---- fast softplus / silu on pairs (bf16 inputs; fp32 inputs use the exact library forms) ----

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

// softplus(x) = max(x, 0) + log1p(w), w = exp(-|x|) in (0, 1]; log1p(w) = w * P(w) with P a
// degree-6 polynomial fitted to log1p(w)/w on [0, 1] by least squares on Chebyshev nodes
// (fit_log1p.py in this directory); relative error below 1.4e-6 in addition to the SFU exp2's.
__device__ __forceinline__ float2 softplus2(float2 x) {
    const float2 na = __fmul2_rn(make_float2(fabsf(x.x), fabsf(x.y)), f2(-kLog2e));
    const float2 w = make_float2(ex2_approx(na.x), ex2_approx(na.y));
    float2 p = __ffma2_rn(w, f2(1.420607697e-02f), f2(-6.660313159e-02f));
    p = __ffma2_rn(p, w, f2(1.494590789e-01f));
    p = __ffma2_rn(p, w, f2(-2.351667285e-01f));
    p = __ffma2_rn(p, w, f2(3.311267793e-01f));
    p = __ffma2_rn(p, w, f2(-4.998728335e-01f));
    p = __ffma2_rn(p, w, f2(9.999988079e-01f));
    return __ffma2_rn(p, w, make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)));
}

// silu(z) = z / (1 + e^-z). For z -> -inf the denominator is +inf and the SFU reciprocal 0.
__device__ __forceinline__ float2 silu2(float2 z) {
    const float2 a = __fmul2_rn(z, f2(-kLog2e));
    const float2 den = __fadd2_rn(make_float2(ex2_approx(a.x), ex2_approx(a.y)), f2(1.f));
    return __fmul2_rn(z, make_float2(rcp_approx(den.x), rcp_approx(den.y)));
}

// ---- element loads / stores ---------------------------------------------------------------

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// bf16 pair in one 32-bit word (element 2i in the low half) -> two floats, exactly.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Load 8 consecutive elements p[0..7] into fp32. kVec: p is 16-byte aligned and all 8 are in
// range (one 128-bit load for bf16, two for fp32), streamed with evict-first.
// Otherwise element i is loaded only if i < nvalid, else 0.
template <typename T, bool kVec>
__device__ __forceinline__ void load8(const T* p, int nvalid, float (&v)[8]);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16, true>(const __nv_bfloat16* p, int nvalid,
                                                           float (&v)[8]) {
    if (nvalid >= 8) {
        uint4 r = __ldcs(reinterpret_cast<const uint4*>(p));
        v[0] = bf16lo(r.x); v[1] = bf16hi(r.x); v[2] = bf16lo(r.y); v[3] = bf16hi(r.y);
        v[4] = bf16lo(r.z); v[5] = bf16hi(r.z); v[6] = bf16lo(r.w); v[7] = bf16hi(r.w);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
}
template <>
__device__ __forceinline__ void load8<float, true>(const float* p, int nvalid, float (&v)[8]) {
    if (nvalid >= 8) {
        float4 a = __ldcs(reinterpret_cast<const float4*>(p));
        float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16, false>(const __nv_bfloat16* p, int nvalid,
                                                            float (&v)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = i < nvalid ? __bfloat162float(p[i]) : 0.f;
}
template <>
__device__ __forceinline__ void load8<float, false>(const float* p, int nvalid, float (&v)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = i < nvalid ? p[i] : 0.f;
}

// Store 8 consecutive outputs (same alignment / range contract as load8).
template <typename T, bool kVec>
__device__ __forceinline__ void store8(T* p, int nvalid, const float (&v)[8]);

template <>
__device__ __forceinline__ void store8<__nv_bfloat16, true>(__nv_bfloat16* p, int nvalid,
                                                            const float (&v)[8]) {
    if (nvalid >= 8) {
        uint4 r;
        __nv_bfloat162 t;
        t = __floats2bfloat162_rn(v[0], v[1]); r.x = *reinterpret_cast<uint32_t*>(&t);
        t = __floats2bfloat162_rn(v[2], v[3]); r.y = *reinterpret_cast<uint32_t*>(&t);
        t = __floats2bfloat162_rn(v[4], v[5]); r.z = *reinterpret_cast<uint32_t*>(&t);
        t = __floats2bfloat162_rn(v[6], v[7]); r.w = *reinterpret_cast<uint32_t*>(&t);
        __stcs(reinterpret_cast<uint4*>(p), r);
    }
}
template <>
__device__ __forceinline__ void store8<float, true>(float* p, int nvalid, const float (&v)[8]) {
    if (nvalid >= 8) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
        __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(v[4], v[5], v[6], v[7]));
    }
}
template <>
__device__ __forceinline__ void store8<__nv_bfloat16, false>(__nv_bfloat16* p, int nvalid,
                                                             const float (&v)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < nvalid) p[i] = __float2bfloat16_rn(v[i]);
}
template <>
__device__ __forceinline__ void store8<float, false>(float* p, int nvalid, const float (&v)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < nvalid) p[i] = v[i];
}

}  // namespace selscan
