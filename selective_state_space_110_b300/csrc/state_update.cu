// Single-token state update (generation step) for sm_103a.
//
// One generated token updates every (b, d) state once ("Mamba and State Space Models",
// world.lapla.si, section "Taken Apart": the head reads one token, computes Delta, B and C,
// and the rods move once; section "What It Does": the state is updated once per token).
// The arithmetic is one step of the scan:
//   Delta = softplus(dt + dt_bias), h[n] = exp(Delta*A[d,n]) h[n] + Delta*B[b,n]*x,
//   y = (sum_n C[b,n] h[n] + D[d] x) * silu(z).
//
// The step is bound by HBM: per (b, d) it reads and writes 64 bytes of fp32 state and does
// 16 exps. Each quad of lanes owns one row; lane g streams states 4g..4g+3 (one 16-byte load
// and one 16-byte store), so a warp moves 8 full rows of contiguous state, fully coalesced.
// The 16-term readout is summed with two quad shuffles. Transcendentals use the accurate
// library functions (softplus via log1p, the decay via expm1): they hide under the traffic.
#include "selscan_device.cuh"
#include "selscan_launch.h"

namespace selscan {

constexpr int kUpdThreads = 256;

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kUpdThreads) state_update_kernel(const UpdateArgs a) {
    const int64_t q = (int64_t)blockIdx.x * kUpdThreads + threadIdx.x;
    const int g = threadIdx.x & 3;
    const int64_t row_raw = q >> 2;
    const bool active = row_raw < a.rows;
    const int64_t row = active ? row_raw : 0;
    const int64_t d = row % a.dim, b = row / a.dim;

    float4 h = *reinterpret_cast<const float4*>(a.state + row * kN + 4 * g);
    const float4 A4 = *reinterpret_cast<const float4*>(a.A + d * kN + 4 * g);
    const Tin* Bp = static_cast<const Tin*>(a.B) + b * kN + 4 * g;
    const Tin* Cp = static_cast<const Tin*>(a.C) + b * kN + 4 * g;
    const float x = to_f32(static_cast<const Tin*>(a.x)[row]);
    const float xdt = to_f32(static_cast<const Tin*>(a.dt)[row]) + (a.dt_bias ? a.dt_bias[d] : 0.f);
    const float dt = a.softplus ? softplus_f<true>(xdt) : xdt;
    const float k = dt * x;

    // exp(Delta*A) h = h + expm1(Delta*A) h: the decay's distance from 1 keeps full relative
    // precision, so thousands of generated tokens accumulate no bias from rounding Abar.
    h.x = fmaf(expm1f(dt * A4.x), h.x, h.x) + k * to_f32(Bp[0]);
    h.y = fmaf(expm1f(dt * A4.y), h.y, h.y) + k * to_f32(Bp[1]);
    h.z = fmaf(expm1f(dt * A4.z), h.z, h.z) + k * to_f32(Bp[2]);
    h.w = fmaf(expm1f(dt * A4.w), h.w, h.w) + k * to_f32(Bp[3]);
    float y = to_f32(Cp[0]) * h.x;
    y = fmaf(to_f32(Cp[1]), h.y, y);
    y = fmaf(to_f32(Cp[2]), h.z, y);
    y = fmaf(to_f32(Cp[3]), h.w, y);
    y += __shfl_xor_sync(0xffffffffu, y, 1);
    y += __shfl_xor_sync(0xffffffffu, y, 2);
    if (!active) return;
    *reinterpret_cast<float4*>(a.state + row * kN + 4 * g) = h;
    if (g == 0) {
        y = fmaf(a.D ? a.D[d] : 0.f, x, y);
        if (a.z) y *= silu_f<true>(to_f32(static_cast<const Tin*>(a.z)[row]));
        static_cast<Tout*>(a.out)[row] = from_f32<Tout>(y);
    }
}

cudaError_t launch_state_update(const UpdateArgs& a, bool in_bf16, bool out_bf16,
                                cudaStream_t stream) {
    using bf = __nv_bfloat16;
    const int64_t threads = a.rows * 4;
    const unsigned grid = (unsigned)((threads + kUpdThreads - 1) / kUpdThreads);
    if (in_bf16) {
        if (out_bf16) state_update_kernel<bf, bf><<<grid, kUpdThreads, 0, stream>>>(a);
        else state_update_kernel<bf, float><<<grid, kUpdThreads, 0, stream>>>(a);
    } else {
        if (out_bf16) state_update_kernel<float, bf><<<grid, kUpdThreads, 0, stream>>>(a);
        else state_update_kernel<float, float><<<grid, kUpdThreads, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace selscan
