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
// 16 exps. A quad of lanes owns one row; lane g streams states 4g..4g+3 (one 16-byte load and
// one 16-byte store, evict-first), so a warp moves 8 full rows of contiguous state, fully
// coalesced; A (per channel) comes through L2. The grid is (channel blocks, batch), so no
// lane divides. The readout is summed with two quad shuffles. bf16 tokens use the SFU exp2 and
// the fitted softplus of the scan; fp32 tokens use the accurate library functions.
//
// Successive decode steps of a model are dependent launches on one stream. The kernel is
// launched with programmatic stream serialization: it lets the next launch in the stream
// start its setup at once and waits (griddepcontrol.wait) for every earlier grid to complete
// and publish its memory before it reads anything, so the launch latency of layer l+1 hides
// under layer l without changing what either computes.
#include "selscan_device.cuh"
#include "selscan_launch.h"

namespace selscan {

constexpr int kUpdThreads = 256;
constexpr int kConvWidth = 4;  // taps of the short convolution (one per lane of a quad)

template <typename Tin>
__device__ __forceinline__ void load4(const Tin* p, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&v)[4]) {
    const float4 r = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[4]) {
    const uint2 r = __ldg(reinterpret_cast<const uint2*>(p));
    v[0] = bf16lo(r.x); v[1] = bf16hi(r.x); v[2] = bf16lo(r.y); v[3] = bf16hi(r.y);
}

// Zero-order hold: Bbar = Delta*B * phi(x), phi(x) = (exp(x) - 1)/x with x = Delta*A. fp32
// tokens take expm1 from the library; bf16 tokens the Taylor series below |x| = 1/16 and
// (abar - 1)/(A*Delta) above it, as in the scan.
__device__ __forceinline__ float upd_phi_exact(float m, float x) { return x != 0.f ? m / x : 1.f; }
__device__ __forceinline__ float upd_phi_fast(float x, float abar, float a, float dinv) {
    const float p = fmaf(fmaf(fmaf(x, 1.f / 24.f, 1.f / 6.f), x, 0.5f), x, 1.f);
    return fabsf(x) < 0.0625f ? p : (abar - 1.f) / a * dinv;
}

// kConv: first the decode step of the block's short causal convolution (width 4 = the quad:
// lane g holds tap g of the window, the window moves by one quad shuffle and the four taps are
// summed by two), whose output is the input x of the state update. kSsm: the state update.
template <typename Tin, typename Tout, bool kPrecise, bool kZoh, bool kConv, bool kSsm>
__global__ void __launch_bounds__(kUpdThreads) state_update_kernel(const UpdateArgs a) {
    // Wait for earlier grids in the stream (a no-op without programmatic serialization),
    // then let the next one begin its launch.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int64_t b = blockIdx.y;
    const int64_t d_raw = ((int64_t)blockIdx.x * kUpdThreads + threadIdx.x) >> 2;
    const int g = threadIdx.x & 3;
    const bool active = d_raw < a.dim;
    const int64_t d = active ? d_raw : 0;
    const int64_t row = b * a.dim + d;

    // Every load is issued before any store: the state stream starts at once and nothing
    // waits on a possible alias of the convolution window.
    float4* const sp = reinterpret_cast<float4*>(a.state + row * kN + 4 * g);
    float4 h = make_float4(0.f, 0.f, 0.f, 0.f), A4 = h;
    float Bv[4] = {0.f, 0.f, 0.f, 0.f}, Cv[4] = {0.f, 0.f, 0.f, 0.f};
    float xdt = 0.f, zv = 0.f, Dd = 0.f;
    if (kSsm) {
        h = __ldcs(sp);
        A4 = __ldg(reinterpret_cast<const float4*>(a.A + d * kN + 4 * g));
        load4<Tin>(static_cast<const Tin*>(a.B) + b * kN + 4 * g, Bv);
        load4<Tin>(static_cast<const Tin*>(a.C) + b * kN + 4 * g, Cv);
        xdt = to_f32(static_cast<const Tin*>(a.dt)[row]) + (a.dt_bias ? a.dt_bias[d] : 0.f);
        zv = a.z ? to_f32(static_cast<const Tin*>(a.z)[row]) : 0.f;
        Dd = a.D ? a.D[d] : 0.f;
    }

    float x;
    if (kConv) {
        Tin* const cs = static_cast<Tin*>(a.conv_state) + row * kConvWidth + g;
        const float s_old = to_f32(*cs);
        const float x_in = to_f32(static_cast<const Tin*>(a.x)[row]);
        const float w = a.conv_weight[d * kConvWidth + g];
        const float cb = a.conv_bias ? a.conv_bias[d] : 0.f;
        // Window oldest first: the new window is old[1..3] followed by the new input.
        const float s_next = __shfl_down_sync(0xffffffffu, s_old, 1, kConvWidth);
        const float s_new = g == kConvWidth - 1 ? x_in : s_next;
        float acc = w * s_new;
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += cb;
        if (a.conv_silu) acc = kPrecise ? silu_f<true>(acc) : silu2(make_float2(acc, acc)).x;
        x = acc;
        if (active) {
            *cs = from_f32<Tin>(s_new);  // a copy of an input value: exact
            if (a.conv_out && g == 0) static_cast<Tin*>(a.conv_out)[row] = from_f32<Tin>(acc);
        }
        if (!kSsm) return;
    } else {
        x = to_f32(static_cast<const Tin*>(a.x)[row]);
    }

    float dt;
    if (!a.softplus) dt = xdt;
    else if (kPrecise) dt = softplus_f<true>(xdt);
    else dt = softplus2(make_float2(xdt, xdt)).x;
    const float k = dt * x;

    const float Av[4] = {A4.x, A4.y, A4.z, A4.w};
    float hv[4] = {h.x, h.y, h.z, h.w};
    if (kPrecise) {
        // exp(Delta*A) h = h + expm1(Delta*A) h: the decay's distance from 1 keeps full
        // relative precision over thousands of generated tokens.
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const float xa = dt * Av[n];
            const float m = expm1f(xa);
            const float f = kZoh ? upd_phi_exact(m, xa) : 1.f;
            hv[n] = fmaf(m, hv[n], hv[n]) + k * Bv[n] * f;
        }
    } else {
        const float s = dt * kLog2e;
        const float dinv = kZoh ? rcp_approx(dt) : 0.f;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const float ab = ex2_approx(s * Av[n]);
            const float f = kZoh ? upd_phi_fast(dt * Av[n], ab, Av[n], dinv) : 1.f;
            hv[n] = fmaf(ab, hv[n], k * Bv[n] * f);
        }
    }
    h = make_float4(hv[0], hv[1], hv[2], hv[3]);
    float y = Cv[0] * h.x;
    y = fmaf(Cv[1], h.y, y);
    y = fmaf(Cv[2], h.z, y);
    y = fmaf(Cv[3], h.w, y);
    y += __shfl_xor_sync(0xffffffffu, y, 1);
    y += __shfl_xor_sync(0xffffffffu, y, 2);
    if (!active) return;
    __stcs(sp, h);
    if (g == 0) {
        y = fmaf(Dd, x, y);
        if (a.z) y *= kPrecise ? silu_f<true>(zv) : silu2(make_float2(zv, zv)).x;
        static_cast<Tout*>(a.out)[row] = from_f32<Tout>(y);
    }
}

template <typename Tin, typename Tout, bool kPrecise, bool kZoh, bool kConv, bool kSsm>
static cudaError_t launch_one(const UpdateArgs& a, int64_t batch, cudaStream_t stream) {
    const int64_t lanes = a.dim * 4;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)((lanes + kUpdThreads - 1) / kUpdThreads), (unsigned)batch, 1);
    cfg.blockDim = dim3(kUpdThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, state_update_kernel<Tin, Tout, kPrecise, kZoh, kConv, kSsm>, a);
}

template <typename Tin, typename Tout, bool kPrecise>
static cudaError_t launch_mode(const UpdateArgs& a, int64_t batch, cudaStream_t stream) {
    if (a.conv_state && !a.state)  // convolution step only
        return launch_one<Tin, Tout, kPrecise, false, true, false>(a, batch, stream);
    if (a.conv_state)
        return a.zoh ? launch_one<Tin, Tout, kPrecise, true, true, true>(a, batch, stream)
                     : launch_one<Tin, Tout, kPrecise, false, true, true>(a, batch, stream);
    return a.zoh ? launch_one<Tin, Tout, kPrecise, true, false, true>(a, batch, stream)
                 : launch_one<Tin, Tout, kPrecise, false, false, true>(a, batch, stream);
}

cudaError_t launch_state_update(const UpdateArgs& a, bool in_bf16, bool out_bf16,
                                cudaStream_t stream) {
    using bf = __nv_bfloat16;
    const int64_t batch = a.rows / a.dim;
    cudaError_t e;
    if (in_bf16) {
        e = out_bf16 ? launch_mode<bf, bf, false>(a, batch, stream)
                     : launch_mode<bf, float, false>(a, batch, stream);
    } else {
        e = out_bf16 ? launch_mode<float, bf, true>(a, batch, stream)
                     : launch_mode<float, float, true>(a, batch, stream);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace selscan
