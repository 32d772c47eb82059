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
// 16 exps. A quad of lanes owns one row (two when that keeps the grid to one wave of CTAs);
// lane g streams states 4g..4g+3 (one 16-byte load and one 16-byte store per row, evict-first),
// so a warp moves 8 full rows of contiguous state per load, fully coalesced; A (per channel)
// comes through L2. The grid is (channel blocks, batch), so no lane divides. The readout is
// summed with two quad shuffles. bf16 tokens use the SFU exp2 and the fitted softplus of the
// scan; fp32 tokens use the accurate library functions.
//
// Successive decode steps of a model are dependent launches on one stream, each too short to
// hide its own load latency. The kernel is launched with programmatic stream serialization:
// the next launch in the stream may start while this one runs, and before it waits
// (griddepcontrol.wait) for every earlier grid to complete and publish its memory, each CTA
// asks for its state and token inputs to be brought into L2, so the latency of reading them
// overlaps the grids before it without changing what either computes.
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

// L2 prefetch of [p, p + bytes) (16-byte aligned, a multiple of 16 bytes). Only a hint, so it
// may run before the grid dependency wait: L2 is the device's point of coherence, and a write
// by an earlier grid after the prefetch updates the lines it brought in.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// kConv: first the decode step of the block's short causal convolution (width 4 = the quad:
// lane g holds tap g of the window, the window moves by one quad shuffle and the four taps are
// summed by two), whose output is the input x of the state update. kSsm: the state update.
// kRq rows per quad: a CTA covers 64 kRq consecutive channels of one batch; row j of quad q of
// warp w is channel 64 kRq blockIdx.x + 8 kRq w + 8 j + q, so each of a warp's row loads moves 8
// whole consecutive states (512 bytes). Every load of every row is issued before any compute.
template <typename Tin, typename Tout, bool kPrecise, bool kZoh, bool kConv, bool kSsm, int kRq>
__global__ void __launch_bounds__(kUpdThreads) state_update_kernel(const UpdateArgs a) {
    constexpr int kRowsPerCta = (kUpdThreads / 4) * kRq;
    const int64_t b = blockIdx.y;
    const int64_t dcta = (int64_t)blockIdx.x * kRowsPerCta;
    // A launch that fills most of the GPU in one wave lets the next grid in the stream start
    // at once, so that grid's prefetch below overlaps this one's whole run; otherwise the next
    // grid may start once this one's wait is over.
    if (a.early_trigger) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Start bringing this CTA's state and token inputs into L2 while the grids before it
    // finish: a prefetch is only a hint, so it may come before the wait below (L2 is the
    // device's point of coherence: a write by an earlier grid after the prefetch updates the
    // lines it brought in). The state range starts at a multiple of 64 bytes of a 16-byte
    // aligned array; a token-input range is taken when its start and size are multiples of 16
    // bytes, as the bulk prefetch requires.
    if (kSsm && threadIdx.x == 0 && dcta < a.dim) {
        const int64_t nrows = min((int64_t)kRowsPerCta, a.dim - dcta);
        const int64_t r0 = b * a.dim + dcta;
        prefetch_l2(a.state + r0 * kN, (uint32_t)(nrows * kN * sizeof(float)));
        const uint32_t nin = (uint32_t)(nrows * sizeof(Tin));
        const Tin* in[3] = {static_cast<const Tin*>(a.x) + r0, static_cast<const Tin*>(a.dt) + r0,
                            a.z ? static_cast<const Tin*>(a.z) + r0 : nullptr};
#pragma unroll
        for (int i = 0; i < 3; ++i)
            if (in[i] && ((reinterpret_cast<uintptr_t>(in[i]) | nin) & 15u) == 0) prefetch_l2(in[i], nin);
    }
    // Wait for earlier grids in the stream (a no-op without programmatic serialization).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!a.early_trigger) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int warp = threadIdx.x >> 5, quad = (threadIdx.x & 31) >> 2;
    const int g = threadIdx.x & 3;
    bool active[kRq];
    int64_t d[kRq], row[kRq];
#pragma unroll
    for (int j = 0; j < kRq; ++j) {
        const int64_t d_raw = dcta + 8 * kRq * warp + 8 * j + quad;
        active[j] = d_raw < a.dim;
        d[j] = active[j] ? d_raw : 0;  // inactive rows compute on channel 0 and store nothing
        row[j] = b * a.dim + d[j];
    }

    // Every load is issued before any store: the state stream starts at once and nothing
    // waits on a possible alias of the convolution window.
    float4 h[kRq], A4[kRq];
    float Bv[4] = {0.f, 0.f, 0.f, 0.f}, Cv[4] = {0.f, 0.f, 0.f, 0.f};
    float xdt[kRq], zv[kRq], Dd[kRq];
#pragma unroll
    for (int j = 0; j < kRq; ++j) {
        h[j] = A4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        xdt[j] = zv[j] = Dd[j] = 0.f;
    }
    if (kSsm) {
#pragma unroll
        for (int j = 0; j < kRq; ++j)
            h[j] = __ldcs(reinterpret_cast<const float4*>(a.state + row[j] * kN + 4 * g));
#pragma unroll
        for (int j = 0; j < kRq; ++j) {
            A4[j] = __ldg(reinterpret_cast<const float4*>(a.A + d[j] * kN + 4 * g));
            xdt[j] = to_f32(static_cast<const Tin*>(a.dt)[row[j]]) + (a.dt_bias ? a.dt_bias[d[j]] : 0.f);
            zv[j] = a.z ? to_f32(static_cast<const Tin*>(a.z)[row[j]]) : 0.f;
            Dd[j] = a.D ? a.D[d[j]] : 0.f;
        }
        load4<Tin>(static_cast<const Tin*>(a.B) + b * kN + 4 * g, Bv);
        load4<Tin>(static_cast<const Tin*>(a.C) + b * kN + 4 * g, Cv);
    }

    float x[kRq];
    if (kConv) {
        float s_old[kRq], x_in[kRq], w[kRq], cb[kRq];
#pragma unroll
        for (int j = 0; j < kRq; ++j) {
            const Tin* cs = static_cast<const Tin*>(a.conv_state) + row[j] * kConvWidth + g;
            s_old[j] = to_f32(*cs);
            x_in[j] = to_f32(static_cast<const Tin*>(a.x)[row[j]]);
            w[j] = a.conv_weight[d[j] * kConvWidth + g];
            cb[j] = a.conv_bias ? a.conv_bias[d[j]] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < kRq; ++j) {
            // Window oldest first: the new window is old[1..3] followed by the new input.
            const float s_next = __shfl_down_sync(0xffffffffu, s_old[j], 1, kConvWidth);
            const float s_new = g == kConvWidth - 1 ? x_in[j] : s_next;
            float acc = w[j] * s_new;
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            acc += cb[j];
            if (a.conv_silu) acc = kPrecise ? silu_f<true>(acc) : silu2(make_float2(acc, acc)).x;
            x[j] = acc;
            if (active[j]) {
                Tin* cs = static_cast<Tin*>(a.conv_state) + row[j] * kConvWidth + g;
                *cs = from_f32<Tin>(s_new);  // a copy of an input value: exact
                if (a.conv_out && g == 0) static_cast<Tin*>(a.conv_out)[row[j]] = from_f32<Tin>(acc);
            }
        }
        if (!kSsm) return;
    } else {
#pragma unroll
        for (int j = 0; j < kRq; ++j) x[j] = to_f32(static_cast<const Tin*>(a.x)[row[j]]);
    }

#pragma unroll
    for (int j = 0; j < kRq; ++j) {
        float dt;
        if (!a.softplus) dt = xdt[j];
        else if (kPrecise) dt = softplus_f<true>(xdt[j]);
        else dt = softplus2(make_float2(xdt[j], xdt[j])).x;
        const float k = dt * x[j];

        const float Av[4] = {A4[j].x, A4[j].y, A4[j].z, A4[j].w};
        float hv[4] = {h[j].x, h[j].y, h[j].z, h[j].w};
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
        const float4 hn = make_float4(hv[0], hv[1], hv[2], hv[3]);
        float y = Cv[0] * hn.x;
        y = fmaf(Cv[1], hn.y, y);
        y = fmaf(Cv[2], hn.z, y);
        y = fmaf(Cv[3], hn.w, y);
        y += __shfl_xor_sync(0xffffffffu, y, 1);
        y += __shfl_xor_sync(0xffffffffu, y, 2);
        if (!active[j]) continue;
        __stcs(reinterpret_cast<float4*>(a.state + row[j] * kN + 4 * g), hn);
        if (g == 0) {
            y = fmaf(Dd[j], x[j], y);
            if (a.z) y *= kPrecise ? silu_f<true>(zv[j]) : silu2(make_float2(zv[j], zv[j])).x;
            static_cast<Tout*>(a.out)[row[j]] = from_f32<Tout>(y);
        }
    }
}

template <typename Tin, typename Tout, bool kPrecise, bool kZoh, bool kConv, bool kSsm, int kRq>
static cudaError_t launch_rq(const UpdateArgs& a, int64_t batch, cudaStream_t stream) {
    constexpr int64_t kRowsPerCta = (kUpdThreads / 4) * kRq;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)((a.dim + kRowsPerCta - 1) / kRowsPerCta), (unsigned)batch, 1);
    cfg.blockDim = dim3(kUpdThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, state_update_kernel<Tin, Tout, kPrecise, kZoh, kConv, kSsm, kRq>, a);
}

// CTAs of a kernel resident per SM (queried once per kernel).
template <typename Tin, typename Tout, bool kPrecise, bool kZoh, bool kConv, bool kSsm, int kRq>
static int resident_ctas() {
    static const int n = [] {
        int v = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &v, state_update_kernel<Tin, Tout, kPrecise, kZoh, kConv, kSsm, kRq>, kUpdThreads,
                0) != cudaSuccess) {
            cudaGetLastError();
            v = 0;
        }
        return v;
    }();
    return n;
}

// One row per quad, unless that grid needs a second wave of CTAs and the grid of two rows per
// quad fits in one: a small second wave would add a whole load latency to the step. The next
// grid is let in early when this one is a single wave over more than half of its CTA slots.
template <typename Tin, typename Tout, bool kPrecise, bool kZoh, bool kConv, bool kSsm>
static cudaError_t launch_one(const UpdateArgs& a, int64_t batch, cudaStream_t stream) {
    const int64_t slots1 = (int64_t)a.sms * resident_ctas<Tin, Tout, kPrecise, kZoh, kConv, kSsm, 1>();
    const int64_t slots2 = (int64_t)a.sms * resident_ctas<Tin, Tout, kPrecise, kZoh, kConv, kSsm, 2>();
    const int64_t ctas1 = (a.dim + kUpdThreads / 4 - 1) / (kUpdThreads / 4) * batch;
    const int64_t ctas2 = (a.dim + kUpdThreads / 2 - 1) / (kUpdThreads / 2) * batch;
    UpdateArgs b = a;
    if (ctas1 > slots1 && ctas2 <= slots2) {
        b.early_trigger = 2 * ctas2 > slots2 ? 1 : 0;
        return launch_rq<Tin, Tout, kPrecise, kZoh, kConv, kSsm, 2>(b, batch, stream);
    }
    b.early_trigger = ctas1 <= slots1 && 2 * ctas1 > slots1 ? 1 : 0;
    return launch_rq<Tin, Tout, kPrecise, kZoh, kConv, kSsm, 1>(b, batch, stream);
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
