// Chunked selective scan (S6 forward) for sm_103a.
//
// What is computed ("Mamba and State Space Models", world.lapla.si, sections "A State of
// Fixed Size", "Chosen by the Token" and "A Scan on the Chip"): per row (b, d) and token t,
//   Delta = softplus(delta + bias), h[n] = exp(Delta*A[d,n]) h[n] + Delta*B[b,n,t]*u,
//   y = (sum_n C[b,n,t] h[n] + D[d] u) * silu(z).
// As on that page, the inputs are read once from HBM, discretised and scanned on chip, and
// only y (plus the final state) is written back; the per-token state never leaves registers.
//
// Work decomposition (B300: 148 SMs, 4 schedulers each, 32 SFU ex2/clk/SM, 128 FP32
// lanes/clk/SM). The recurrence costs 16 exp2 and 64 FP32 lane-ops per (b, d, t), so the
// kernel is bound by the SFU and FMA pipes, not by HBM; the layout below is chosen to keep
// both pipes busy and every SM evenly loaded:
//   - A row (b, d) is owned by a quad of 4 lanes; lane g of the quad keeps states
//     4g..4g+3 in registers and updates them with packed f32x2 FMAs. A warp holds 8 rows,
//     a CTA (4 warps) 32 consecutive channels of one batch.
//   - The sequence is walked in chunks of 32 tokens. Per chunk the CTA stages B and C
//     (shared by all channels of the batch) into shared memory as fp32, once.
//   - Lane g loads tokens 8g..8g+7 of its row (one 128-bit load per tensor), computes
//     Delta and Delta*u there (once per element) and hands them to its quad through shared
//     memory. After the 32 steps the quad's partial readouts are summed through a swizzled
//     shared-memory transpose so lane g again owns tokens 8g..8g+7, where the D skip and
//     the silu gate are applied and y is stored with one 128-bit store.
//   - Long sequences with few rows are cut into time segments that run in parallel
//     (grid.y). A first pass (kLocalEnd) scans segments 0..S-2 from a zero state and keeps
//     only each segment's end state and its summed Delta. The full pass then starts
//     segment s from the true state, obtained by folding the earlier segments:
//     h <- exp(A * sum(Delta)) h + h_local_end (the associative combine of the recurrence).
#include "selscan_device.cuh"
#include "selscan_launch.h"

namespace selscan {

constexpr int kChunk = 32;               // tokens per chunk
constexpr int kWarps = 4;                // warps per CTA
constexpr int kThreads = kWarps * 32;    // 128
constexpr int kRowsPerWarp = 8;          // quads per warp
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;  // 32 channels
constexpr int kDkStride = 2 * kChunk + 4;  // floats per row of (Delta, k) pairs; +4 staggers
                                           // rows across bank groups

enum class Mode { kFull, kLocalEnd };

// B/C staging layout: s_bc[t][32] holds B[0..15] and C[0..15] of token t as eight 16-byte
// chunks. Even tokens store B in chunks 0..3 and C in 4..7, odd tokens the other way
// round. Lane g then reads its 4 B values at chunk g + 4*(t&1) and its 4 C values at
// chunk g + 4*(1-(t&1)): per token the warp touches 4 distinct chunks (conflict-free
// broadcast), the offsets are compile-time immediates once t is unrolled, and the staging
// stores of two adjacent tokens fall in disjoint bank groups.
__device__ __forceinline__ int bc_chunk_b(int g, int t) { return g + 4 * (t & 1); }
__device__ __forceinline__ int bc_chunk_c(int g, int t) { return g + 4 * (1 - (t & 1)); }

template <typename Tin, typename Tout, bool kVec, bool kPrecise, Mode kMode>
__global__ void __launch_bounds__(kThreads) scan_chunked_kernel(const ScanArgs a) {
    constexpr bool kFull = kMode == Mode::kFull;
    __shared__ __align__(16) float s_bc[2][kChunk][32];
    __shared__ __align__(16) float s_dk[kWarps][kRowsPerWarp][kDkStride];
    __shared__ __align__(16) float s_red[kFull ? kWarps : 1][kFull ? 8 * 32 * 4 : 4];

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int rl = lane >> 2;  // row within the warp
    const int g = lane & 3;    // quarter of the state owned by this lane
    const int64_t b = blockIdx.z;
    const int seg = blockIdx.y;
    const int64_t d = (int64_t)blockIdx.x * kRowsPerCta + warp * kRowsPerWarp + rl;
    const bool active = d < a.dim;
    const int64_t dc = active ? d : 0;
    const int64_t row = b * a.dim + dc;
    const int64_t L = a.seqlen;
    const int64_t t_begin = (int64_t)seg * a.seg_len;
    const int64_t t_end = min(L, t_begin + a.seg_len);
    const int nprev = a.nseg - 1;  // segments with a stored local end state

    // Per-lane constants: A for states 4g..4g+3 (pre-scaled by log2(e) for the SFU exp2).
    float4 A4 = *reinterpret_cast<const float4*>(a.A + dc * kN + 4 * g);
    if (!kPrecise) { A4.x *= kLog2e; A4.y *= kLog2e; A4.z *= kLog2e; A4.w *= kLog2e; }
    const float2 a01 = make_float2(A4.x, A4.y), a23 = make_float2(A4.z, A4.w);
    const float bias = a.delta_bias ? a.delta_bias[dc] : 0.f;
    const float Dd = a.D ? a.D[dc] : 0.f;

    // ---- initial state ----
    float2 h01 = make_float2(0.f, 0.f), h23 = make_float2(0.f, 0.f);
    if (kFull) {
        if (a.initial_state) {
            float4 s = *reinterpret_cast<const float4*>(a.initial_state + row * kN + 4 * g);
            h01 = make_float2(s.x, s.y); h23 = make_float2(s.z, s.w);
        }
        // Fold the local end states of the segments before this one.
        for (int j = 0; j < seg; ++j) {
            const float ds = a.ws_dsum[row * nprev + j];
            const float4 hl = *reinterpret_cast<const float4*>(a.ws_hloc + (row * nprev + j) * kN + 4 * g);
            if (kPrecise) {  // exp(A*S) h + h_local, with exp written as 1 + expm1
                const float m0 = expm1f(a01.x * ds), m1 = expm1f(a01.y * ds);
                const float m2 = expm1f(a23.x * ds), m3 = expm1f(a23.y * ds);
                h01 = make_float2(fmaf(m0, h01.x, h01.x) + hl.x, fmaf(m1, h01.y, h01.y) + hl.y);
                h23 = make_float2(fmaf(m2, h23.x, h23.x) + hl.z, fmaf(m3, h23.y, h23.y) + hl.w);
            } else {
                const float p0 = ex2_approx(a01.x * ds), p1 = ex2_approx(a01.y * ds);
                const float p2 = ex2_approx(a23.x * ds), p3 = ex2_approx(a23.y * ds);
                h01 = make_float2(fmaf(p0, h01.x, hl.x), fmaf(p1, h01.y, hl.y));
                h23 = make_float2(fmaf(p2, h23.x, hl.z), fmaf(p3, h23.y, hl.w));
            }
        }
    }

    const Tin* __restrict__ u_row = static_cast<const Tin*>(a.u) + row * L;
    const Tin* __restrict__ d_row = static_cast<const Tin*>(a.delta) + row * L;
    const Tin* __restrict__ z_row = a.z ? static_cast<const Tin*>(a.z) + row * L : nullptr;
    Tout* __restrict__ o_row = static_cast<Tout*>(a.out) + row * L;
    const Tin* __restrict__ Bb = static_cast<const Tin*>(a.B) + b * kN * L;
    const Tin* __restrict__ Cb = static_cast<const Tin*>(a.C) + b * kN * L;

    float* dkrow = &s_dk[warp][rl][0];
    float dsum = 0.f, dsum_c = 0.f;  // Kahan sum of Delta (kLocalEnd)
    int buf = 0;

    for (int64_t t0 = t_begin; t0 < t_end; t0 += kChunk) {
        __syncwarp();
        // ---- stage B (and C) of this chunk: thread -> (token tt, state quad j) ----
        {
            const int tt = tid >> 2, j = tid & 3;
            const int64_t t = t0 + tt;
            const bool ok = t < t_end;
            float4 bv = make_float4(0.f, 0.f, 0.f, 0.f), cv = bv;
            if (ok) {
                bv.x = to_f32(Bb[(4 * j + 0) * L + t]); bv.y = to_f32(Bb[(4 * j + 1) * L + t]);
                bv.z = to_f32(Bb[(4 * j + 2) * L + t]); bv.w = to_f32(Bb[(4 * j + 3) * L + t]);
                if (kFull) {
                    cv.x = to_f32(Cb[(4 * j + 0) * L + t]); cv.y = to_f32(Cb[(4 * j + 1) * L + t]);
                    cv.z = to_f32(Cb[(4 * j + 2) * L + t]); cv.w = to_f32(Cb[(4 * j + 3) * L + t]);
                }
            }
            float* r = &s_bc[buf][tt][0];
            *reinterpret_cast<float4*>(r + 4 * bc_chunk_b(j, tt)) = bv;
            if (kFull) *reinterpret_cast<float4*>(r + 4 * bc_chunk_c(j, tt)) = cv;
        }

        // ---- this lane's 8 tokens: Delta and Delta*u, once per element ----
        const int64_t tl = t0 + 8 * g;
        const int64_t left = t_end - tl;
        const int nval = !active || left <= 0 ? 0 : (left >= 8 ? 8 : (int)left);
        float uf[8], df[8], zf[8];
        load8<Tin, kVec>(u_row + tl, nval, uf);
        load8<Tin, kVec>(d_row + tl, nval, df);
        if (kFull && z_row) load8<Tin, kVec>(z_row + tl, nval, zf);
        {
            float dl[8], kl[8];
            float part = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float x = df[i] + bias;
                float dt = a.softplus ? softplus_f<kPrecise>(x) : x;
                dt = i < nval ? dt : 0.f;  // padding tokens: Abar = 1, no input -> h unchanged
                dl[i] = dt;
                kl[i] = dt * uf[i];
                part += dt;
            }
            if (!kFull) {  // Kahan-compensated running sum of Delta over the segment
                const float yk = part - dsum_c;
                const float tk = dsum + yk;
                dsum_c = (tk - dsum) - yk;
                dsum = tk;
            }
#pragma unroll
            for (int m = 0; m < 4; ++m)
                *reinterpret_cast<float4*>(dkrow + 16 * g + 4 * m) =
                    make_float4(dl[2 * m], kl[2 * m], dl[2 * m + 1], kl[2 * m + 1]);
        }
        __syncthreads();

        // ---- the recurrence over the chunk's 32 tokens ----
        const float* pbc = &s_bc[buf][0][4 * g];
        float yp[kChunk];
#pragma unroll
        for (int s = 0; s < kChunk; s += 2) {
            const float4 q = *reinterpret_cast<const float4*>(dkrow + 2 * s);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = s + e;
                const float dt = e ? q.z : q.x;
                const float k = e ? q.w : q.y;
                const float4 Bv = *reinterpret_cast<const float4*>(pbc + 32 * t + 4 * (bc_chunk_b(0, t)));
                const float2 dd = make_float2(dt, dt);
                const float2 e01 = __fmul2_rn(dd, a01);
                const float2 e23 = __fmul2_rn(dd, a23);
                const float2 kk = make_float2(k, k);
                const float2 kb01 = __fmul2_rn(kk, make_float2(Bv.x, Bv.y));
                const float2 kb23 = __fmul2_rn(kk, make_float2(Bv.z, Bv.w));
                if (kPrecise) {
                    // Abar = 1 + expm1(Delta*A): the decay's distance from 1 keeps full
                    // relative precision, so a slowly decaying state accumulates no bias
                    // from rounding Abar itself (h = h + em1*h in one fma, then + Bbar*x).
                    const float2 m01 = make_float2(expm1f(e01.x), expm1f(e01.y));
                    const float2 m23 = make_float2(expm1f(e23.x), expm1f(e23.y));
                    h01 = __fadd2_rn(__ffma2_rn(m01, h01, h01), kb01);
                    h23 = __fadd2_rn(__ffma2_rn(m23, h23, h23), kb23);
                } else {
                    const float2 ab01 = make_float2(ex2_approx(e01.x), ex2_approx(e01.y));
                    const float2 ab23 = make_float2(ex2_approx(e23.x), ex2_approx(e23.y));
                    h01 = __ffma2_rn(ab01, h01, kb01);
                    h23 = __ffma2_rn(ab23, h23, kb23);
                }
                if (kFull) {
                    const float4 Cv = *reinterpret_cast<const float4*>(pbc + 32 * t + 4 * (bc_chunk_c(0, t)));
                    float2 y2 = __fmul2_rn(make_float2(Cv.x, Cv.y), h01);
                    y2 = __ffma2_rn(make_float2(Cv.z, Cv.w), h23, y2);
                    yp[t] = y2.x + y2.y;
                }
            }
        }

        if (kFull) {
            // ---- sum the quad's partial readouts; lane g ends with tokens 8g..8g+7 ----
            // Lane l stores its partials of tokens 4j..4j+3 at slot l ^ ((j >> 1) & 3) of
            // block j: conflict-free stores, and conflict-free loads below.
            float* red = &s_red[warp][0];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<float4*>(red + 4 * (32 * j + (lane ^ ((j >> 1) & 3)))) =
                    make_float4(yp[4 * j], yp[4 * j + 1], yp[4 * j + 2], yp[4 * j + 3]);
            __syncwarp();
            float Y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) Y[i] = 0.f;
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * g + jj;
#pragma unroll
                for (int gp = 0; gp < 4; ++gp) {
                    const float4 v = *reinterpret_cast<const float4*>(
                        red + 4 * (32 * j + ((4 * rl + gp) ^ g)));
                    Y[4 * jj + 0] += v.x; Y[4 * jj + 1] += v.y;
                    Y[4 * jj + 2] += v.z; Y[4 * jj + 3] += v.w;
                }
            }
            // ---- D skip, silu gate, store ----
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float y = fmaf(Dd, uf[i], Y[i]);
                if (z_row) y *= silu_f<kPrecise>(zf[i]);
                Y[i] = y;
            }
            store8<Tout, kVec>(o_row + tl, nval, Y);
        }
        buf ^= 1;
    }

    if (kFull) {
        if (active && a.final_state && seg == a.nseg - 1)
            *reinterpret_cast<float4*>(a.final_state + row * kN + 4 * g) =
                make_float4(h01.x, h01.y, h23.x, h23.y);
    } else {
        // Lane g summed Delta over tokens 8g..8g+7 of every chunk; the row's total is the
        // sum over its quad (all 32 lanes take part in the shuffles).
        float s = dsum - dsum_c;
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        if (active) {
            *reinterpret_cast<float4*>(a.ws_hloc + (row * nprev + seg) * kN + 4 * g) =
                make_float4(h01.x, h01.y, h23.x, h23.y);
            if (g == 0) a.ws_dsum[row * nprev + seg] = s;
        }
    }
}

template <typename Tin, typename Tout, bool kVec, bool kPrecise>
static cudaError_t launch_typed(const ScanArgs& a, int64_t batch, cudaStream_t stream) {
    const unsigned gx = (unsigned)((a.dim + kRowsPerCta - 1) / kRowsPerCta);
    if (a.nseg > 1) {
        dim3 grid(gx, (unsigned)(a.nseg - 1), (unsigned)batch);
        scan_chunked_kernel<Tin, Tout, kVec, kPrecise, Mode::kLocalEnd><<<grid, kThreads, 0, stream>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    dim3 grid(gx, (unsigned)a.nseg, (unsigned)batch);
    scan_chunked_kernel<Tin, Tout, kVec, kPrecise, Mode::kFull><<<grid, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
static cudaError_t launch_io(const ScanArgs& a, int64_t batch, bool vec, bool precise,
                             cudaStream_t stream) {
    if (vec) {
        return precise ? launch_typed<Tin, Tout, true, true>(a, batch, stream)
                       : launch_typed<Tin, Tout, true, false>(a, batch, stream);
    }
    return precise ? launch_typed<Tin, Tout, false, true>(a, batch, stream)
                   : launch_typed<Tin, Tout, false, false>(a, batch, stream);
}

cudaError_t launch_scan_fwd(const ScanArgs& a, int64_t batch, bool in_bf16, bool out_bf16,
                            bool vec, bool precise, cudaStream_t stream) {
    using bf = __nv_bfloat16;
    if (in_bf16) {
        return out_bf16 ? launch_io<bf, bf>(a, batch, vec, precise, stream)
                        : launch_io<bf, float>(a, batch, vec, precise, stream);
    }
    return out_bf16 ? launch_io<float, bf>(a, batch, vec, precise, stream)
                    : launch_io<float, float>(a, batch, vec, precise, stream);
}

int scan_chunk_tokens() { return kChunk; }
int scan_rows_per_cta() { return kRowsPerCta; }
int scan_rows_per_warp() { return kRowsPerWarp; }

}  // namespace selscan
