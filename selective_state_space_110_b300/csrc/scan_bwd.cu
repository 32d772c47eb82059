// Backward of the selective scan (S6, Euler) for sm_103a, with recomputation.
//
// "Mamba and State Space Models" (world.lapla.si), section "A Scan on the Chip": the states
// that training's backward pass needs are not stored but computed again. Here the forward
// state is kept only every kChunk tokens (one checkpoint pass); the backward walks the chunks
// from last to first, recomputes the chunk's kChunk states into shared memory from its
// checkpoint, and runs the adjoint recurrence of the scan backwards through them:
//   ds_t = dout_t * silu(z_t),   dz_t = dout_t * s_t * silu'(z_t),   s_t = C_t . h_t + D u_t
//   g_t  = ds_t * C_t + Abar_{t+1} * g_{t+1}          (adjoint of h_t; g starts at dfinal)
//   dk_t = sum_n g_t B_t,   dDelta_t = sum_n g_t h_{t-1} Abar_t A + dk_t u_t
//   du_t = dk_t Delta_t + ds_t D,   ddelta_t = dDelta_t * sigmoid(delta_t + bias) (softplus)
//   dA += g h_{t-1} Abar Delta,  dD += ds u,  dbias += ddelta,  dB_t += g k,  dC_t += ds h_t
//
// Layout as in the forward: a quad of 4 lanes per channel, lane g holding states 4g..4g+3; a CTA
// holds 32 channels of one batch. Lane g owns tokens 4g..4g+3 of each 16-token chunk: it loads
// their inputs, computes their per-token values and writes their gradients; the quad gets
// per-token values by width-4 shuffles. The inputs of the next chunk are loaded into registers
// while the current chunk computes. B and C of a chunk are staged in shared memory one row per
// token (BcStage).
//
// Long sequences with few rows are cut into time segments that run in parallel (grid.y), as in
// the forward: a forward pass over segments 0..S-2 from a zero state keeps each one's local end
// state and summed Delta; a reverse pass over segments 1..S-1 from a zero adjoint keeps each
// one's local start adjoint (the adjoint of the state before the segment) and summed Delta. The
// full backward of segment s then starts its forward from the fold of the earlier segments,
// h <- exp(A sum Delta) h + h_local_end, and its adjoint from the fold of the later ones,
// g <- g_local_start + exp(A sum Delta) g (the adjoint recurrence is linear in g as well).
//
// dB and dC are sums over every channel of a batch. Each warp sums its 8 rows' terms: built for
// 3 CTAs per SM, by a per-token reduce-scatter in three shuffle rounds (lane (q, g) ends with
// one of the 32 dB | dC sums of the token); built for 2, by two contractions per chunk from
// shared memory (dC_t = sum ds_t h_t over the stored states; dB_t = sum g_t k_t over the
// adjoints, stored in place of the states). The CTA adds its 6 warps in shared memory and
// writes one partial per token and value. dA, dD and
// dbias are kept per (batch, channel). A second kernel adds the partials in a fixed order, so
// the gradients are deterministic (no atomics).
#include <cstddef>

#include "selscan_device.cuh"
#include "selscan_launch.h"

namespace selscan {

constexpr int kBChunk = 16;                 // tokens per chunk (and per checkpoint)
constexpr int kBWarps = 6;
constexpr int kBThreads = 32 * kBWarps;     // 192: 48 channels
constexpr int kBRows = 8 * kBWarps;         // channels per CTA
constexpr int kBSlots = 32;                 // dB[0..15], dC[0..15] per token
// Row stride of the per-(row, token) coefficient tiles of the contractions (one 16-token chunk).
constexpr int kBCoefStride = kBChunk;
// CTAs of 6 warps (48 channels, 64 KB of shared memory): 3 fit an SM. A grid of Mamba-2.8B size
// (4 x 107 CTAs on 148 SMs) then holds at most 144 channels on any SM, where CTAs of 4 warps at
// 5 per SM held 160. Built for 3 per SM (96 registers: 18 warps leave 5 on some schedulers) when
// the grid needs the slots, for 2 (159-168 registers, no spills) when it fits one wave at 2.
constexpr int kBMinCtas = 3;
constexpr int kBMinCtasRoomy = 2;

struct BwdSmem {
    float bc[2][kBChunk][32];                // B | C per token (layout: BcStage)
    float4 H[kBWarps][kBChunk][32];          // recomputed states h_t, then adjoints g_t
    float P[kBWarps][kBChunk][kBSlots];      // warp sums of dB | dC per token
    float DS[kBWarps][8][kBCoefStride];      // ds_t per row of the warp and token
    float K[kBWarps][8][kBCoefStride];       // k_t = Delta_t u_t per row of the warp and token
};

template <typename Tin>
__device__ __forceinline__ float ld1(const Tin* p) { return to_f32(*p); }

// v * exp(s*a) for s*a <= 0 in fp32 with a small relative error at every decay strength. The
// product x = s*a is rounded; its rounding error lo = fma(s, a, -x) is carried to first order
// (exp(x + lo) = exp(x) (1 + lo)), since at |x| ~ 30 the rounding alone would be 2e-6 of the
// decay. A weak decay is formed as v + expm1(x) v (its distance from 1 exact to rounding), a
// strong one (x < -ln 2) as expf(x) v.
__device__ __forceinline__ float precise_decay(float s, float a, float v) {
    const float x = s * a;
    const float lo = fmaf(s, a, -x);
    if (x < -0.69314718f) {
        const float ev = expf(x) * v;
        return fmaf(ev, lo, ev);
    }
    const float m = expm1f(x);
    return fmaf(fmaf(lo, m + 1.f, m), v, v);
}

template <bool kPrecise>
__device__ __forceinline__ float sigmoid_f(float x) {
    return kPrecise ? 1.f / (1.f + expf(-x)) : rcp_approx(1.f + ex2_approx(-x * kLog2e));
}

// Four consecutive tokens t..t+3 of one row; zeros from token n on. kVec: one 8-byte (bf16)
// or 16-byte (fp32) load, which needs seqlen % 4 == 0 (t is a multiple of 4).
template <typename T, bool kVec>
struct Quad4;
template <bool kVec>
struct Quad4<__nv_bfloat16, kVec> {
    uint2 r;
    __device__ __forceinline__ void load(const __nv_bfloat16* p, int64_t t, int64_t n) {
        if (kVec) {
            r = t < n ? __ldg(reinterpret_cast<const uint2*>(p + t)) : make_uint2(0u, 0u);
        } else {
            const uint16_t* q = reinterpret_cast<const uint16_t*>(p);
            const uint32_t v0 = t < n ? q[t] : 0u, v1 = t + 1 < n ? q[t + 1] : 0u;
            const uint32_t v2 = t + 2 < n ? q[t + 2] : 0u, v3 = t + 3 < n ? q[t + 3] : 0u;
            r = make_uint2(v0 | (v1 << 16), v2 | (v3 << 16));
        }
    }
    __device__ __forceinline__ float get(int i) const {
        return i == 0 ? bf16lo(r.x) : i == 1 ? bf16hi(r.x) : i == 2 ? bf16lo(r.y) : bf16hi(r.y);
    }
};
template <bool kVec>
struct Quad4<float, kVec> {
    float4 r;
    __device__ __forceinline__ void load(const float* p, int64_t t, int64_t n) {
        if (kVec) {
            r = t < n ? __ldg(reinterpret_cast<const float4*>(p + t)) : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            r.x = t < n ? p[t] : 0.f;
            r.y = t + 1 < n ? p[t + 1] : 0.f;
            r.z = t + 2 < n ? p[t + 2] : 0.f;
            r.w = t + 3 < n ? p[t + 3] : 0.f;
        }
    }
    __device__ __forceinline__ float get(int i) const {
        return i == 0 ? r.x : i == 1 ? r.y : i == 2 ? r.z : r.w;
    }
};

// Stores four consecutive values of one row at t..t+3, those before token n only.
template <typename T, bool kVec>
__device__ __forceinline__ void store4(T* p, int64_t t, int64_t n, const float (&v)[4]) {
    if (t >= n) return;
    if (kVec) {
        if constexpr (sizeof(T) == 2) {
            uint2 w;
            w.x = (uint32_t)__bfloat16_as_ushort(from_f32<T>(v[0])) |
                  ((uint32_t)__bfloat16_as_ushort(from_f32<T>(v[1])) << 16);
            w.y = (uint32_t)__bfloat16_as_ushort(from_f32<T>(v[2])) |
                  ((uint32_t)__bfloat16_as_ushort(from_f32<T>(v[3])) << 16);
            *reinterpret_cast<uint2*>(p + t) = w;
        } else {
            *reinterpret_cast<float4*>(p + t) = make_float4(v[0], v[1], v[2], v[3]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (t + i < n) p[t + i] = from_f32<T>(v[i]);
    }
}

// B | C of one chunk in shared memory, one row per token.
// fp32 inputs: 8 granules of 4 floats per row (0..3 = B states 4q.., 4..7 = C), granule index
// XOR-swizzled by (token & 7). bf16 inputs, kept as bf16 (lossless): 4 granules of 16 bytes per
// row, granule q = {B 4q..4q+3, C 4q..4q+3}, so a lane gets its B and C values with one 16-byte
// load; granule index XOR-swizzled by ((token >> 1) & 3). Both swizzles keep the staging stores
// free of bank conflicts.
template <typename Tin>
struct BcStage;
template <>
struct BcStage<float> {
    static __device__ __forceinline__ int off(int tt, int gr) { return tt * 32 + 4 * (gr ^ (tt & 7)); }
    // Staging thread: 4 values of granule ch (0..3 B, 4..7 C) of token tt.
    static __device__ __forceinline__ void put(float* base, int tt, int ch, const float (&v)[4]) {
        *reinterpret_cast<float4*>(base + off(tt, ch)) = make_float4(v[0], v[1], v[2], v[3]);
    }
    static __device__ __forceinline__ float4 get_b(const float* base, int t, int g) {
        return *reinterpret_cast<const float4*>(base + off(t, g));
    }
    static __device__ __forceinline__ void get_bc(const float* base, int t, int g, float4& b, float4& c) {
        b = *reinterpret_cast<const float4*>(base + off(t, g));
        c = *reinterpret_cast<const float4*>(base + off(t, 4 + g));
    }
};
template <>
struct BcStage<__nv_bfloat16> {
    static __device__ __forceinline__ int off(int tt, int q) {  // in 32-bit words
        return tt * 16 + 4 * (q ^ ((tt >> 1) & 3));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
    }
    static __device__ __forceinline__ void put(float* base, int tt, int ch, const float (&v)[4]) {
        // v holds bf16 values widened to fp32: narrowing them back is exact.
        uint32_t* w = reinterpret_cast<uint32_t*>(base) + off(tt, ch & 3) + 2 * (ch >> 2);
        *reinterpret_cast<uint2*>(w) = make_uint2(pack(v[0], v[1]), pack(v[2], v[3]));
    }
    static __device__ __forceinline__ float4 get_b(const float* base, int t, int g) {
        const uint2 r = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint32_t*>(base) + off(t, g));
        return make_float4(bf16lo(r.x), bf16hi(r.x), bf16lo(r.y), bf16hi(r.y));
    }
    static __device__ __forceinline__ void get_bc(const float* base, int t, int g, float4& b, float4& c) {
        const uint4 r = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint32_t*>(base) + off(t, g));
        b = make_float4(bf16lo(r.x), bf16hi(r.x), bf16lo(r.y), bf16hi(r.y));
        c = make_float4(bf16lo(r.z), bf16hi(r.z), bf16lo(r.w), bf16hi(r.w));
    }
};

// Modes of the backward kernel: the full backward of a segment, the forward local-end pass
// (segments 0..S-2) and the adjoint local-start pass (segments 1..S-1).
enum BwdMode : int { kBwdFull = 0, kBwdFwdLocal = 1, kBwdAdjLocal = 2 };

// One warp's sums over its 8 rows for the 16 tokens of a chunk: P[t][slot0 + n] =
// sum_r coef[r][t] V[t][r][n] for the 16 states n, with V the warp's [token][lane] float4 tile
// (lane 4r + j holds states 4j..4j+3 of row r). Lane (tq, j) takes tokens tq and tq + 8 and
// states 4j..4j+3, and visits the rows in the order (i + tq) & 7, so that each quarter-warp's
// 16-byte loads fall on 8 different bank groups and its coefficient loads on distinct banks.
__device__ __forceinline__ void warp_rows_contract(const float4* V, const float* coef, float* P,
                                                   int slot0, int lane) {
    const int tq = lane >> 2, j = lane & 3;
    float2 a01 = f2(0.f), a23 = f2(0.f), b01 = f2(0.f), b23 = f2(0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = (i + tq) & 7;
        const float4 v0 = V[tq * 32 + 4 * r + j], v1 = V[(tq + 8) * 32 + 4 * r + j];
        const float2 c0 = f2(coef[r * kBCoefStride + tq]), c1 = f2(coef[r * kBCoefStride + tq + 8]);
        a01 = __ffma2_rn(c0, make_float2(v0.x, v0.y), a01);
        a23 = __ffma2_rn(c0, make_float2(v0.z, v0.w), a23);
        b01 = __ffma2_rn(c1, make_float2(v1.x, v1.y), b01);
        b23 = __ffma2_rn(c1, make_float2(v1.z, v1.w), b23);
    }
    *reinterpret_cast<float4*>(P + tq * kBSlots + slot0 + 4 * j) = make_float4(a01.x, a01.y, a23.x, a23.y);
    *reinterpret_cast<float4*>(P + (tq + 8) * kBSlots + slot0 + 4 * j) =
        make_float4(b01.x, b01.y, b23.x, b23.y);
}

template <typename Tin, typename Tg, bool kPrecise, bool kVec, int kMode, int kMinCtas>
__global__ void __launch_bounds__(kBThreads, kMinCtas) scan_bwd_kernel(const BwdArgs a) {
    extern __shared__ __align__(16) unsigned char bwd_smem[];
    BwdSmem& sm = *reinterpret_cast<BwdSmem*>(bwd_smem);
    // The dB | dC sums over a warp's rows: with the registers of 2 CTAs per SM, two contractions
    // per chunk from shared memory (the states, then the adjoints written over them); at 3 per SM
    // (96 registers) a per-token shuffle reduce-scatter, which needs fewer live registers.
    constexpr bool kContract = kMinCtas <= 2;
    static_assert(kContract == (kMinCtas == kBMinCtasRoomy), "launch sizes shared memory by this");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = lane >> 2, g = lane & 3;
    const int64_t b = blockIdx.z;
    const int seg = kMode == kBwdAdjLocal ? (int)blockIdx.y + 1 : (int)blockIdx.y;
    const int nprev = a.nseg - 1;
    const int64_t d_raw = (int64_t)blockIdx.x * kBRows + warp * 8 + quad;
    const bool active = d_raw < a.dim;
    const int64_t d = active ? d_raw : 0;
    const int64_t row = b * a.dim + d;
    const int64_t L = a.seqlen;
    const int64_t Lr = active ? L : 0;  // tokens of this lane's row (none past dim)
    const int nchunks = (int)((L + kBChunk - 1) / kBChunk);
    const int seg_chunks = (int)(a.seg_len / kBChunk);
    const int c_begin = seg * seg_chunks;  // this segment's chunks: [c_begin, c_end)
    const int c_end = min(nchunks, c_begin + seg_chunks);

    const float4 A4 = *reinterpret_cast<const float4*>(a.A + d * kN + 4 * g);
    const float Av[4] = {A4.x, A4.y, A4.z, A4.w};
    const float2 A01 = make_float2(A4.x, A4.y), A23 = make_float2(A4.z, A4.w);
    const float bias = a.delta_bias ? a.delta_bias[d] : 0.f;
    const float Dd = a.D ? a.D[d] : 0.f;
    // Per-token steps are kept as Delta * kScale: the SFU path takes exp(Delta A) as
    // 2^(Delta log2(e) A).
    constexpr float kScale = kPrecise ? 1.f : kLog2e;

    const Tin* u_row = static_cast<const Tin*>(a.u) + row * L;
    const Tin* d_row = static_cast<const Tin*>(a.delta) + row * L;
    const Tin* z_row = a.z ? static_cast<const Tin*>(a.z) + row * L : nullptr;
    const Tg* o_row = static_cast<const Tg*>(a.dout) + row * L;
    float* ckpt = a.ws_ckpt + (row * nchunks) * kN + 4 * g;

    // B | C staging: thread -> token s_tt of the chunk, granule s_ch (0..3 B, 4..7 C); the first
    // 16 x 8 threads stage.
    const int s_tt = tid & 15, s_ch = tid >> 4;
    const bool stager = s_ch < 8;
    const Tin* s_src = (s_ch < 4 ? static_cast<const Tin*>(a.B) : static_cast<const Tin*>(a.C)) +
                       b * kN * L + (int64_t)(4 * (s_ch & 3)) * L;
    float sb[4];
    auto fetch_bc = [&](int c, bool withC) {
        const int64_t t = (int64_t)c * kBChunk + s_tt;
        const bool ok = stager && t < L && (withC || s_ch < 4);
#pragma unroll
        for (int j = 0; j < 4; ++j) sb[j] = ok ? ld1(s_src + j * L + t) : 0.f;
    };
    using Stage = BcStage<Tin>;
    auto put_bc = [&](int buf, bool withC) {
        if (stager && (withC || s_ch < 4)) Stage::put(&sm.bc[buf][0][0], s_tt, s_ch, sb);
    };
    // v * exp(Delta A_n) + add (s = Delta * kScale). fp32 inputs write a weak decay as 1 + expm1:
    // the decay's distance from 1 keeps full relative precision, so a slowly decaying state or
    // adjoint accumulates no bias from rounding the decay itself over thousands of tokens. A
    // strong decay (exponent below -ln 2) is taken from expf instead: there 1 + expm1 would
    // carry expm1's absolute rounding (~6e-8) as a relative error of 6e-8 / exp(x) in the
    // decayed value, which the gradient of the initial state (a product of decays) shows.
    auto decay_fma = [&](float s, int n, float v, float add) -> float {
        if (kPrecise) return precise_decay(s, Av[n], v) + add;
        return fmaf(ex2_approx(s * Av[n]), v, add);
    };
    // The SFU path of four states at once as two packed pairs (the same roundings as decay_fma):
    // v <- 2^(s A) v + k B.
    auto decay_step2 = [&](float s, float k, const float4& Bv, float (&v)[4]) {
        const float2 s2 = f2(s), k2 = f2(k);
        const float2 x01 = __fmul2_rn(s2, A01), x23 = __fmul2_rn(s2, A23);
        const float2 e01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
        const float2 e23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
        const float2 h01 = __ffma2_rn(e01, make_float2(v[0], v[1]), __fmul2_rn(k2, make_float2(Bv.x, Bv.y)));
        const float2 h23 = __ffma2_rn(e23, make_float2(v[2], v[3]), __fmul2_rn(k2, make_float2(Bv.z, Bv.w)));
        v[0] = h01.x; v[1] = h01.y; v[2] = h23.x; v[3] = h23.y;
    };
    auto delta_of = [&](float x) -> float {
        if (!a.softplus) return x;
        return kPrecise ? softplus_f<true>(x) : softplus2(make_float2(x, x)).x;
    };

    // exp(A_n * S) for a summed Delta S (fold of a segment).
    auto seg_decay_fma = [&](float S, int n, float v, float add) -> float {
        if (kPrecise) return precise_decay(S, Av[n], v) + add;
        return fmaf(ex2_approx(S * kLog2e * Av[n]), v, add);
    };
    // Kahan sum of Delta over this lane's owned tokens (local passes).
    float dsum = 0.f, dsum_c = 0.f;
    auto add_delta = [&](const float (&dl)[4]) {
        const float part_sum = (dl[0] + dl[1] + dl[2] + dl[3]) * (1.f / kScale);
        const float yk = part_sum - dsum_c;
        const float tk = dsum + yk;
        dsum_c = (tk - dsum) - yk;
        dsum = tk;
    };
    auto quad_delta_sum = [&]() -> float {
        float v = dsum - dsum_c;
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        return v;
    };

    float h[4] = {0.f, 0.f, 0.f, 0.f};
    if (kMode == kBwdFull && !a.ckpt_given) {  // initial state, then the earlier segments' fold
        if (a.initial_state && active) {
            const float4 s0 = *reinterpret_cast<const float4*>(a.initial_state + row * kN + 4 * g);
            h[0] = s0.x; h[1] = s0.y; h[2] = s0.z; h[3] = s0.w;
        }
        for (int k = 0; k < seg && active; ++k) {
            const float S = a.ws_fsum[row * nprev + k];
            const float4 hl = *reinterpret_cast<const float4*>(a.ws_hloc + (row * nprev + k) * kN + 4 * g);
            h[0] = seg_decay_fma(S, 0, h[0], hl.x);
            h[1] = seg_decay_fma(S, 1, h[1], hl.y);
            h[2] = seg_decay_fma(S, 2, h[2], hl.z);
            h[3] = seg_decay_fma(S, 3, h[3], hl.w);
        }
    }

    // ---- checkpoint pass: the forward state before every chunk (the local-end pass: the
    // forward only) ----
    // (skipped when the forward pass saved the checkpoints)
    if (kMode == kBwdFwdLocal || (kMode == kBwdFull && !a.ckpt_given)) {
        Quad4<Tin, kVec> pd, pu;
        if (c_begin < c_end) {
            const int64_t tl = (int64_t)c_begin * kBChunk + 4 * g;
            pd.load(d_row, tl, Lr);
            pu.load(u_row, tl, Lr);
            fetch_bc(c_begin, false);
        }
        for (int c = c_begin; c < c_end; ++c) {
            const int64_t tl = (int64_t)c * kBChunk + 4 * g;
            if (kMode == kBwdFull && active)
                *reinterpret_cast<float4*>(ckpt + (int64_t)c * kN) = make_float4(h[0], h[1], h[2], h[3]);
            put_bc(c & 1, false);
            float dl[4], kl[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {  // tokens past the end are the identity step
                const float dt = tl + i < Lr ? delta_of(pd.get(i) + bias) : 0.f;
                dl[i] = dt * kScale;
                kl[i] = dt * pu.get(i);
            }
            if (kMode == kBwdFwdLocal) add_delta(dl);
            if (c + 1 < c_end) {
                pd.load(d_row, tl + kBChunk, Lr);
                pu.load(u_row, tl + kBChunk, Lr);
                fetch_bc(c + 1, false);
            }
            __syncthreads();  // B of chunk c staged (buffer c & 1)
            const float* bcb = &sm.bc[c & 1][0][0];
#pragma unroll
            for (int t = 0; t < kBChunk; ++t) {
                const float s = __shfl_sync(0xffffffffu, dl[t & 3], t >> 2, 4);
                const float k = __shfl_sync(0xffffffffu, kl[t & 3], t >> 2, 4);
                const float4 Bv = Stage::get_b(bcb, t, g);
                if constexpr (kPrecise) {
                    h[0] = decay_fma(s, 0, h[0], k * Bv.x);
                    h[1] = decay_fma(s, 1, h[1], k * Bv.y);
                    h[2] = decay_fma(s, 2, h[2], k * Bv.z);
                    h[3] = decay_fma(s, 3, h[3], k * Bv.w);
                } else {
                    decay_step2(s, k, Bv, h);
                }
            }
        }
    }
    if (kMode == kBwdFwdLocal) {
        const float S = quad_delta_sum();
        if (active) {
            *reinterpret_cast<float4*>(a.ws_hloc + (row * nprev + seg) * kN + 4 * g) =
                make_float4(h[0], h[1], h[2], h[3]);
            if (g == 0) a.ws_fsum[row * nprev + seg] = S;
        }
        return;
    }
    __syncthreads();  // the last chunk's readers of the staging buffers are done

    // ---- reverse pass ----
    float gad[4] = {0.f, 0.f, 0.f, 0.f};  // adjoint of the state
    if (kMode == kBwdFull && active) {  // dfinal, then the fold of the later segments
        if (a.dfinal_state) {
            const float4 f = *reinterpret_cast<const float4*>(a.dfinal_state + row * kN + 4 * g);
            gad[0] = f.x; gad[1] = f.y; gad[2] = f.z; gad[3] = f.w;
        }
        for (int k = nprev; k > seg; --k) {
            const float S = a.ws_bsum[row * nprev + (k - 1)];
            const float4 gl = *reinterpret_cast<const float4*>(a.ws_gloc + (row * nprev + (k - 1)) * kN + 4 * g);
            gad[0] = seg_decay_fma(S, 0, gad[0], gl.x);
            gad[1] = seg_decay_fma(S, 1, gad[1], gl.y);
            gad[2] = seg_decay_fma(S, 2, gad[2], gl.z);
            gad[3] = seg_decay_fma(S, 3, gad[3], gl.w);
        }
    }
    float dA_acc[4] = {0.f, 0.f, 0.f, 0.f};
    float dD_acc = 0.f, db_acc = 0.f;
    Tg* du_row = static_cast<Tg*>(a.du) + row * L;
    Tg* dd_row = static_cast<Tg*>(a.ddelta) + row * L;
    Tg* dz_row = a.z ? static_cast<Tg*>(a.dz) + row * L : nullptr;
    float* part = a.ws_part + ((int64_t)blockIdx.x * a.batch + b) * L * kBSlots;  // [t][slot]

    Quad4<Tin, kVec> pd, pu, pz;
    Quad4<Tg, kVec> po;
    if (c_begin < c_end) {
        const int64_t tl = (int64_t)(c_end - 1) * kBChunk + 4 * g;
        pd.load(d_row, tl, Lr);
        pu.load(u_row, tl, Lr);
        if (z_row) pz.load(z_row, tl, Lr);
        po.load(o_row, tl, Lr);
        fetch_bc(c_end - 1, true);
    }
    for (int c = c_end - 1; c >= c_begin; --c) {
        const int64_t t0 = (int64_t)c * kBChunk;
        const int64_t tl = t0 + 4 * g;
        float4 hk4 = make_float4(0.f, 0.f, 0.f, 0.f);  // rows past dim run on zeros
        if (active) hk4 = *reinterpret_cast<const float4*>(ckpt + (int64_t)c * kN);
        put_bc(0, true);
        // Owned tokens: per-token values from the prefetched inputs.
        float dl[4], kl[4], dsl[4], dzf[4], ul[4], sgx[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool ok = tl + i < Lr;
            const float x = pd.get(i) + bias;
            const float dt = ok ? delta_of(x) : 0.f;  // tokens past the end: identity step
            const float u = pu.get(i), o = po.get(i);
            dl[i] = dt * kScale;
            kl[i] = dt * u;
            ul[i] = u;
            sgx[i] = a.softplus ? sigmoid_f<kPrecise>(x) : 1.f;
            if (z_row) {
                const float zv = pz.get(i), sz = sigmoid_f<kPrecise>(zv);
                dsl[i] = o * zv * sz;
                dzf[i] = o * sz * (1.f + zv * (1.f - sz));
            } else {
                dsl[i] = o;
                dzf[i] = 0.f;
            }
        }
        if (c > c_begin) {
            pd.load(d_row, tl - kBChunk, Lr);
            pu.load(u_row, tl - kBChunk, Lr);
            if (z_row) pz.load(z_row, tl - kBChunk, Lr);
            po.load(o_row, tl - kBChunk, Lr);
            fetch_bc(c - 1, true);
        }
        __syncthreads();  // B | C of the chunk staged
        const float* bcb = &sm.bc[0][0][0];
        float4* Hw = &sm.H[warp][0][0];
        if (kMode == kBwdAdjLocal) {  // the adjoint alone, last token first
            add_delta(dl);
#pragma unroll
            for (int t = kBChunk - 1; t >= 0; --t) {
                const float s = __shfl_sync(0xffffffffu, dl[t & 3], t >> 2, 4);
                const float ds = __shfl_sync(0xffffffffu, dsl[t & 3], t >> 2, 4);
                float4 Bv, Cv;
                Stage::get_bc(bcb, t, g, Bv, Cv);
                gad[0] = decay_fma(s, 0, fmaf(ds, Cv.x, gad[0]), 0.f);
                gad[1] = decay_fma(s, 1, fmaf(ds, Cv.y, gad[1]), 0.f);
                gad[2] = decay_fma(s, 2, fmaf(ds, Cv.z, gad[2]), 0.f);
                gad[3] = decay_fma(s, 3, fmaf(ds, Cv.w, gad[3]), 0.f);
            }
            __syncthreads();  // the chunk's staging is read before the next one is written
            continue;
        }

        if constexpr (kContract) {  // ds_t and k_t of the quad's row for the contractions
            *reinterpret_cast<float4*>(&sm.DS[warp][quad][4 * g]) = make_float4(dsl[0], dsl[1], dsl[2], dsl[3]);
            *reinterpret_cast<float4*>(&sm.K[warp][quad][4 * g]) = make_float4(kl[0], kl[1], kl[2], kl[3]);
        }
        // Recompute the chunk's states (into shared memory) and the readouts s_t - D u_t.
        float sl[4];
        {
            float hh[4] = {hk4.x, hk4.y, hk4.z, hk4.w};
#pragma unroll
            for (int t = 0; t < kBChunk; ++t) {
                const float s = __shfl_sync(0xffffffffu, dl[t & 3], t >> 2, 4);
                const float k = __shfl_sync(0xffffffffu, kl[t & 3], t >> 2, 4);
                float4 Bv, Cv;
                Stage::get_bc(bcb, t, g, Bv, Cv);
                float y;
                if constexpr (kPrecise) {
                    hh[0] = decay_fma(s, 0, hh[0], k * Bv.x);
                    hh[1] = decay_fma(s, 1, hh[1], k * Bv.y);
                    hh[2] = decay_fma(s, 2, hh[2], k * Bv.z);
                    hh[3] = decay_fma(s, 3, hh[3], k * Bv.w);
                    y = Cv.x * hh[0];
                    y = fmaf(Cv.y, hh[1], y);
                    y = fmaf(Cv.z, hh[2], y);
                    y = fmaf(Cv.w, hh[3], y);
                } else {
                    decay_step2(s, k, Bv, hh);
                    float2 y2 = __fmul2_rn(make_float2(Cv.x, Cv.y), make_float2(hh[0], hh[1]));
                    y2 = __ffma2_rn(make_float2(Cv.z, Cv.w), make_float2(hh[2], hh[3]), y2);
                    y = y2.x + y2.y;
                }
                Hw[t * 32 + lane] = make_float4(hh[0], hh[1], hh[2], hh[3]);
                y += __shfl_xor_sync(0xffffffffu, y, 1);
                y += __shfl_xor_sync(0xffffffffu, y, 2);
                if (g == (t >> 2)) sl[t & 3] = y;
            }
        }
        if (z_row) {
            float dzv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) dzv[i] = dzf[i] * fmaf(Dd, ul[i], sl[i]);
            store4<Tg, kVec>(dz_row, tl, Lr, dzv);
        }
        __syncwarp();
        if constexpr (kContract) {
            // dC_t = sum over the warp's 8 rows of ds_t h_t, from the states just stored.
            warp_rows_contract(Hw, &sm.DS[warp][0][0], &sm.P[warp][0][0], 16, lane);
            __syncwarp();  // H is read before the adjoints overwrite it
        }

        // Adjoint recurrence, last token of the chunk first. The chunk's dA terms are summed
        // apart and then added to the running sum: two-level summation keeps the rounding of
        // sums over hundreds of thousands of tokens near that of the per-chunk sums.
        float dkl[4], dal[4];  // owner: dk_t and the Abar part of dDelta_t
        float dA_chunk[4] = {0.f, 0.f, 0.f, 0.f};
        float4 ht = make_float4(0.f, 0.f, 0.f, 0.f);  // h_t, for the reduce-scattered dC terms
        if constexpr (!kContract) ht = Hw[(kBChunk - 1) * 32 + lane];
#pragma unroll
        for (int t = kBChunk - 1; t >= 0; --t) {
            const float s = __shfl_sync(0xffffffffu, dl[t & 3], t >> 2, 4);
            const float k = __shfl_sync(0xffffffffu, kl[t & 3], t >> 2, 4);
            const float ds = __shfl_sync(0xffffffffu, dsl[t & 3], t >> 2, 4);
            float4 Bv, Cv;
            Stage::get_bc(bcb, t, g, Bv, Cv);
            const float4 hp = t > 0 ? Hw[(t - 1) * 32 + lane] : hk4;
            const float Bs[4] = {Bv.x, Bv.y, Bv.z, Bv.w}, Cs[4] = {Cv.x, Cv.y, Cv.z, Cv.w};
            const float hts[4] = {ht.x, ht.y, ht.z, ht.w}, hps[4] = {hp.x, hp.y, hp.z, hp.w};
            float dk = 0.f, da = 0.f, v[8];  // v: dB terms g_t k_t, then dC terms ds_t h_t
            if constexpr (kPrecise) {
#pragma unroll
                for (int n = 0; n < 4; ++n) gad[n] = fmaf(ds, Cs[n], gad[n]);
                if constexpr (kContract)  // g_t replaces h_t, which the token after it last read
                    Hw[t * 32 + lane] = make_float4(gad[0], gad[1], gad[2], gad[3]);
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    v[4 + n] = ds * hts[n];
                    v[n] = gad[n] * k;
                    dk = fmaf(gad[n], Bs[n], dk);
                    // the adjoint times Abar (weak decays as 1 + expm1, see decay_fma)
                    const float gab = precise_decay(s, Av[n], gad[n]);
                    const float w = gab * hps[n];  // dAbar * Abar
                    da = fmaf(w, Av[n], da);
                    dA_chunk[n] = fmaf(w, s, dA_chunk[n]);
                    gad[n] = gab;
                }
            } else {  // the same steps on packed pairs of states (0, 1) and (2, 3)
                const float2 s2 = f2(s), k2 = f2(k), ds2 = f2(ds);
                float2 g01 = __ffma2_rn(ds2, make_float2(Cs[0], Cs[1]), make_float2(gad[0], gad[1]));
                float2 g23 = __ffma2_rn(ds2, make_float2(Cs[2], Cs[3]), make_float2(gad[2], gad[3]));
                if constexpr (kContract) {
                    Hw[t * 32 + lane] = make_float4(g01.x, g01.y, g23.x, g23.y);
                } else {
                    const float2 vc01 = __fmul2_rn(ds2, make_float2(hts[0], hts[1]));
                    const float2 vc23 = __fmul2_rn(ds2, make_float2(hts[2], hts[3]));
                    const float2 vb01 = __fmul2_rn(g01, k2), vb23 = __fmul2_rn(g23, k2);
                    v[0] = vb01.x; v[1] = vb01.y; v[2] = vb23.x; v[3] = vb23.y;
                    v[4] = vc01.x; v[5] = vc01.y; v[6] = vc23.x; v[7] = vc23.y;
                }
                float2 dk2 = __fmul2_rn(g01, make_float2(Bs[0], Bs[1]));
                dk2 = __ffma2_rn(g23, make_float2(Bs[2], Bs[3]), dk2);
                const float2 x01 = __fmul2_rn(s2, A01), x23 = __fmul2_rn(s2, A23);
                g01 = __fmul2_rn(g01, make_float2(ex2_approx(x01.x), ex2_approx(x01.y)));
                g23 = __fmul2_rn(g23, make_float2(ex2_approx(x23.x), ex2_approx(x23.y)));
                const float2 w01 = __fmul2_rn(g01, make_float2(hps[0], hps[1]));  // dAbar * Abar
                const float2 w23 = __fmul2_rn(g23, make_float2(hps[2], hps[3]));
                float2 da2 = __fmul2_rn(w01, A01);
                da2 = __ffma2_rn(w23, A23, da2);
                const float2 c01 = __ffma2_rn(w01, s2, make_float2(dA_chunk[0], dA_chunk[1]));
                const float2 c23 = __ffma2_rn(w23, s2, make_float2(dA_chunk[2], dA_chunk[3]));
                dA_chunk[0] = c01.x; dA_chunk[1] = c01.y; dA_chunk[2] = c23.x; dA_chunk[3] = c23.y;
                gad[0] = g01.x; gad[1] = g01.y; gad[2] = g23.x; gad[3] = g23.y;
                dk = dk2.x + dk2.y;
                da = da2.x + da2.y;
            }
            ht = hp;
            dk += __shfl_xor_sync(0xffffffffu, dk, 1);
            dk += __shfl_xor_sync(0xffffffffu, dk, 2);
            da += __shfl_xor_sync(0xffffffffu, da, 1);
            da += __shfl_xor_sync(0xffffffffu, da, 2);
            if (g == (t >> 2)) { dkl[t & 3] = dk; dal[t & 3] = da; }
            if constexpr (!kContract) {
                // Sums of the 8 rows' dB | dC terms, reduce-scattered over lane bits 4, 3, 2:
                // lane (q, g) ends with dB of state 4g+q (q < 4) or dC of state 4g+q-4.
                const bool x16 = (lane >> 4) & 1, x8 = (lane >> 3) & 1, x4 = (lane >> 2) & 1;
                float w4[4], w2[2];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float send = x16 ? v[i] : v[i + 4], keep = x16 ? v[i + 4] : v[i];
                    w4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float send = x8 ? w4[i] : w4[i + 2], keep = x8 ? w4[i + 2] : w4[i];
                    w2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                }
                const float send = x4 ? w2[0] : w2[1], keep = x4 ? w2[1] : w2[0];
                sm.P[warp][t][(quad >> 2) * 16 + 4 * g + (quad & 3)] =
                    keep + __shfl_xor_sync(0xffffffffu, send, 4);
            }
        }
        if constexpr (kContract) {
            __syncwarp();
            // dB_t = sum over the warp's 8 rows of g_t k_t, from the adjoints just stored.
            warp_rows_contract(Hw, &sm.K[warp][0][0], &sm.P[warp][0][0], 0, lane);
        }
#pragma unroll
        for (int n = 0; n < 4; ++n) dA_acc[n] += dA_chunk[n];
        // Owner: per-token gradients of its tokens.
        {
            float duv[4], ddv[4], dD_c = 0.f, db_c = 0.f;
            const float* dso = dsl;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                duv[i] = fmaf(dkl[i], dl[i] * (1.f / kScale), dso[i] * Dd);
                ddv[i] = fmaf(dkl[i], ul[i], dal[i]) * sgx[i];
                if (tl + i < Lr) {
                    dD_c = fmaf(dso[i], ul[i], dD_c);
                    db_c += ddv[i];
                }
            }
            dD_acc += dD_c;
            db_acc += db_c;
            store4<Tg, kVec>(du_row, tl, Lr, duv);
            store4<Tg, kVec>(dd_row, tl, Lr, ddv);
        }
        __syncthreads();  // every warp's dB | dC sums of the chunk are in P
        // CTA sums of dB_t / dC_t over the kBWarps warps -> this CTA's partials [t][slot].
#pragma unroll
        for (int r = 0; r < (kBSlots * kBChunk + kBThreads - 1) / kBThreads; ++r) {
            const int item = tid + r * kBThreads;
            if (item >= kBSlots * kBChunk) break;
            const int slot = item & 31, tt = item >> 5;
            const int64_t t = t0 + tt;
            if (t < L) {
                float acc = sm.P[0][tt][slot];
#pragma unroll
                for (int w = 1; w < kBWarps; ++w) acc += sm.P[w][tt][slot];
                part[t * kBSlots + slot] = acc;
            }
        }
    }

    if (kMode == kBwdAdjLocal) {
        const float S = quad_delta_sum();
        if (active) {
            *reinterpret_cast<float4*>(a.ws_gloc + (row * nprev + (seg - 1)) * kN + 4 * g) =
                make_float4(gad[0], gad[1], gad[2], gad[3]);
            if (g == 0) a.ws_bsum[row * nprev + (seg - 1)] = S;
        }
        return;
    }

    // ---- per-channel partials (summed over batches and segments by the reduction kernel) ----
    const int64_t rs = row * a.nseg + seg;
    if (active) {
        if (a.dinitial_state && seg == 0)
            *reinterpret_cast<float4*>(a.dinitial_state + row * kN + 4 * g) =
                make_float4(gad[0], gad[1], gad[2], gad[3]);
        constexpr float sc = 1.f / kScale;  // the dA terms were taken with Delta * kScale
        *reinterpret_cast<float4*>(a.ws_dA + rs * kN + 4 * g) =
            make_float4(dA_acc[0] * sc, dA_acc[1] * sc, dA_acc[2] * sc, dA_acc[3] * sc);
    }
    dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, 1);
    dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, 2);
    db_acc += __shfl_xor_sync(0xffffffffu, db_acc, 1);
    db_acc += __shfl_xor_sync(0xffffffffu, db_acc, 2);
    if (active && g == 0) {
        a.ws_dD[rs] = dD_acc;
        a.ws_db[rs] = db_acc;
    }
}

// Adds the per-CTA / per-row partials in a fixed order: dB, dC over channel blocks; dA, dD,
// dbias over batches.
__global__ void scan_bwd_reduce_kernel(const BwdArgs a, int64_t nblk) {
    const int64_t L = a.seqlen;
    const int64_t nbc = a.batch * L * kBSlots;            // dB and dC entries
    const int64_t nda = a.dim * kN;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nbc + nda + 2 * a.dim;
         i += stride) {
        if (i < nbc) {  // i = (b * L + t) * 32 + slot
            const int64_t slot = i % kBSlots, t = (i / kBSlots) % L, b = i / (kBSlots * L);
            float s = 0.f;
            for (int64_t k = 0; k < nblk; ++k) s += a.ws_part[k * nbc + i];
            float* dst = slot < kN ? a.dB : a.dC;
            dst[(b * kN + (slot % kN)) * L + t] = s;
        } else if (i < nbc + nda) {
            const int64_t j = i - nbc;  // d*16 + n
            const int64_t d = j / kN, n = j % kN;
            float s = 0.f;
            for (int64_t b = 0; b < a.batch; ++b)
                for (int k = 0; k < a.nseg; ++k) s += a.ws_dA[((b * a.dim + d) * a.nseg + k) * kN + n];
            a.dA[j] = s;
        } else {
            const int64_t j = i - nbc - nda;
            const int64_t dd = j % a.dim;
            const bool isD = j < a.dim;
            const float* src = isD ? a.ws_dD : a.ws_db;
            float s = 0.f;
            for (int64_t b = 0; b < a.batch; ++b)
                for (int k = 0; k < a.nseg; ++k) s += src[(b * a.dim + dd) * a.nseg + k];
            if (isD && a.dD) a.dD[dd] = s;
            if (!isD && a.ddelta_bias) a.ddelta_bias[dd] = s;
        }
    }
}

template <typename Tin, typename Tg, bool kPrecise, bool kVec, int kMode>
static void launch_bwd_one(const BwdArgs& a, dim3 grid, cudaStream_t stream) {
    // The contraction tiles (DS, K: the last members) only for the instantiation that uses them:
    // 3 CTAs per SM without them take 192 KB of shared memory and leave more of the SM's
    // 256 KB to the L1 cache.
    constexpr int smem_contract = (int)sizeof(BwdSmem);
    constexpr int smem_shuffle = (int)offsetof(BwdSmem, DS);
    if ((int64_t)grid.x * grid.y * grid.z <= (int64_t)a.sms * kBMinCtasRoomy) {
        auto k = scan_bwd_kernel<Tin, Tg, kPrecise, kVec, kMode, kBMinCtasRoomy>;
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_contract);
        k<<<grid, kBThreads, smem_contract, stream>>>(a);
    } else {
        auto k = scan_bwd_kernel<Tin, Tg, kPrecise, kVec, kMode, kBMinCtas>;
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_shuffle);
        k<<<grid, kBThreads, smem_shuffle, stream>>>(a);
    }
}

template <typename Tin, typename Tg, bool kPrecise, bool kVec>
static cudaError_t launch_bwd_modes(const BwdArgs& a, unsigned gx, cudaStream_t stream) {
    if (a.nseg > 1) {  // the local passes: forward over segments 0..S-2, adjoint over 1..S-1
        const dim3 grid(gx, (unsigned)(a.nseg - 1), (unsigned)a.batch);
        if (!a.ckpt_given) launch_bwd_one<Tin, Tg, kPrecise, kVec, kBwdFwdLocal>(a, grid, stream);
        launch_bwd_one<Tin, Tg, kPrecise, kVec, kBwdAdjLocal>(a, grid, stream);
    }
    launch_bwd_one<Tin, Tg, kPrecise, kVec, kBwdFull>(a, dim3(gx, (unsigned)a.nseg, (unsigned)a.batch), stream);
    return cudaGetLastError();
}

template <typename Tin, typename Tg, bool kPrecise>
static cudaError_t launch_bwd_typed(const BwdArgs& a, cudaStream_t stream) {
    const unsigned gx = (unsigned)((a.dim + kBRows - 1) / kBRows);
    cudaError_t e = a.seqlen % 4 == 0 ? launch_bwd_modes<Tin, Tg, kPrecise, true>(a, gx, stream)
                                      : launch_bwd_modes<Tin, Tg, kPrecise, false>(a, gx, stream);
    if (e != cudaSuccess) return e;
    scan_bwd_reduce_kernel<<<4 * 148, 256, 0, stream>>>(a, (int64_t)gx);
    return cudaGetLastError();
}

cudaError_t launch_scan_bwd(const BwdArgs& a, bool in_bf16, bool grad_bf16, cudaStream_t stream) {
    using bf = __nv_bfloat16;
    if (in_bf16) {
        return grad_bf16 ? launch_bwd_typed<bf, bf, false>(a, stream)
                         : launch_bwd_typed<bf, float, false>(a, stream);
    }
    return grad_bf16 ? launch_bwd_typed<float, bf, true>(a, stream)
                     : launch_bwd_typed<float, float, true>(a, stream);
}

BwdWorkspace scan_bwd_workspace(int64_t batch, int64_t dim, int64_t seqlen, int nseg,
                                bool with_ckpt) {
    const int64_t rows = batch * dim;
    const int64_t nchunks = (seqlen + kBChunk - 1) / kBChunk;
    const int64_t nblk = (dim + kBRows - 1) / kBRows;
    const int64_t nprev = nseg - 1;
    auto up = [](int64_t x) { return (x + 63) / 64 * 64; };  // 256-byte alignment
    BwdWorkspace w{};
    int64_t o = 0;
    w.ckpt = o; o += with_ckpt ? up(rows * nchunks * kN) : 0;
    w.part = o; o += up(nblk * batch * seqlen * kBSlots);
    w.dA = o; o += up(rows * nseg * kN);
    w.dD = o; o += up(rows * nseg);
    w.db = o; o += up(rows * nseg);
    w.hloc = o; o += up(rows * nprev * kN);
    w.fsum = o; o += up(rows * nprev);
    w.gloc = o; o += up(rows * nprev * kN);
    w.bsum = o; o += up(rows * nprev);
    w.total = o;
    return w;
}

int scan_bwd_chunk_tokens() { return kBChunk; }
int scan_bwd_rows_per_cta() { return kBRows; }
int scan_bwd_ctas_per_sm() { return kBMinCtas; }
int scan_bwd_ctas_per_sm_roomy() { return kBMinCtasRoomy; }

}  // namespace selscan
