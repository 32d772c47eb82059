// Chunked selective scan (S6 forward) for sm_103a.
//
// What is computed ("Mamba and State Space Models", world.lapla.si, sections "A State of
// Fixed Size", "Chosen by the Token" and "A Scan on the Chip"): per row (b, d) and token t,
//   Delta = softplus(delta + bias), h[n] = exp(Delta*A[d,n]) h[n] + Delta*B[b,n,t]*u,
//   y = (sum_n C[b,n,t] h[n] + D[d] u) * silu(z).
// As on that page, the inputs are read once from HBM, discretised and scanned on chip, and
// only y (plus the final state) is written back; the per-token state never leaves registers.
//
// Cost model on B300 (148 SMs; per SM and clock: 32 ex2 on the SFU, 128 fp32 FMA lanes, one
// warp-instruction per scheduler, and one shared-memory wavefront = one 32-bit word delivered
// to each of 32 lanes). Every (t, n) needs one exp2 with its own argument and four fp32
// operations (Delta*A, k*B, the state FMA, the readout FMA): the SFU and the FMA pipe each
// allow 2 elements per clock per SM. Every (row, t) also needs all 16 B and 16 C values of
// token t in the registers of the lanes that hold the row's states; delivered from shared
// memory that is 32 words, one wavefront, per element, which would cap the scan at 1 element
// per clock. The layout below is built around those budgets:
//   - A quad of 4 lanes owns kR rows (b, d), (b, d+1).. of one batch; lane g keeps states
//     4g..4g+3 of each of its rows in registers and updates them with packed f32x2
//     operations. The B and C values a lane fetches for a token serve all kR of its rows, so
//     with kR = 2 the shared-memory delivery is half a wavefront per element.
//   - A CTA owns 32 consecutive channels of one batch and walks the sequence in chunks of
//     32/kR tokens. B and C of a chunk (shared by every channel of the batch) arrive by TMA
//     into a 3-deep ring of shared-memory stages, completion tracked by mbarriers, so their
//     fetch overlaps the scan of earlier chunks. The CTA converts them once to fp32, one
//     128-byte row per token (chunk c of token t at position c ^ (t & 7): conflict-free both
//     for the conversion stores and for the lanes' 16-byte loads).
//   - Each lane owns 8 consecutive tokens of one of its quad's rows: it loads them (one
//     128-bit load per tensor, issued one chunk ahead), computes Delta and k = Delta*u once per
//     element in registers, and its quad receives them by width-4 shuffles, which use no
//     shared-memory bandwidth. The exp2 arguments of two tokens come from one packed multiply.
//   - The quad's 4 partial readouts of a token are summed where the owner lane can use them.
//     With two rows per quad this is a reduce-scatter in registers (two exchange steps by
//     shuffles, no shared memory: step 1 pairs the lanes that hold the two rows in swapped
//     register slots, step 2 the lanes that own the two halves of the chunk); with one row,
//     each lane writes its partials to shared memory every 4 tokens and the owner sums them
//     at the end of the chunk. The owner applies the D skip and the silu gate (packed f32x2)
//     and stores its 8 outputs with one 128-bit store.
//   - Long sequences with few rows are cut into time segments that run in parallel
//     (grid.y). A first pass (kLocalEnd) scans segments 0..S-2 from a zero state and keeps
//     each segment's end state and summed Delta. The full pass then starts segment s from the
//     true state, folding the earlier segments with the associative combine of the
//     recurrence: h <- exp(A * sum Delta) h + h_local_end.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "selscan_device.cuh"
#include "selscan_launch.h"
#include "sm100_async.cuh"

namespace selscan {

constexpr int kRowsPerCta = 32;      // channels per CTA of the default geometry
constexpr int kMaxChunk = 32;  // time segments are multiples of this many tokens

// Geometry for kR rows per quad (and per lane) and kW warps per CTA. kR = 2 halves the B/C
// shared-memory traffic per element but also the number of warps; the launcher picks it per
// shape. The default CTA holds 32 channels; the wide CTA (8 warps, 128 channels of two rows
// per quad) is for the balanced launch, where its registers alone keep it to one CTA per SM.
constexpr int kWideWarps = 8;
constexpr int kPdlTrigger = 1, kPdlWaitStart = 2, kPdlWaitEnd = 4;  // ScanArgs::pdl bits
template <int kR, int kW = 4 / kR>
struct Geo {
    static_assert(kR == 1 || kR == 2, "rows per lane must be 1 or 2");
    static constexpr int kWarps = kW;
    static constexpr int kThreads = 32 * kWarps;
    static constexpr int kRowsPerWarp = 8 * kR;
    static constexpr int kRowsPerCta = kRowsPerWarp * kWarps;
    static constexpr int kChunk = 32 / kR;      // tokens per chunk: each lane owns 8 of one row
    static constexpr int kBlocks = kChunk / 4;  // 4-token blocks per chunk
    static constexpr int kMinCtas = kW != 4 / kR ? 1 : kR == 1 ? 5 : 6;  // register budget
};


// Error bits a kernel can raise; read (and cleared) by read_device_status().
__device__ unsigned int g_device_status;

enum class Mode { kFull, kLocalEnd };

template <int kInBytes, int kR>
struct ScanStages {
    static constexpr int kStages = 3;
    static constexpr int kTileBytes = 16 * Geo<kR>::kChunk * kInBytes;
};

template <int kInBytes, int kR, int kW>
struct __align__(128) ScanSmem {
    using St = ScanStages<kInBytes, kR>;
    static constexpr int kChunk = Geo<kR>::kChunk;
    // TMA destinations: raw B and C tiles, [stage][B|C][n][t] in the input dtype.
    unsigned char raw[St::kStages][2][St::kTileBytes];
    // fp32 B/C per token: 8 chunks of 4 floats (B states 0-15, C states 0-15); chunk c of
    // token t sits at position c ^ (t & 7).
    float bc[2][kChunk][32];
    // Partial readouts: [warp][row of the quad][4-token block][slot] with slot = lane ^ swz.
    float4 red[kW][kR][Geo<kR>::kBlocks][32];
    unsigned long long full[St::kStages];
};

// ---- 8-token raw vectors of u / delta / z ---------------------------------------------------

template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
    uint4 v;
};
template <>
struct Raw8<float> {
    float4 a, b;
};

// Loads p[0..7] (one or two 128-bit streaming loads; the vector path only ever sees 0 or 8
// valid tokens) or zeros.
__device__ __forceinline__ void load_raw(Raw8<__nv_bfloat16>& r, const __nv_bfloat16* p, bool ok) {
    r.v = ok ? __ldcs(reinterpret_cast<const uint4*>(p)) : make_uint4(0, 0, 0, 0);
}
__device__ __forceinline__ void load_raw(Raw8<float>& r, const float* p, bool ok) {
    if (ok) {
        r.a = __ldcs(reinterpret_cast<const float4*>(p));
        r.b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    } else {
        r.a = r.b = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}
__device__ __forceinline__ void unpack(const Raw8<__nv_bfloat16>& r, float (&v)[8]) {
    v[0] = bf16lo(r.v.x); v[1] = bf16hi(r.v.x); v[2] = bf16lo(r.v.y); v[3] = bf16hi(r.v.y);
    v[4] = bf16lo(r.v.z); v[5] = bf16hi(r.v.z); v[6] = bf16lo(r.v.w); v[7] = bf16hi(r.v.w);
}
__device__ __forceinline__ void unpack(const Raw8<float>& r, float (&v)[8]) {
    v[0] = r.a.x; v[1] = r.a.y; v[2] = r.a.z; v[3] = r.a.w;
    v[4] = r.b.x; v[5] = r.b.y; v[6] = r.b.z; v[7] = r.b.w;
}

// ---- zero-order hold: Bbar = Delta*B * phi(x), phi(x) = (exp(x) - 1)/x, x = Delta*A ----
__device__ __forceinline__ float inv_or_zero(float v) { return v != 0.f ? 1.f / v : 0.f; }
// fp32 inputs: m = expm1(x) from the library; phi(0) = 1.
__device__ __forceinline__ float phi_exact(float m, float x) { return x != 0.f ? m / x : 1.f; }
// bf16 inputs: x2 = x*log2(e) (the SFU argument), abar = 2^x2, inv_a = 1/A, dinv = 1/Delta.
// For |x| < 1/16 the Taylor series 1 + x/2 + x^2/6 + x^3/24 (truncation below 1e-7
// relative); above, (abar - 1)/(A*Delta), where abar - 1 has lost no significant digits.
__device__ __forceinline__ float phi_fast(float x2, float abar, float inv_a, float dinv) {
    const float x = x2 * 0.69314718055994531f;
    const float p = fmaf(fmaf(fmaf(x, 1.f / 24.f, 1.f / 6.f), x, 0.5f), x, 1.f);
    return fabsf(x) < 0.0625f ? p : (abar - 1.f) * inv_a * dinv;
}

// Compensated (Kahan) accumulation of an increment into a pair of state numbers: nc holds the
// negated rounding error not yet added. t = h + (inc + nc) is rounded; (h - t) + y recovers
// what the rounding dropped (exactly, since t and h are close).
__device__ __forceinline__ void kahan_step(float2& h, float2& nc, float2 inc) {
    const float2 y = __fadd2_rn(inc, nc);
    const float2 t = __fadd2_rn(h, y);
    nc = __fadd2_rn(__fadd2_rn(h, make_float2(-t.x, -t.y)), y);
    h = t;
}

// Owner lane (within the quad) of row j, token t of a chunk, and its register slot t & 7.
template <int kR>
__device__ __forceinline__ constexpr int owner_of(int j, int t) {
    return kR == 1 ? (t >> 3) : (2 * j + (t >> 3));
}
// XOR swizzle of the partial-readout slots of (row j, block q); the reader of block q of row j
// is the owner lane swz(j, q), so each quarter-warp of its loads hits 8 distinct bank groups.
template <int kR>
__device__ __forceinline__ constexpr int red_swz(int j, int q) {
    return kR == 1 ? ((q >> 1) & 3) : ((2 * j + (q >> 1)) & 3);
}

template <int kR, typename Tin, typename Tout, bool kVec, bool kPrecise, bool kZoh, Mode kMode,
          bool kCkpt = false, int kW = 4 / kR>
__global__ void __launch_bounds__(Geo<kR, kW>::kThreads, Geo<kR, kW>::kMinCtas)
    scan_kernel(const ScanArgs a, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC) {
    constexpr bool kFull = kMode == Mode::kFull;
    using Gm = Geo<kR, kW>;
    constexpr int kThreads = Gm::kThreads;
    constexpr int kRowsPerWarp = Gm::kRowsPerWarp;
    constexpr int kRowsPerCta = Gm::kRowsPerCta;
    constexpr int kChunk = Gm::kChunk;
    constexpr int kBlocks = Gm::kBlocks;
    using St = ScanStages<sizeof(Tin), kR>;
    constexpr int kS = St::kStages;
    __shared__ ScanSmem<sizeof(Tin), kR, kW> sm;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int quad = lane >> 2;
    const int g = lane & 3;  // quarter of the state owned by this lane
    // This CTA's block of 32 channels and time segment (grid: channel blocks x segments x
    // batches, offset by bx0 / b0 when only some blocks are cut into segments).
    // (Only the wide CTA of the balanced plan is offset or skips blocks; the default geometry
    // always starts at block 0.)
    constexpr bool kOffset = kW == kWideWarps;
    if constexpr (kOffset) {
        if (a.pdl & kPdlWaitStart) asm volatile("griddepcontrol.wait;" ::: "memory");
        if (a.pdl & kPdlTrigger) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    // Before any exit of a launch that must not finish ahead of the grids before it.
    auto pdl_exit = [&]() {
        if constexpr (kOffset) {
            if (a.pdl & kPdlWaitEnd) asm volatile("griddepcontrol.wait;" ::: "memory");
        }
    };
    const int64_t b = kOffset ? a.b0 + blockIdx.z : (int64_t)blockIdx.z;
    const int seg = blockIdx.y;
    const int64_t bx = kOffset ? a.bx0 + blockIdx.x : (int64_t)blockIdx.x;
    // The whole-block launch of the balanced plan leaves the blocks its segments cover.
    if (kOffset && a.skip_bx0 >= 0 && b == a.skip_b && bx >= a.skip_bx0) {
        pdl_exit();
        return;
    }
    const int64_t dim = a.dim;
    const int64_t d0 = bx * kRowsPerCta + warp * kRowsPerWarp + quad * kR;
    const int64_t L = a.seqlen;
    const int64_t t_begin = (int64_t)seg * a.seg_len;
    const int64_t t_end = min(L, t_begin + a.seg_len);
    const int nchunks = t_end > t_begin ? (int)((t_end - t_begin + kChunk - 1) / kChunk) : 0;
    const int nprev = a.nseg - 1;  // segments with a stored local end state
    // First workspace row of this quad: rows of the cut blocks, in the launch's block order.
    auto ws_row0 = [&]() -> int64_t {
        return ((int64_t)blockIdx.z * gridDim.x + blockIdx.x) * kRowsPerCta + warp * kRowsPerWarp + quad * kR;
    };

    // Rows of this quad; inactive rows (past dim) compute on row 0's parameters and store nothing.
    // With two rows per quad the full pass sums the quad's partial readouts in registers
    // (kQuadSum, below); for that, register slot j of lane g holds row j ^ (g >> 1) of the quad,
    // so slot 0 is always the row the lane owns.
    constexpr bool kQuadSum = kR == 2 && kFull;
    const int jbit = kQuadSum ? (g >> 1) : 0;
    bool act[kR];
    int64_t row[kR];
#pragma unroll
    for (int j = 0; j < kR; ++j) {
        act[j] = d0 + (j ^ jbit) < dim;
        row[j] = b * dim + (act[j] ? d0 + (j ^ jbit) : 0);
    }
    // The row and tokens this lane owns: Delta, k, the epilogue and the stores.
    const int jo = kR == 1 ? 0 : (g >> 1);
    const int to = 8 * (kR == 1 ? g : (g & 1));
    const bool own_act = kQuadSum ? act[0] : act[jo];
    const int64_t own_row = kQuadSum ? row[0] : row[jo];
    const int64_t own_d = own_row - b * dim;
    // Lane (within the quad) that owns slot j's row for tokens 8h..8h+7 of a chunk.
    int src_lane[kR][2];
#pragma unroll
    for (int j = 0; j < kR; ++j) {
        src_lane[j][0] = owner_of<kR>(j ^ jbit, 0);
        src_lane[j][1] = owner_of<kR>(j ^ jbit, 8);
    }

    // ---- TMA ring: initialise the barriers and start the first stages ----
    if (kVec) {
        if (tid == 0) {
#pragma unroll
            for (int s = 0; s < kS; ++s) mbar_init(&sm.full[s], 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (tid == 0) {
            for (int c = 0; c < kS && c < nchunks; ++c) {
                const int x = (int)(t_begin + (int64_t)c * kChunk);
                mbar_arrive_expect_tx(&sm.full[c], (kFull ? 2 : 1) * St::kTileBytes);
                tma_load_2d(sm.raw[c][0], &tmB, &sm.full[c], x, (int)(b * kN));
                if (kFull) tma_load_2d(sm.raw[c][1], &tmC, &sm.full[c], x, (int)(b * kN));
            }
        }
    }

    // Per-row constants: A for states 4g..4g+3, pre-scaled by log2(e) for the SFU exp2, as
    // (A_n, A_n) pairs so that one packed multiply forms the arguments of two tokens.
    float4 A4[kR], invA[kR];  // invA: 1/A (natural units), zero-order hold only
    float2 aa[kR][4];
#pragma unroll
    for (int j = 0; j < kR; ++j) {
        A4[j] = *reinterpret_cast<const float4*>(a.A + (row[j] - b * dim) * kN + 4 * g);
        if (kZoh) invA[j] = make_float4(inv_or_zero(A4[j].x), inv_or_zero(A4[j].y),
                                        inv_or_zero(A4[j].z), inv_or_zero(A4[j].w));
        if (!kPrecise) {
            A4[j].x *= kLog2e; A4[j].y *= kLog2e; A4[j].z *= kLog2e; A4[j].w *= kLog2e;
        }
        aa[j][0] = f2(A4[j].x); aa[j][1] = f2(A4[j].y); aa[j][2] = f2(A4[j].z); aa[j][3] = f2(A4[j].w);
    }
    const float bias = a.delta_bias ? a.delta_bias[own_d] : 0.f;
    const float Dd = a.D ? a.D[own_d] : 0.f;

    // ---- initial state, then fold the local end states of earlier segments ----
    float2 h01[kR], h23[kR];
    // fp32 inputs: Kahan compensation of each state number (the negated rounding error still
    // to be added). A decay exp(Delta*A) within a few ulp of 1 changes the state by less than
    // half an ulp per token, which plain fp32 rounding drops at every token, the same way
    // each time (up to L/2 ulp of bias over L tokens; at Delta ~ 1e-8 that is 1.4e-5 relative
    // after 384 tokens). The compensated sum keeps those increments.
    float2 nc01[kR], nc23[kR];
#pragma unroll
    for (int j = 0; j < kR; ++j) {
        h01[j] = make_float2(0.f, 0.f);
        h23[j] = make_float2(0.f, 0.f);
        nc01[j] = make_float2(0.f, 0.f);
        nc23[j] = make_float2(0.f, 0.f);
        if (!kFull) continue;
        if (a.initial_state) {
            const float4 s = *reinterpret_cast<const float4*>(a.initial_state + row[j] * kN + 4 * g);
            h01[j] = make_float2(s.x, s.y); h23[j] = make_float2(s.z, s.w);
        }
        for (int i = 0; i < seg; ++i) {
            const int64_t sr = ws_row0() + (j ^ jbit);
            const float ds = a.ws_dsum[sr * nprev + i];
            const float4 hl = *reinterpret_cast<const float4*>(a.ws_hloc + (sr * nprev + i) * kN + 4 * g);
            if (kPrecise) {  // exp(A*S) h + h_local, with exp written as 1 + expm1
                const float m0 = expm1f(A4[j].x * ds), m1 = expm1f(A4[j].y * ds);
                const float m2 = expm1f(A4[j].z * ds), m3 = expm1f(A4[j].w * ds);
                h01[j] = make_float2(fmaf(m0, h01[j].x, h01[j].x) + hl.x, fmaf(m1, h01[j].y, h01[j].y) + hl.y);
                h23[j] = make_float2(fmaf(m2, h23[j].x, h23[j].x) + hl.z, fmaf(m3, h23[j].y, h23[j].y) + hl.w);
            } else {
                const float p0 = ex2_approx(A4[j].x * ds), p1 = ex2_approx(A4[j].y * ds);
                const float p2 = ex2_approx(A4[j].z * ds), p3 = ex2_approx(A4[j].w * ds);
                h01[j] = make_float2(fmaf(p0, h01[j].x, hl.x), fmaf(p1, h01[j].y, hl.y));
                h23[j] = make_float2(fmaf(p2, h23[j].x, hl.z), fmaf(p3, h23[j].y, hl.w));
            }
        }
    }

    const Tin* __restrict__ u_row = static_cast<const Tin*>(a.u) + own_row * L;
    const Tin* __restrict__ d_row = static_cast<const Tin*>(a.delta) + own_row * L;
    const Tin* __restrict__ z_row = a.z ? static_cast<const Tin*>(a.z) + own_row * L : nullptr;
    Tout* __restrict__ o_row = static_cast<Tout*>(a.out) + own_row * L;
    const Tin* __restrict__ Bb = static_cast<const Tin*>(a.B) + b * kN * L;
    const Tin* __restrict__ Cb = static_cast<const Tin*>(a.C) + b * kN * L;

    // Offsets (floats) of this lane's B chunk g ^ m within a token row, for m = 0..3; chunk
    // positions for t & 7 = m are g ^ m (+16 floats when m >= 4) for B and the other half for C.
    int offB[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) offB[m] = 4 * (g ^ m);

    float dsum = 0.f, dsum_c = 0.f;  // Kahan sum of Delta over owned tokens (kLocalEnd)

    // The vector path prefetches the next chunk's 8 owned tokens into registers.
    Raw8<Tin> nu, nd, nz;
    if (kVec && nchunks > 0) {
        const int64_t tl = t_begin + to;
        const bool ok = own_act && tl < t_end;
        load_raw(nu, u_row + tl, ok);
        load_raw(nd, d_row + tl, ok);
        if (kFull && z_row) load_raw(nz, z_row + tl, ok);
    }

    bool timed_out = false;
    for (int c = 0; c < nchunks; ++c) {
        const int64_t t0 = t_begin + (int64_t)c * kChunk;
        const int stage = c % kS;
        const uint32_t parity = (uint32_t)((c / kS) & 1);
        const int buf = c & 1;
        const int64_t tl = t0 + to;
        const int64_t left = t_end - tl;
        const int nval = !own_act || left <= 0 ? 0 : (left >= 8 ? 8 : (int)left);

        // ---- this lane's 8 owned tokens of u, delta (and z) ----
        float uf[8], df[8], zf[8];
        if (kVec) {
            unpack(nu, uf);
            unpack(nd, df);
            if (kFull && z_row) unpack(nz, zf);
            if (c + 1 < nchunks) {  // prefetch the next chunk
                const int64_t tn = tl + kChunk;
                const bool ok = own_act && tn < t_end;
                load_raw(nu, u_row + tn, ok);
                load_raw(nd, d_row + tn, ok);
                if (kFull && z_row) load_raw(nz, z_row + tn, ok);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uf[i] = i < nval ? to_f32(u_row[tl + i]) : 0.f;
                df[i] = i < nval ? to_f32(d_row[tl + i]) : 0.f;
                if (kFull && z_row) zf[i] = i < nval ? to_f32(z_row[tl + i]) : 0.f;
            }
        }

        // ---- Delta and k = Delta*u of the owned tokens; padding tokens get Delta = 0 ----
        float dl[8], kl[8];
        {
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                float2 x = __fadd2_rn(make_float2(df[i], df[i + 1]), f2(bias));
                float2 dt;
                if (!a.softplus) {
                    dt = x;
                } else if (kPrecise) {
                    dt = make_float2(softplus_f<true>(x.x), softplus_f<true>(x.y));
                } else {
                    dt = softplus2(x);
                }
                dl[i] = dt.x; dl[i + 1] = dt.y;
            }
            if (nval < 8) {
#pragma unroll
                for (int i = 0; i < 8; ++i) dl[i] = i < nval ? dl[i] : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                const float2 kv = __fmul2_rn(make_float2(dl[i], dl[i + 1]), make_float2(uf[i], uf[i + 1]));
                kl[i] = kv.x; kl[i + 1] = kv.y;
            }
            if (!kFull) {  // Kahan-compensated running sum of Delta over the segment
                float part = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) part += dl[i];
                const float yk = part - dsum_c;
                const float tk = dsum + yk;
                dsum_c = (tk - dsum) - yk;
                dsum = tk;
            }
        }

        // ---- B and C of this chunk -> fp32 per-token rows (item = chunk-column x token) ----
        if (kVec && !mbar_wait_bounded(&sm.full[stage], parity)) timed_out = true;
        constexpr int kItems = kChunk * (kFull ? 8 : 4);  // (token, 4-state chunk) pairs
        if constexpr (kVec && kFull && kW == kWideWarps && 2 * kItems == kThreads) {
            // The wide CTA: one half chunk (2 states) per thread, so that no thread idles. Lane
            // order (half, token, chunk): a half-warp's 8-byte stores cover 8 tokens x 2 halves,
            // 16 distinct bank pairs through the XOR swizzle.
            const int hf = tid & 1, tt = (tid >> 1) % kChunk, ch = (tid >> 1) / kChunk;
            const int isC = ch >> 2, q = ch & 3;
            const Tin* tile = reinterpret_cast<const Tin*>(sm.raw[stage][isC]);
            const float2 v = make_float2(to_f32(tile[(4 * q + 2 * hf + 0) * kChunk + tt]),
                                         to_f32(tile[(4 * q + 2 * hf + 1) * kChunk + tt]));
            *reinterpret_cast<float2*>(&sm.bc[buf][tt][4 * (ch ^ (tt & 7)) + 2 * hf]) = v;
        } else
#pragma unroll
        for (int cc = 0; cc < (kItems + kThreads - 1) / kThreads; ++cc) {
            const int item = tid + kThreads * cc;
            if (kItems < kThreads && item >= kItems) break;
            const int tt = item % kChunk;
            const int ch = item / kChunk;  // 0..7: B quads 0-3, C quads 0-3
            const int isC = ch >> 2, q = ch & 3;
            float4 v;
            if (kVec) {
                const Tin* tile = reinterpret_cast<const Tin*>(sm.raw[stage][isC]);
                v.x = to_f32(tile[(4 * q + 0) * kChunk + tt]);
                v.y = to_f32(tile[(4 * q + 1) * kChunk + tt]);
                v.z = to_f32(tile[(4 * q + 2) * kChunk + tt]);
                v.w = to_f32(tile[(4 * q + 3) * kChunk + tt]);
            } else {
                const Tin* src = isC ? Cb : Bb;
                const int64_t t = t0 + tt;
                const bool ok = t < t_end;
                v.x = ok ? to_f32(src[(4 * q + 0) * L + t]) : 0.f;
                v.y = ok ? to_f32(src[(4 * q + 1) * L + t]) : 0.f;
                v.z = ok ? to_f32(src[(4 * q + 2) * L + t]) : 0.f;
                v.w = ok ? to_f32(src[(4 * q + 3) * L + t]) : 0.f;
            }
            *reinterpret_cast<float4*>(&sm.bc[buf][tt][4 * (ch ^ (tt & 7))]) = v;
        }
        if (__syncthreads_or(timed_out)) {
            // A B/C stage never arrived: record it and leave, after giving the copies this
            // CTA still has in flight a bounded chance to land.
            if (tid == 0) {
                atomicOr(&g_device_status, 1u);
                for (int k = 1; k < kS && c + k < nchunks; ++k)
                    mbar_wait_bounded(&sm.full[(c + k) % kS], (uint32_t)(((c + k) / kS) & 1));
            }
            pdl_exit();
            return;
        }
        // Every thread has read stage `stage`: refill it with chunk c + kS.
        if (kVec && tid == 0 && c + kS < nchunks) {
            const int x = (int)(t0 + (int64_t)kS * kChunk);
            mbar_arrive_expect_tx(&sm.full[stage], (kFull ? 2 : 1) * St::kTileBytes);
            tma_load_2d(sm.raw[stage][0], &tmB, &sm.full[stage], x, (int)(b * kN));
            if (kFull) tma_load_2d(sm.raw[stage][1], &tmC, &sm.full[stage], x, (int)(b * kN));
        }

        // ---- the recurrence over the chunk's tokens, 4 at a time ----
        const float* const bcb = &sm.bc[buf][0][0];
        float wk[2][4];  // kQuadSum: blocks 0 and 1 summed over lanes g and g ^ 2
        float Yo[8];     // kQuadSum: the quad's sums of the lane's 8 owned tokens
#pragma unroll
        for (int q = 0; q < kBlocks; ++q) {
            // The state before every 16th token, for a backward pass that reuses it.
            if (kCkpt && kFull && (q & 3) == 0) {
                const int64_t tq = t0 + 4 * q;
                if (tq < t_end) {
                    const int64_t nck = (L + 15) / 16;
#pragma unroll
                    for (int j = 0; j < kR; ++j)
                        if (act[j])
                            *reinterpret_cast<float4*>(a.ckpt + (row[j] * nck + tq / 16) * kN + 4 * g) =
                                make_float4(h01[j].x, h01[j].y, h23[j].x, h23[j].y);
                }
            }
            // exp2 arguments of tokens (4q, 4q+1) and (4q+2, 4q+3), per row and state
            float2 ea[kR][4], eb[kR][4];
            float dq[kR][4];
#pragma unroll
            for (int j = 0; j < kR; ++j) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = 4 * q + e;
                    const int src = kQuadSum ? src_lane[j][(t >> 3) & 1] : owner_of<kR>(j, t);
                    dq[j][e] = __shfl_sync(0xffffffffu, dl[t & 7], src, 4);
                }
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    ea[j][n] = __fmul2_rn(make_float2(dq[j][0], dq[j][1]), aa[j][n]);
                    eb[j][n] = __fmul2_rn(make_float2(dq[j][2], dq[j][3]), aa[j][n]);
                }
            }
            float yq[kR][4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = 4 * q + e;
                const int m = t & 7;
                const float* rowp = bcb + 32 * t + offB[m & 3];
                const float4 Bv = *reinterpret_cast<const float4*>(rowp + ((m & 4) ? 16 : 0));
                const float4 Cv = *reinterpret_cast<const float4*>(rowp + ((m & 4) ? 0 : 16));
#pragma unroll
                for (int j = 0; j < kR; ++j) {
                    const int src = kQuadSum ? src_lane[j][(t >> 3) & 1] : owner_of<kR>(j, t);
                    const float kt = __shfl_sync(0xffffffffu, kl[t & 7], src, 4);
                    const float2 kk = f2(kt);
                    float arg[4];
#pragma unroll
                    for (int n = 0; n < 4; ++n)
                        arg[n] = e == 0 ? ea[j][n].x : e == 1 ? ea[j][n].y : e == 2 ? eb[j][n].x : eb[j][n].y;
                    float2 kb01 = __fmul2_rn(kk, make_float2(Bv.x, Bv.y));
                    float2 kb23 = __fmul2_rn(kk, make_float2(Bv.z, Bv.w));
                    if (kPrecise) {
                        // Abar = 1 + expm1(Delta*A): the decay's distance from 1 keeps full
                        // relative precision, so a slowly decaying state accumulates no bias
                        // from rounding Abar itself.
                        const float2 m01 = make_float2(expm1f(arg[0]), expm1f(arg[1]));
                        const float2 m23 = make_float2(expm1f(arg[2]), expm1f(arg[3]));
                        if (kZoh) {  // Bbar = Delta*B * (exp(x)-1)/x with x = Delta*A
                            kb01 = __fmul2_rn(kb01, make_float2(phi_exact(m01.x, arg[0]), phi_exact(m01.y, arg[1])));
                            kb23 = __fmul2_rn(kb23, make_float2(phi_exact(m23.x, arg[2]), phi_exact(m23.y, arg[3])));
                        }
                        // h <- h + (m h + kb), summed with compensation.
                        kahan_step(h01[j], nc01[j], __ffma2_rn(m01, h01[j], kb01));
                        kahan_step(h23[j], nc23[j], __ffma2_rn(m23, h23[j], kb23));
                    } else {
                        const float2 ab01 = make_float2(ex2_approx(arg[0]), ex2_approx(arg[1]));
                        const float2 ab23 = make_float2(ex2_approx(arg[2]), ex2_approx(arg[3]));
                        if (kZoh) {  // Bbar = Delta*B * (exp(x)-1)/x with x = Delta*A
                            const float dinv = rcp_approx(dq[j][e]);
                            kb01 = __fmul2_rn(kb01, make_float2(phi_fast(arg[0], ab01.x, invA[j].x, dinv),
                                                                phi_fast(arg[1], ab01.y, invA[j].y, dinv)));
                            kb23 = __fmul2_rn(kb23, make_float2(phi_fast(arg[2], ab23.x, invA[j].z, dinv),
                                                                phi_fast(arg[3], ab23.y, invA[j].w, dinv)));
                        }
                        h01[j] = __ffma2_rn(ab01, h01[j], kb01);
                        h23[j] = __ffma2_rn(ab23, h23[j], kb23);
                    }
                    if (kFull) {
                        float2 y2 = __fmul2_rn(make_float2(Cv.x, Cv.y), h01[j]);
                        y2 = __ffma2_rn(make_float2(Cv.z, Cv.w), h23[j], y2);
                        yq[j][e] = y2.x + y2.y;
                    }
                }
            }
            if constexpr (kQuadSum) {
                // The quad's sums of the block's 4 readouts of each of its 2 rows, reduce-
                // scattered in registers. Step 1 (lanes g, g ^ 2): slot 0 (the own row) plus the
                // partner's slot 1, which holds the same row.
                float w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) w[e] = yq[0][e] + __shfl_xor_sync(0xffffffffu, yq[1][e], 2);
                if (q < 2) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) wk[q][e] = w[e];
                } else {
                    // Step 2 (lanes g, g ^ 1), with block q - 2: lane g keeps the block in the
                    // half of the chunk it owns (tokens 8 (g & 1)..) and adds the partner's copy.
                    const bool hi = (g & 1) != 0;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float keep = hi ? w[e] : wk[q - 2][e], send = hi ? wk[q - 2][e] : w[e];
                        Yo[4 * (q - 2) + e] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
                    }
                }
            } else if (kFull) {
#pragma unroll
                for (int j = 0; j < kR; ++j)
                    sm.red[warp][j][q][lane ^ red_swz<kR>(j, q)] =
                        make_float4(yq[j][0], yq[j][1], yq[j][2], yq[j][3]);
            }
        }

        if (kFull) {
            // ---- sum the quad's partial readouts of the owned tokens ----
            float2 Y[4];
            if constexpr (kQuadSum) {
#pragma unroll
                for (int i = 0; i < 4; ++i) Y[i] = make_float2(Yo[2 * i], Yo[2 * i + 1]);
            } else {
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i) Y[i] = make_float2(0.f, 0.f);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int q = to / 4 + jj;
#pragma unroll
                    for (int gp = 0; gp < 4; ++gp) {
                        const float4 v = sm.red[warp][jo][q][(4 * quad + gp) ^ g];
                        Y[2 * jj] = __fadd2_rn(Y[2 * jj], make_float2(v.x, v.y));
                        Y[2 * jj + 1] = __fadd2_rn(Y[2 * jj + 1], make_float2(v.z, v.w));
                    }
                }
            }
            // ---- D skip, silu gate, store ----
            float out8[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float2 y = __ffma2_rn(f2(Dd), make_float2(uf[2 * i], uf[2 * i + 1]), Y[i]);
                if (z_row) {
                    const float2 zz = make_float2(zf[2 * i], zf[2 * i + 1]);
                    y = __fmul2_rn(y, kPrecise ? make_float2(silu_f<true>(zz.x), silu_f<true>(zz.y))
                                               : silu2(zz));
                }
                out8[2 * i] = y.x; out8[2 * i + 1] = y.y;
            }
            store8<Tout, kVec>(o_row + tl, nval, out8);
            if (!kQuadSum) __syncwarp();  // the partials are read before the next chunk rewrites them
        }
    }

    if (kPrecise) {  // fold in what the compensation still holds
#pragma unroll
        for (int j = 0; j < kR; ++j) {
            h01[j] = __fadd2_rn(h01[j], nc01[j]);
            h23[j] = __fadd2_rn(h23[j], nc23[j]);
        }
    }
    if (kFull) {
        if (a.final_state && seg == a.nseg - 1) {
#pragma unroll
            for (int j = 0; j < kR; ++j)
                if (act[j])
                    *reinterpret_cast<float4*>(a.final_state + row[j] * kN + 4 * g) =
                        make_float4(h01[j].x, h01[j].y, h23[j].x, h23[j].y);
        }
    } else {
        // Each owner lane summed Delta over its tokens of every chunk; the row's total is the
        // sum over the row's owner lanes (all 32 lanes take part in the shuffles).
        float s = dsum - dsum_c;
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        if (kR == 1) s += __shfl_xor_sync(0xffffffffu, s, 2);
#pragma unroll
        for (int j = 0; j < kR; ++j)
            if (act[j])
                *reinterpret_cast<float4*>(a.ws_hloc + ((ws_row0() + j) * nprev + seg) * kN + 4 * g) =
                    make_float4(h01[j].x, h01[j].y, h23[j].x, h23[j].y);
        if (own_act && (kR == 1 ? g == 0 : (g & 1) == 0)) a.ws_dsum[(ws_row0() + jo) * nprev + seg] = s;
    }
    pdl_exit();
}

// ---- host side ---------------------------------------------------------------------------------

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// Map of B or C viewed as a 2-D array (batch*16 rows, seqlen tokens); box = one chunk x 16 rows.
cudaError_t make_bc_map(CUtensorMap* m, const void* base, int64_t batch, int64_t seqlen,
                        bool bf16, int chunk) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const size_t es = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {(cuuint64_t)seqlen, (cuuint64_t)(batch * kN)};
    cuuint64_t strides[1] = {(cuuint64_t)(seqlen * es)};
    cuuint32_t box[2] = {(cuuint32_t)chunk, (cuuint32_t)kN};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                    const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The launches of one scan with kW warps per CTA (see ScanArgs for the three plans).
template <int kR, typename Tin, typename Tout, bool kVec, bool kPrecise, bool kZoh = false,
          int kW = 4 / kR>
cudaError_t launch_typed(const ScanArgs& args, int64_t batch, cudaStream_t stream) {
    using G = Geo<kR, kW>;
    CUtensorMap mB{}, mC{};
    if (kVec && args.seqlen > 0) {
        const bool bf = sizeof(Tin) == 2;
        cudaError_t e = make_bc_map(&mB, args.B, batch, args.seqlen, bf, G::kChunk);
        if (e == cudaSuccess) e = make_bc_map(&mC, args.C, batch, args.seqlen, bf, G::kChunk);
        if (e != cudaSuccess) return e;
    }
    const unsigned gx = (unsigned)((args.dim + G::kRowsPerCta - 1) / G::kRowsPerCta);
    auto full_kernel = [&]() {
        if constexpr (!kZoh) {
            if (args.ckpt) return scan_kernel<kR, Tin, Tout, kVec, kPrecise, kZoh, Mode::kFull, true, kW>;
        }
        return scan_kernel<kR, Tin, Tout, kVec, kPrecise, kZoh, Mode::kFull, false, kW>;
    };
    constexpr auto local_kernel = scan_kernel<kR, Tin, Tout, kVec, kPrecise, kZoh, Mode::kLocalEnd, false, kW>;
    auto launch = [&](auto kernel, dim3 grid, const ScanArgs& a) -> cudaError_t {
        if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
        if (a.pdl & (kPdlWaitStart | kPdlWaitEnd)) {  // may start before the launch before it ends
            cudaLaunchConfig_t cfg{};
            cfg.gridDim = grid;
            cfg.blockDim = dim3(G::kThreads, 1, 1);
            cfg.dynamicSmemBytes = 0;
            cfg.stream = stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a, mB, mC);
            return e != cudaSuccess ? e : cudaGetLastError();
        }
        kernel<<<grid, G::kThreads, 0, stream>>>(a, mB, mC);
        return cudaGetLastError();
    };
    cudaError_t e = cudaSuccess;
    if (args.nsplit == 0) {  // whole blocks only
        ScanArgs a = args;
        a.nseg = 1; a.seg_len = std::max<int64_t>(a.seqlen, 1); a.bx0 = 0; a.b0 = 0; a.skip_bx0 = -1;
        a.pdl = 0;
        return launch(full_kernel(), dim3(gx, 1, (unsigned)batch), a);
    }
    if (args.nfull == 0) {  // every block cut into segments
        ScanArgs a = args;
        a.bx0 = 0; a.b0 = 0; a.skip_bx0 = -1;
        a.pdl = 0;
        if (a.nseg > 1) e = launch(local_kernel, dim3(gx, (unsigned)(a.nseg - 1), (unsigned)batch), a);
        if (e == cudaSuccess) e = launch(full_kernel(), dim3(gx, (unsigned)a.nseg, (unsigned)batch), a);
        return e;
    }
    // Balanced: the cut blocks are the last nsplit blocks of the last batch. Local-end pass of
    // their first nseg-1 segments, the whole blocks (one CTA per SM), then their segments.
    // The three launches overlap their starts (programmatic dependent launch): the whole
    // blocks start on the SMs the local-end pass leaves free and wait for it before they exit;
    // the segments, which fold its results, wait for the whole-block grid (and so for both) before
    // they begin, but are already launched when it ends.
    const int64_t bx_cut = (int64_t)gx - args.nsplit;
    ScanArgs cut = args;
    cut.bx0 = bx_cut; cut.b0 = batch - 1; cut.skip_bx0 = -1;
    cut.pdl = kPdlTrigger;
    e = launch(local_kernel, dim3((unsigned)args.nsplit, (unsigned)(args.nseg - 1), 1), cut);
    if (e != cudaSuccess) return e;
    ScanArgs whole = args;
    whole.nseg = 1; whole.seg_len = std::max<int64_t>(whole.seqlen, 1); whole.bx0 = 0; whole.b0 = 0;
    whole.skip_bx0 = bx_cut; whole.skip_b = batch - 1;
    whole.pdl = kPdlTrigger | kPdlWaitEnd;
    e = launch(full_kernel(), dim3(gx, 1, (unsigned)batch), whole);
    if (e != cudaSuccess) return e;
    cut.pdl = kPdlWaitStart;
    return launch(full_kernel(), dim3((unsigned)args.nsplit, (unsigned)args.nseg, 1), cut);
}

// Two rows per lane only for the fast bf16 vector path (the shapes where it pays off); every
// other input combination runs one row per lane. The balanced plan runs the wide CTA, which
// only the fast bf16 path has.
template <typename Tin, typename Tout>
cudaError_t launch_io(const ScanArgs& a, int64_t batch, bool vec, bool precise,
                      cudaStream_t stream) {
    if (a.zoh) {  // zero-order hold: one row per lane, every load path
        if (vec) {
            return precise ? launch_typed<1, Tin, Tout, true, true, true>(a, batch, stream)
                           : launch_typed<1, Tin, Tout, true, false, true>(a, batch, stream);
        }
        return precise ? launch_typed<1, Tin, Tout, false, true, true>(a, batch, stream)
                       : launch_typed<1, Tin, Tout, false, false, true>(a, batch, stream);
    }
    if constexpr (sizeof(Tin) == 2) {
        if (vec && !precise && a.wide)
            return launch_typed<2, Tin, Tout, true, false, false, kWideWarps>(a, batch, stream);
        if (vec && !precise && a.rows_per_lane == 2)
            return launch_typed<2, Tin, Tout, true, false>(a, batch, stream);
    }
    if (vec) {
        return precise ? launch_typed<1, Tin, Tout, true, true>(a, batch, stream)
                       : launch_typed<1, Tin, Tout, true, false>(a, batch, stream);
    }
    return precise ? launch_typed<1, Tin, Tout, false, true>(a, batch, stream)
                   : launch_typed<1, Tin, Tout, false, false>(a, batch, stream);
}

}  // namespace

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

cudaError_t read_device_status(unsigned int* status, bool reset, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(status, g_device_status, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && reset && *status) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(zero), 0,
                                    cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    return e;
}

__global__ void wait_selftest_kernel(long long limit_cycles) {
    __shared__ unsigned long long bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // Phase 0 of `bar` never completes: nothing arrives on it.
    const long long start = clock64();
    bool done = false;
    while (!done && clock64() - start < limit_cycles) done = mbar_try_wait(&bar, 0);
    if (!done && threadIdx.x == 0) atomicOr(&g_device_status, 1u);
}

cudaError_t launch_wait_selftest(long long limit_cycles, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_cycles);
    return cudaGetLastError();
}

int scan_chunk_tokens() { return kMaxChunk; }
int scan_rows_per_cta() { return kRowsPerCta; }
int scan_ctas_per_sm(int rows_per_lane) {
    return rows_per_lane == 2 ? Geo<2>::kMinCtas : Geo<1>::kMinCtas;
}
int scan_wide_rows_per_cta() { return Geo<2, kWideWarps>::kRowsPerCta; }

}  // namespace selscan
