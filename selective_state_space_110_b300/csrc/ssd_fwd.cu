// Mamba-2 state space duality (SSD) layer for sm_103a: chunks of 128 tokens on the tcgen05
// tensor cores, the state carried from chunk to chunk in tensor memory.
//
// "Mamba and State Space Models" (world.lapla.si), section "Mamba-2": with A a number times the
// identity, a head's layer is one lower-triangular matrix, entry (i, j) = C_i . B_j times all
// the decay between steps j and i. Mamba-2 cuts the sequence into chunks: inside a chunk it
// multiplies matrices on the tensor cores; between chunks only the state is passed on. Per
// (batch b, head h) and chunk, with Delta_t = softplus(dt + dt_bias), a_t = Delta_t A_h, cs the
// running sum of a inside the chunk (inclusive) and S the state (dstate x headdim) before it:
//   G  = C B^T                                               (128 x 128, K = dstate)
//   M  = G * exp(cs_i - cs_j) * Delta_j  for j <= i, else 0  (the chunk's block of the matrix)
//   Y  = M X + exp(cs_i) * (C S) + D x, then times silu(z)   (X: the chunk's x, 128 x headdim)
//   S <- exp(cs_last) S + B^T (w * X),  w_j = exp(cs_last - cs_j) * Delta_j
// which is the recurrence H_t = exp(a_t) H_{t-1} + Delta_t x_t B_t^T, y_t = C_t . H_t + D x_t
// evaluated a chunk at a time.
//
// One CTA per (b, h) walks the chunks in order; 256 threads, thread (row, half) serving
// tensor-memory lane `row` (the chunk's token row, or the state row n) and one half of the
// columns. C, B and X arrive by TMA into 128-byte-swizzled tiles (the layout the MMA
// descriptors read). The four products run as tcgen05.mma (bf16 operands, fp32 accumulators in
// tensor memory), issued by one thread and completed through mbarriers; the threads move data
// between tensor memory, registers and shared memory in between. The operands the kernel
// derives (M, w * X and the state S) are fp32 values; each is passed to the tensor cores as
// the sum of two bf16 matrices (hi = bf16(v), lo = bf16(v - hi)), two MMAs accumulating into
// the same result, so the products keep about 16 significand bits. B, C and x are bf16 inputs
// and enter exactly.
//
// Tensor memory (512 columns, one CTA per SM): [0,128) G, [128,192) M X, [192,256) C S,
// [256,320) the state S (row n, column p), fp32.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "selscan_device.cuh"
#include "selscan_launch.h"
#include "sm100_async.cuh"

namespace selscan {

constexpr int kQ = 128;              // tokens per chunk (the MMA's M)
constexpr int kHeadDim = 64;         // P
constexpr int kSsdState = 128;       // N
constexpr int kSsdThreads = 256;
constexpr int kTile = 16384;         // one 128-row x 128-byte swizzled tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColG = 0, kColYd = 128, kColYo = 192, kColS = 256;

// Shared-memory tiles, kTile bytes each from a 1024-byte aligned base.
enum SsdTile : int {
    kTC0 = 0, kTC1,    // C of the chunk: rows i, states 0..63 | 64..127 (K-major)
    kTB0, kTB1,        // B: rows j, states 0..63 | 64..127 (K-major for G, MN-major for B^T)
    kTX,               // x: rows j, headdim 0..63 (MN-major)
    kTGH0, kTGH1,      // M hi: rows i, columns j 0..63 | 64..127 (K-major)
    kTGL0, kTGL1,      // M lo
    kTSH, kTSL,        // state S hi / lo: rows n, headdim 0..63 (MN-major)
    kTXH, kTXL,        // w * X hi / lo: rows j, headdim (MN-major)
    kNumTiles
};
constexpr int kSsdSmemBytes = kNumTiles * kTile + 1024;

__device__ unsigned int g_ssd_status;

// Byte offset of 16-byte chunk `ch` (0..7) of row `r` in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128(int r, int ch) {
    return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 lo, __nv_bfloat16 hi) {
    return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

// Eight fp32 values -> 16-byte chunks of their bf16 hi and lo parts.
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * e]), h1 = __float2bfloat16_rn(v[2 * e + 1]);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * e] - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * e + 1] - __bfloat162float(h1));
        h[e] = pack2(h0, h1);
        l[e] = pack2(l0, l1);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void unpack8(const uint4& r, float* v) {
    v[0] = bf16lo(r.x); v[1] = bf16hi(r.x); v[2] = bf16lo(r.y); v[3] = bf16hi(r.y);
    v[4] = bf16lo(r.z); v[5] = bf16hi(r.z); v[6] = bf16lo(r.w); v[7] = bf16hi(r.w);
}

template <typename Tout>
__device__ __forceinline__ void store32(Tout* dst, const float (&v)[32]);
template <>
__device__ __forceinline__ void store32<float>(float* dst, const float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
        reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}
template <>
__device__ __forceinline__ void store32<__nv_bfloat16>(__nv_bfloat16* dst, const float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            w[e] = pack2(__float2bfloat16_rn(v[8 * q + 2 * e]), __float2bfloat16_rn(v[8 * q + 2 * e + 1]));
        reinterpret_cast<uint4*>(dst)[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <typename Tout>
__global__ void __launch_bounds__(kSsdThreads, 1)
    ssd_fwd_kernel(const SsdArgs a, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC) {
    extern __shared__ uint8_t dyn_smem[];
    __shared__ unsigned long long bar_tma, bar_g1, bar_g2, bar_g4;
    __shared__ uint32_t tmem_slot;
    __shared__ float s_cs[kQ];  // running sum of Delta*A*log2(e) in the chunk, inclusive
    __shared__ float s_dl[kQ];  // Delta
    __shared__ float s_wsum[4];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    auto tile = [&](int i) { return sm + i * kTile; };
    auto tile_addr = [&](int i) { return smem_u32(sm) + (uint32_t)(i * kTile); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;  // tensor-memory lane this thread reads and writes
    const int h = blockIdx.x, b = blockIdx.y;
    const int64_t H = a.nheads, L = a.seqlen;
    const int g = (int)(h / (H / a.ngroups));
    const float A2 = a.A[h] * kLog2e;
    const float bias = a.dt_bias ? a.dt_bias[h] : 0.f;
    const float Dh = a.D ? a.D[h] : 0.f;
    const int nchunks = (int)((L + kQ - 1) / kQ);
    const __nv_bfloat16* dt = static_cast<const __nv_bfloat16*>(a.dt);
    const __nv_bfloat16* zp = static_cast<const __nv_bfloat16*>(a.z);
    Tout* yp = static_cast<Tout*>(a.y);

    if (warp == 0) tmem_alloc(&tmem_slot, kTmemCols);
    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_g1, 1);
        mbar_init(&bar_g2, 1);
        mbar_init(&bar_g4, 1);
        fence_mbar_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const uint32_t tlane = (uint32_t)(quarter * 32) << 16;

    // S (hi / lo) for the next C S product: row n = row, headdim columns 32*half..+31.
    auto put_state_split = [&](const float (&v)[32]) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 hi, lo;
            split8(&v[8 * q], hi, lo);
            *reinterpret_cast<uint4*>(tile(kTSH) + sw128(row, 4 * half + q)) = hi;
            *reinterpret_cast<uint4*>(tile(kTSL) + sw128(row, 4 * half + q)) = lo;
        }
    };

    bool has_state = a.initial_state != nullptr;
    bool ok = true;
    if (has_state) {  // initial state (p, n) -> S[n][p]
        float v[32];
        const float* src = a.initial_state + ((int64_t)b * H + h) * kHeadDim * kSsdState + row;
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = src[(int64_t)(32 * half + i) * kSsdState];
        tmem_st32(tmem + tlane + kColS + 32 * half, v);
        put_state_split(v);
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    for (int c = 0; c < nchunks; ++c) {
        const int64_t t0 = (int64_t)c * kQ;
        const uint32_t par = (uint32_t)(c & 1);
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar_tma, 5 * kTile);
            tma_load_4d(tile(kTC0), &tmC, &bar_tma, 0, g, (int)t0, b);
            tma_load_4d(tile(kTC1), &tmC, &bar_tma, 64, g, (int)t0, b);
            tma_load_4d(tile(kTB0), &tmB, &bar_tma, 0, g, (int)t0, b);
            tma_load_4d(tile(kTB1), &tmB, &bar_tma, 64, g, (int)t0, b);
            tma_load_4d(tile(kTX), &tmX, &bar_tma, 0, h, (int)t0, b);
        }
        // Delta and the running sum of Delta*A over the chunk (one token per thread of warps 0-3).
        if (tid < kQ) {
            const int64_t t = t0 + tid;
            float dl = 0.f;  // tokens past the end: no step, no decay
            if (t < L) {
                const float v = __bfloat162float(dt[((int64_t)b * L + t) * H + h]) + bias;
                dl = a.softplus ? softplus_f<true>(v) : v;
            }
            float s = dl * A2;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += n;
            }
            if (lane == 31) s_wsum[warp] = s;
            s_dl[tid] = dl;
            s_cs[tid] = s;
        }
        __syncthreads();
        if (tid < kQ) {
            float off = 0.f;
            for (int w = 0; w < warp; ++w) off += s_wsum[w];
            s_cs[tid] += off;
        }
        ok = mbar_wait_bounded(&bar_tma, par);
        if (!__syncthreads_and(ok)) { ok = false; break; }
        tc_fence_after_sync();

        // G = C B^T; with a carried state also C S (hi + lo).
        if (tid == 0) {
            const uint32_t i_g1 = umma_idesc_bf16(128, 128, false, false);
#pragma unroll 1
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = (uint32_t)(k & 3) * 32;
                umma_bf16(tmem + kColG, umma_desc_sw128(tile_addr(kTC0 + (k >> 2)) + off, 16, 1024),
                          umma_desc_sw128(tile_addr(kTB0 + (k >> 2)) + off, 16, 1024), i_g1, k > 0);
            }
            if (has_state) {
                const uint32_t i_g3 = umma_idesc_bf16(128, 64, false, true);
#pragma unroll 1
                for (int part = 0; part < 2; ++part)
#pragma unroll 1
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t off = (uint32_t)(k & 3) * 32;
                        umma_bf16(tmem + kColYo,
                                  umma_desc_sw128(tile_addr(kTC0 + (k >> 2)) + off, 16, 1024),
                                  umma_desc_sw128(tile_addr(part ? kTSL : kTSH) + (uint32_t)k * 2048, kTile, 1024),
                                  i_g3, (part | k) != 0);
                    }
            }
            umma_commit(&bar_g1);
        }
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar_g1, par));
        tc_fence_after_sync();

        // M = G * exp(cs_i - cs_j) * Delta_j (j <= i) as bf16 hi / lo, row i = row, columns
        // 64*half..+63 (tile kTGH0 + half).
        if (ok) {
            const float cs_i = s_cs[row];
            const bool live = t0 + row < L;
#pragma unroll 1
            for (int part = 0; part < 2; ++part) {
                float v[32];
                tmem_ld32(tmem + tlane + kColG + 64 * half + 32 * part, v);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float m[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = 64 * half + 32 * part + 8 * q + e;
                        m[e] = (live && j <= row) ? v[8 * q + e] * ex2_approx(cs_i - s_cs[j]) * s_dl[j] : 0.f;
                    }
                    uint4 hi, lo;
                    split8(m, hi, lo);
                    *reinterpret_cast<uint4*>(tile(kTGH0 + half) + sw128(row, 4 * part + q)) = hi;
                    *reinterpret_cast<uint4*>(tile(kTGL0 + half) + sw128(row, 4 * part + q)) = lo;
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        if (!__syncthreads_and(ok)) { ok = false; break; }
        tc_fence_after_sync();

        // Y_diag = (M hi + M lo) X.
        if (tid == 0) {
            const uint32_t i_g2 = umma_idesc_bf16(128, 64, false, true);
#pragma unroll 1
            for (int part = 0; part < 2; ++part)
#pragma unroll 1
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (uint32_t)(k & 3) * 32;
                    umma_bf16(tmem + kColYd,
                              umma_desc_sw128(tile_addr((part ? kTGL0 : kTGH0) + (k >> 2)) + off, 16, 1024),
                              umma_desc_sw128(tile_addr(kTX) + (uint32_t)k * 2048, kTile, 1024), i_g2,
                              (part | k) != 0);
                }
            umma_commit(&bar_g2);
        }
        // Meanwhile: w * X (hi / lo) for the state update (warps 0-3, row j = row), and the
        // decay of the carried state by exp(cs_last) (warps 4-7, state row n = row).
        const float cs_last = s_cs[kQ - 1];
        if (half == 0) {
            const float w = ex2_approx(cs_last - s_cs[row]) * s_dl[row];
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                float v[8];
                unpack8(*reinterpret_cast<const uint4*>(tile(kTX) + sw128(row, ch)), v);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] *= w;
                uint4 hi, lo;
                split8(v, hi, lo);
                *reinterpret_cast<uint4*>(tile(kTXH) + sw128(row, ch)) = hi;
                *reinterpret_cast<uint4*>(tile(kTXL) + sw128(row, ch)) = lo;
            }
        } else if (has_state) {
            const float dec = ex2_approx(cs_last);
#pragma unroll 1
            for (int part = 0; part < 2; ++part) {
                float v[32];
                tmem_ld32(tmem + tlane + kColS + 32 * part, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= dec;
                tmem_st32(tmem + tlane + kColS + 32 * part, v);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();

        // S (+)= B^T (w X): A = B^T (MN-major, states in two 64-blocks), B = w X (MN-major).
        if (tid == 0) {
            const uint32_t i_g4 = umma_idesc_bf16(128, 64, true, true);
#pragma unroll 1
            for (int part = 0; part < 2; ++part)
#pragma unroll 1
                for (int k = 0; k < 8; ++k)
                    umma_bf16(tmem + kColS,
                              umma_desc_sw128(tile_addr(kTB0) + (uint32_t)k * 2048, kTile, 1024),
                              umma_desc_sw128(tile_addr(part ? kTXL : kTXH) + (uint32_t)k * 2048, kTile, 1024),
                              i_g4, (has_state || part || k) ? 1u : 0u);
            umma_commit(&bar_g4);
        }

        // y = Y_diag + exp(cs_i) * (C S) + D x, times silu(z): row i = row, headdim
        // columns 32*half..+31.
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar_g2, par));
        tc_fence_after_sync();
        if (ok) {
            float yd[32], yo[32];
            tmem_ld32(tmem + tlane + kColYd + 32 * half, yd);
            if (has_state) tmem_ld32(tmem + tlane + kColYo + 32 * half, yo);
            const int64_t t = t0 + row;
            if (t < L) {
                const float e = has_state ? ex2_approx(s_cs[row]) : 0.f;
                const int64_t off = (((int64_t)b * L + t) * H + h) * kHeadDim + 32 * half;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float xv[8], zv[8];
                    unpack8(*reinterpret_cast<const uint4*>(tile(kTX) + sw128(row, 4 * half + q)), xv);
                    if (zp) unpack8(*reinterpret_cast<const uint4*>(zp + off + 8 * q), zv);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float y = yd[8 * q + i] + Dh * xv[i];
                        if (has_state) y = fmaf(e, yo[8 * q + i], y);
                        if (zp) y *= silu_f<false>(zv[i]);
                        yd[8 * q + i] = y;
                    }
                }
                store32<Tout>(yp + off, yd);
            }
        }

        // The updated state -> hi / lo for the next chunk's C S.
        ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded(&bar_g4, par));
        tc_fence_after_sync();
        if (ok) {
            float v[32];
            tmem_ld32(tmem + tlane + kColS + 32 * half, v);
            put_state_split(v);
        }
        has_state = true;
        fence_proxy_async_smem();
        tc_fence_before_sync();
        if (!__syncthreads_and(ok)) { ok = false; break; }
        tc_fence_after_sync();
    }

    if (ok && a.final_state) {  // S[n][p] -> final_state (p, n)
        float v[32];
        if (has_state) {
            tmem_ld32(tmem + tlane + kColS + 32 * half, v);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        float* dst = a.final_state + ((int64_t)b * H + h) * kHeadDim * kSsdState + row;
#pragma unroll
        for (int i = 0; i < 32; ++i) dst[(int64_t)(32 * half + i) * kSsdState] = v[i];
    }
    if (!ok && tid == 0) atomicOr(&g_ssd_status, 1u);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---- host side ---------------------------------------------------------------------------------

namespace {

PFN_cuTensorMapEncodeTiled_v12000 ssd_encode_fn() {
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

// bf16 tensor (inner, d1, seqlen, batch), contiguous; box = 64 inner x 1 x 128 tokens x 1,
// 128-byte swizzle; tokens past seqlen read as zeros.
cudaError_t make_ssd_map(CUtensorMap* m, const void* base, int64_t inner, int64_t d1,
                         int64_t seqlen, int64_t batch) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = ssd_encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)d1, (cuuint64_t)seqlen, (cuuint64_t)batch};
    cuuint64_t strides[3] = {(cuuint64_t)(inner * 2), (cuuint64_t)(inner * d1 * 2),
                             (cuuint64_t)(inner * d1 * seqlen * 2)};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)kQ, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <typename Tout>
cudaError_t launch_ssd_typed(const SsdArgs& a, cudaStream_t stream) {
    CUtensorMap mX{}, mB{}, mC{};
    if (a.seqlen > 0) {
        cudaError_t e = make_ssd_map(&mX, a.x, kHeadDim, a.nheads, a.seqlen, a.batch);
        if (e == cudaSuccess) e = make_ssd_map(&mB, a.B, kSsdState, a.ngroups, a.seqlen, a.batch);
        if (e == cudaSuccess) e = make_ssd_map(&mC, a.C, kSsdState, a.ngroups, a.seqlen, a.batch);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaFuncSetAttribute(ssd_fwd_kernel<Tout>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSsdSmemBytes);
    if (e != cudaSuccess) return e;
    ssd_fwd_kernel<Tout><<<dim3((unsigned)a.nheads, (unsigned)a.batch), kSsdThreads, kSsdSmemBytes,
                           stream>>>(a, mX, mB, mC);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ssd_fwd(const SsdArgs& a, bool out_bf16, cudaStream_t stream) {
    return out_bf16 ? launch_ssd_typed<__nv_bfloat16>(a, stream) : launch_ssd_typed<float>(a, stream);
}

cudaError_t read_ssd_status(unsigned int* status, bool reset, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(status, g_ssd_status, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && reset) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_ssd_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                    stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    return e;
}

}  // namespace selscan
