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
// One CTA per (b, h) walks the chunks in order: 320 threads, 8 worker warps, one issuing warp
// and one sums warp. Worker thread (row, half) serves tensor-memory lane `row` (the chunk's
// token row, or the state row n) and one half of the columns; lane 0 of the issuing warp starts
// every TMA load and every MMA; the sums warp computes each chunk's Delta and running sums (lane
// l: tokens 4l..4l+3) and the column factors of M's decay ahead of use, and publishes them once
// the workers have built the previous chunk's M. Within a 16-token piece k of columns,
// exp(cs_i - cs_j) Delta_j = 2^(cs_i - cs_16k) * [2^(cs_16k - cs_j) Delta_j]: the workers take
// one exp per row and piece; a piece whose decay exceeds 2^64 keeps one exp per element. C, B and x arrive by TMA into 128-byte-swizzled tiles, double-buffered so that the
// next chunk's tiles load while this one computes. The products run as tcgen05.mma (bf16 operands, fp32 accumulators in tensor
// memory); their completion reaches the workers through mbarriers (tcgen05.commit), and the
// workers hand finished operands to the issuer through mbarriers they arrive on.
//
// The workers are the busy side, so the tensor cores get their operands early and the workers
// never wait on a product in steady state. Per chunk c the workers (1) scale x by w and decay
// the state, (2) write the output of chunk c-1, (3) build M of chunk c, (4) split the updated
// state for the next C S. Meanwhile C B^T of chunk c (into
// the G buffer of c's parity, free since the output of c-2) and C S run before (1) ends, the
// state update during (2) and M X during (4) and the next chunk's (1). Chunk c's output is
// y = exp(cs_i) (C S) + M X + D x: C S and M X have accumulators of their own, so neither
// product waits for the other chunk's output to be read.
//
// The operands the kernel derives (M, w * X and the state S) are fp32 values; each enters the
// tensor cores as the sum of two bf16 matrices (hi = bf16(v), lo = bf16(v - hi)), which keeps
// about 16 significand bits: the hi and lo products accumulate into the same fp32 accumulator.
// M is written over the columns of G it comes from and read from there as the A operand of
// M X. B, C and x are bf16 inputs and enter exactly.
//
// Tensor memory (512 columns, one CTA per SM): [0,128) and [128,256) G of even and odd chunks,
// then M in place (columns [16k, 16k+8) M hi and [16k+8, 16k+16) M lo of j = 16k..16k+15, bf16
// pairs); [256,320) the state S (row n, column p); [320,384) and [384,448) C S of even and odd
// chunks; [448,512) M X.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "selscan_device.cuh"
#include "selscan_launch.h"
#include "sm100_async.cuh"

namespace selscan {

constexpr int kQ = 128;              // tokens per chunk (the MMA's M)
constexpr int kHeadDim = 64;         // P
constexpr int kSsdState = 128;       // N
constexpr int kWorkers = 256;        // threads that move data (8 warps)
constexpr int kSsdThreads = kWorkers + 64;  // plus a warp that issues TMA loads and MMAs and one
                                            // that computes each chunk's Delta sums
constexpr int kTile = 16384;         // one 128-row x 128-byte swizzled tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColG0 = 0, kColG1 = 128, kColS = 256, kColCS0 = 320, kColCS1 = 384, kColMX = 448;

// Shared-memory tiles, kTile bytes each from a 1024-byte aligned base. Input buffer s holds
// tiles 5s .. 5s+4: C (rows i, states 0..63 | 64..127; K-major), B (rows j, states 0..63 |
// 64..127; K-major for G, MN-major for B^T), x (rows j, headdim 0..63; MN-major).
constexpr int kInC = 0, kInB = 2, kInX = 4, kInTiles = 5;
constexpr int kTSH = 10, kTSL = 11;  // state hi | lo: rows n, headdim (MN-major), adjacent
constexpr int kTXH = 12, kTXL = 13;  // w * X hi | lo: rows j, headdim (MN-major), adjacent
constexpr int kNumTiles = 14;
// Largest decay (log2 units) over a 16-token piece for which M's decay is taken as a row factor
// times a column factor: 2^64 times Delta stays far inside the fp32 range.
constexpr float kFactorSpan = 64.f;
constexpr int kSsdSmemBytes = kNumTiles * kTile + 1024;

__device__ unsigned int g_ssd_status;

// Byte offset of 16-byte chunk `ch` (0..7) of row `r` in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128(int r, int ch) {
    return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4));
}

// A pair of fp32 values -> packed bf16 pairs of their hi and lo parts.
__device__ __forceinline__ void split2(float2 v, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
    const uint32_t hu = *reinterpret_cast<const uint32_t*>(&h);
    const float2 hf = make_float2(__uint_as_float(hu << 16), __uint_as_float(hu & 0xffff0000u));
    const float2 r = __ffma2_rn(hf, make_float2(-1.f, -1.f), v);
    const __nv_bfloat162 l = __floats2bfloat162_rn(r.x, r.y);
    hi = hu;
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Eight fp32 values -> 16-byte chunks of their bf16 hi and lo parts.
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
    split2(make_float2(v[0], v[1]), hi.x, lo.x);
    split2(make_float2(v[2], v[3]), hi.y, lo.y);
    split2(make_float2(v[4], v[5]), hi.z, lo.z);
    split2(make_float2(v[6], v[7]), hi.w, lo.w);
}

__device__ __forceinline__ void unpack8(const uint4& r, float* v) {
    v[0] = bf16lo(r.x); v[1] = bf16hi(r.x); v[2] = bf16lo(r.y); v[3] = bf16hi(r.y);
    v[4] = bf16lo(r.z); v[5] = bf16hi(r.z); v[6] = bf16lo(r.w); v[7] = bf16hi(r.w);
}

template <typename Tout>
__device__ __forceinline__ void store16(Tout* dst, const float (&v)[16]);
template <>
__device__ __forceinline__ void store16<float>(float* dst, const float (&v)[16]) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
        reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}
template <>
__device__ __forceinline__ void store16<__nv_bfloat16>(__nv_bfloat16* dst, const float (&v)[16]) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 p = __floats2bfloat162_rn(v[8 * q + 2 * e], v[8 * q + 2 * e + 1]);
            w[e] = *reinterpret_cast<const uint32_t*>(&p);
        }
        reinterpret_cast<uint4*>(dst)[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
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
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 p = __floats2bfloat162_rn(v[8 * q + 2 * e], v[8 * q + 2 * e + 1]);
            w[e] = *reinterpret_cast<const uint32_t*>(&p);
        }
        reinterpret_cast<uint4*>(dst)[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// D[tmem] (+)= A[tmem] * B[smem] (A: 128 rows in tensor-memory lanes, bf16 pairs along columns).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// The job of a CTA: chain ci = b * H + h, chunks [c_first, c_first + nchunks), and for a cut
// chain its index tc among the cut chains and its segment.
struct SsdJob {
    int64_t ci, tc;
    int c_first, nchunks, seg;
    bool cut;
};
__device__ __forceinline__ SsdJob ssd_job(const SsdArgs& a, int nchunks_all) {
    SsdJob j{0, 0, 0, nchunks_all, 0, false};
    if (a.job_mode == 0) {
        j.ci = (int64_t)blockIdx.y * a.nheads + blockIdx.x;
    } else if (a.job_mode == 3) {
        j.ci = blockIdx.x;
    } else {
        const int64_t k = blockIdx.x;
        const int per = a.job_mode == 1 ? a.nseg - 1 : a.nseg;  // jobs per cut chain
        j.tc = k / per;
        j.seg = (int)(k % per);
        j.ci = a.n_whole + j.tc;
        j.c_first = j.seg * a.seg_chunks;
        j.nchunks = min(a.seg_chunks, nchunks_all - j.c_first);
        j.cut = true;
    }
    return j;
}

// Initial state of a job (NULL = zeros), where its end state goes (NULL = nowhere), and where
// the local-end pass puts a segment's summed Delta*A.
__device__ __forceinline__ const float* ssd_job_init(const SsdArgs& a, const SsdJob& j) {
    constexpr int64_t kStateElems = (int64_t)kHeadDim * kSsdState;
    const float* chain_init = a.initial_state ? a.initial_state + j.ci * kStateElems : nullptr;
    if (!j.cut || j.seg == 0) return chain_init;
    if (a.job_mode == 1) return nullptr;  // a later segment's end state from zero (local end)
    return a.ws_sinit + (j.tc * (a.nseg - 1) + j.seg - 1) * kStateElems;  // folded
}
__device__ __forceinline__ float* ssd_job_final(const SsdArgs& a, const SsdJob& j) {
    constexpr int64_t kStateElems = (int64_t)kHeadDim * kSsdState;
    float* chain_final = a.final_state ? a.final_state + j.ci * kStateElems : nullptr;
    if (!j.cut) return chain_final;
    if (a.job_mode == 1) return a.ws_sloc + (j.tc * (a.nseg - 1) + j.seg) * kStateElems;
    return j.seg == a.nseg - 1 ? chain_final : nullptr;
}

// kStateOnly: the local-end jobs of the balanced launch, which need a segment's end state
// alone: per chunk the sums, w X and the state decay and update, no C B^T, C S, M, M X or output.
template <typename Tout, bool kStateOnly>
__global__ void __launch_bounds__(kSsdThreads, 1)
    ssd_fwd_kernel(const SsdArgs a, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC) {
    // The whole-chain launch that follows the local-end jobs does not depend on them: let it
    // start on the SMs they leave free.
    if (a.job_mode == 1) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ uint8_t dyn_smem[];
    // Completion of the TMA loads (per input buffer) and of the MMA groups (tcgen05.commit: G
    // per buffer, the state update, M X); hand-offs from the 256 worker threads to the issuer
    // (x ready, M ready, state split ready, output of a chunk read, per buffer).
    __shared__ unsigned long long bar_tma[2], bar_gg[2], bar_g4, bar_g2;
    __shared__ unsigned long long bar_x, bar_m, bar_s, bar_y[2];
    // The sums warp and the workers: a chunk's Delta and running sums are published (bar_sums),
    // and the workers' last reads of them are done (bar_free).
    __shared__ unsigned long long bar_sums, bar_free;
    __shared__ unsigned long long bar_drain;  // failure path: the issuer's MMAs in flight
    __shared__ uint32_t tmem_slot;
    __shared__ __align__(16) float s_cs[kQ];  // running sum of Delta*A*log2(e), inclusive
    __shared__ __align__(16) float s_w[kQ];   // w_j = 2^(cs_last - cs_j) * Delta_j
    // M's decay within 16-token piece k as a product: the column factor
    // 2^(cs_16k - cs_j) * Delta_j (Delta_j itself in pieces that are not factored), and the
    // piece's span cs_16k - cs_16k+15 (log2 units).
    __shared__ __align__(16) float s_cf[kQ];
    __shared__ float s_span[kQ / 16];
    __shared__ int s_ok;
    // Where this CTA's end state and (local-end jobs) summed Delta*A go, and whether it writes
    // y: set once by thread 0, read at the end, so that no register holds them meanwhile.
    __shared__ float* sh_final;
    __shared__ float* sh_dsum;
    __shared__ int sh_store_y;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    auto tile = [&](int i) { return sm + i * kTile; };
    auto tile_addr = [&](int i) { return smem_u32(sm) + (uint32_t)(i * kTile); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t H = a.nheads, L = a.seqlen;
    const int nchunks_all = (int)((L + kQ - 1) / kQ);
    // This CTA's job (one chain, or a segment of a cut chain in the balanced launch).
    const SsdJob job = ssd_job(a, nchunks_all);
    const int nchunks = job.nchunks;
    const int h = (int)(job.ci % H), b = (int)(job.ci / H);
    const int g = (int)(h / (H / a.ngroups));
    const int t_base = job.c_first * kQ;  // first token of this CTA's chunks (< 2^31)
    const bool init_state = ssd_job_init(a, job) != nullptr;
    if (tid == 0) {
        const bool local_end = a.job_mode == 1 && job.cut;  // writes no output
        sh_final = ssd_job_final(a, job);
        sh_dsum = local_end ? a.ws_dsum + job.tc * (a.nseg - 1) + job.seg : nullptr;
        sh_store_y = local_end ? 0 : 1;
    }

    if (warp == 0) tmem_alloc(&tmem_slot, kTmemCols);
    if (tid == 0) {
        mbar_init(&bar_tma[0], 1);
        mbar_init(&bar_tma[1], 1);
        mbar_init(&bar_gg[0], 1);
        mbar_init(&bar_gg[1], 1);
        mbar_init(&bar_g4, 1);
        mbar_init(&bar_g2, 1);
        mbar_init(&bar_x, kWorkers);
        mbar_init(&bar_m, kWorkers);
        mbar_init(&bar_s, kWorkers);
        mbar_init(&bar_y[0], kWorkers);
        mbar_init(&bar_y[1], kWorkers);
        mbar_init(&bar_sums, 32);
        mbar_init(&bar_drain, 1);
        mbar_init(&bar_free, kWorkers);
        fence_mbar_init();
        s_ok = 1;
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    const int row = quarter * 32 + lane;  // tensor-memory lane a worker thread reads and writes
    const uint32_t tlane = (uint32_t)(quarter * 32) << 16;
    // The state (row n = row, headdim columns 32*half..+31) -> hi / lo tiles.
    auto put_state_split = [&](const float (&v)[32]) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 hi, lo;
            split8(&v[8 * q], hi, lo);
            *reinterpret_cast<uint4*>(tile(kTSH) + sw128(row, 4 * half + q)) = hi;
            *reinterpret_cast<uint4*>(tile(kTSL) + sw128(row, 4 * half + q)) = lo;
        }
    };
    if (init_state && warp < kWorkers / 32) {  // initial state (p, n) -> S[n][p], split
        float v[32];
        const float* src = ssd_job_init(a, job) + row;
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = src[(int64_t)(32 * half + i) * kSsdState];
        tmem_st32(tmem + tlane + kColS + 32 * half, v);
        put_state_split(v);
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    if (warp == kWorkers / 32) {
        // ---------------- issuing thread: TMA loads and tensor-core products ----------------
        if (lane == 0 && nchunks > 0) {
            prefetch_tmap(&tmX);
            prefetch_tmap(&tmB);
            prefetch_tmap(&tmC);
            auto issue_tma = [&](int c) {  // chunk c -> input buffer c & 1
                const int base = kInTiles * (c & 1);
                unsigned long long* bar = &bar_tma[c & 1];
                // (the state-only jobs read no C)
                mbar_arrive_expect_tx(bar, (kStateOnly ? kInTiles - 2 : kInTiles) * kTile);
                const int tc0 = t_base + c * kQ;
                if (!kStateOnly) {
                    tma_load_4d(tile(base + kInC), &tmC, bar, 0, g, tc0, b);
                    tma_load_4d(tile(base + kInC + 1), &tmC, bar, 64, g, tc0, b);
                }
                tma_load_4d(tile(base + kInB), &tmB, bar, 0, g, tc0, b);
                tma_load_4d(tile(base + kInB + 1), &tmB, bar, 64, g, tc0, b);
                tma_load_4d(tile(base + kInX), &tmX, bar, 0, h, tc0, b);
            };
            // Waits for the output of chunk cc to be read (per-buffer barrier, one phase per
            // two chunks).
            auto wait_y = [&](int cc) { return mbar_wait_bounded(&bar_y[cc & 1], (uint32_t)((cc >> 1) & 1)); };
            issue_tma(0);
            if (nchunks > 1) issue_tma(1);
            int tma_issued = nchunks > 1 ? 2 : 1, tma_landed = 0;  // chunks
            const uint32_t i_g1 = umma_idesc_bf16(128, 128, false, false);  // C B^T
            const uint32_t i_cs = umma_idesc_bf16(128, 64, false, true);    // C S, M X
            const uint32_t i_s = umma_idesc_bf16(128, 64, true, true);      // B^T (w X)
            bool ok = true;
            if constexpr (kStateOnly) {
                for (int c = 0; c < nchunks && ok; ++c) {
                    const uint32_t par = (uint32_t)(c & 1);
                    const int in = kInTiles * (c & 1);
                    const bool had_state = c > 0 || init_state;
                    ok = mbar_wait_bounded(&bar_tma[c & 1], (uint32_t)((c >> 1) & 1));
                    if (ok) tma_landed = c + 1;
                    // S (+)= B^T (wX)_hi + B^T (wX)_lo, after the workers decayed S and wrote w X
                    if (ok) ok = mbar_wait_bounded(&bar_x, par);
                    if (!ok) break;
                    tc_fence_after_sync();
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            umma_bf16(tmem + kColS, umma_desc_sw128(tile_addr(in + kInB) + (uint32_t)k * 2048, kTile, 1024),
                                      umma_desc_sw128(tile_addr(part ? kTXL : kTXH) + (uint32_t)k * 2048, kTile, 1024), i_s,
                                      (had_state || part || k) ? 1u : 0u);
                    umma_commit(&bar_g4);
                    // Once that product has read input buffer c & 1, it takes chunk c + 2.
                    if (c + 2 < nchunks) {
                        ok = mbar_wait_bounded(&bar_g4, par);
                        if (!ok) break;
                        issue_tma(c + 2);
                        tma_issued = c + 3;
                    }
                }
            } else {
                for (int c = 0; c < nchunks && ok; ++c) {
                    const int in = kInTiles * (c & 1);
                    const uint32_t par = (uint32_t)(c & 1);
                    const uint32_t gcol = (c & 1) ? kColG1 : kColG0;
                    const bool had_state = c > 0 || init_state;
                    ok = mbar_wait_bounded(&bar_tma[c & 1], (uint32_t)((c >> 1) & 1));
                    if (ok) tma_landed = c + 1;
                    // G buffer c & 1 (M of chunk c-2) and C S buffer c & 1 are free once the
                    // output of chunk c-2 has been read.
                    if (ok && c >= 2) ok = wait_y(c - 2);
                    if (!ok) break;
                    tc_fence_after_sync();
                    // G = C B^T
    #pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t off = (uint32_t)(k & 3) * 32;
                        umma_bf16(tmem + gcol, umma_desc_sw128(tile_addr(in + kInC + (k >> 2)) + off, 16, 1024),
                                  umma_desc_sw128(tile_addr(in + kInB + (k >> 2)) + off, 16, 1024), i_g1, k > 0);
                    }
                    umma_commit(&bar_gg[c & 1]);
                    // C S = C S_hi + C S_lo, the state as it was before this chunk
                    if (had_state) {
                        if (c > 0) {
                            ok = mbar_wait_bounded(&bar_s, par ^ 1u);
                            if (!ok) break;
                            tc_fence_after_sync();
                        }
                        const uint32_t ccol = (c & 1) ? kColCS1 : kColCS0;
    #pragma unroll
                        for (int part = 0; part < 2; ++part)
    #pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const uint32_t off = (uint32_t)(k & 3) * 32;
                                umma_bf16(tmem + ccol, umma_desc_sw128(tile_addr(in + kInC + (k >> 2)) + off, 16, 1024),
                                          umma_desc_sw128(tile_addr(part ? kTSL : kTSH) + (uint32_t)k * 2048, kTile, 1024),
                                          i_cs, (part || k) ? 1u : 0u);
                            }
                    }
                    // S (+)= B^T (wX)_hi + B^T (wX)_lo, after the workers decayed S and wrote w X
                    ok = mbar_wait_bounded(&bar_x, par);
                    if (!ok) break;
                    tc_fence_after_sync();
    #pragma unroll
                    for (int part = 0; part < 2; ++part)
    #pragma unroll
                        for (int k = 0; k < 8; ++k)
                            umma_bf16(tmem + kColS, umma_desc_sw128(tile_addr(in + kInB) + (uint32_t)k * 2048, kTile, 1024),
                                      umma_desc_sw128(tile_addr(part ? kTXL : kTXH) + (uint32_t)k * 2048, kTile, 1024), i_s,
                                      (had_state || part || k) ? 1u : 0u);
                    umma_commit(&bar_g4);
                    // Once the previous chunk's output is read: its input buffer takes chunk c + 1,
                    // and the M X accumulator is free.
                    if (c > 0) {
                        ok = wait_y(c - 1);
                        if (!ok) break;
                        if (c + 1 < nchunks) {
                            issue_tma(c + 1);
                            tma_issued = c + 2;
                        }
                    }
                    // M X = M_hi X + M_lo X, M read from tensor memory (in place of G)
                    ok = mbar_wait_bounded(&bar_m, par);
                    if (!ok) break;
                    tc_fence_after_sync();
    #pragma unroll
                    for (int part = 0; part < 2; ++part)
    #pragma unroll
                        for (int k = 0; k < 8; ++k)
                            umma_bf16_ts(tmem + kColMX, tmem + gcol + 16 * k + (part ? 8 : 0),
                                         umma_desc_sw128(tile_addr(in + kInX) + (uint32_t)k * 2048, kTile, 1024), i_cs,
                                         (part || k) ? 1u : 0u);
                    umma_commit(&bar_g2);
                }
            }
            if (!ok) {
                // A wait gave up: record it, then give the copies and products this CTA still
                // has in flight a bounded chance to finish before the CTA leaves and frees its
                // tensor memory.
                s_ok = 0;
                for (int cc = tma_landed; cc < tma_issued; ++cc)
                    mbar_wait_bounded(&bar_tma[cc & 1], (uint32_t)((cc >> 1) & 1));
                umma_commit(&bar_drain);
                mbar_wait_bounded(&bar_drain, 0);
            }
        }
        __syncwarp();
    } else if (warp == kWorkers / 32 + 1) {
        // ---------------- sums warp: Delta and running sums of each chunk ----------------
        // Lane l takes tokens 4l .. 4l+3 of the chunk: softplus, a running sum over its four
        // tokens, then an inclusive scan of the lane totals across the warp.
        const float A2 = a.A[h] * kLog2e;
        const float bias = a.dt_bias ? a.dt_bias[h] : 0.f;
        const __nv_bfloat16* dt = static_cast<const __nv_bfloat16*>(a.dt);
        float raw[4];
        auto load_dt = [&](int c) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t t = (int64_t)(t_base + c * kQ + 4 * lane + i);
                raw[i] = (c < nchunks && t < L) ? __bfloat162float(dt[((int64_t)b * L + t) * H + h]) : 0.f;
            }
        };
        load_dt(0);
        bool ok = true;
        float dsum = 0.f;  // lane 31: the sum of the chunk totals
        for (int c = 0; c < nchunks; ++c) {
            float dl[4], al[4], cs[4];
            float run = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t t = (int64_t)(t_base + c * kQ + 4 * lane + i);
                const float v = raw[i] + bias;
                dl[i] = t < L ? (a.softplus ? softplus_f<true>(v) : v) : 0.f;
                al[i] = dl[i] * A2;
                run += al[i];
                cs[i] = run;
            }
            load_dt(c + 1);
            // Sums of the lane totals before this lane (the chunk), before it within its piece
            // of 4 lanes, and after it (the chunk): scans that add, never subtract, so that a
            // decay between nearby tokens keeps its precision however far the chunk decays.
            float incl = run, pincl = run, rincl = run;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
                const float r = __shfl_down_sync(0xffffffffu, rincl, o);
                if (lane + o < 32) rincl += r;
            }
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, pincl, o, 4);
                if ((lane & 3) >= o) pincl += n;
            }
            float excl = __shfl_up_sync(0xffffffffu, incl, 1);
            float pexcl = __shfl_up_sync(0xffffffffu, pincl, 1, 4);
            float after = __shfl_down_sync(0xffffffffu, rincl, 1);
            if (lane == 0) excl = 0.f;
            if ((lane & 3) == 0) pexcl = 0.f;
            if (lane == 31) after = 0.f;
            // The buffer held chunk c - 1: wait until the workers have read it (they have then
            // built that chunk's M; the next chunk's sums are ready by then).
            if (c >= 1) ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded(&bar_free, (uint32_t)((c - 1) & 1)));
            if (!ok) break;
            float csv[4], pl[4], wv[4];
            float suf = 0.f;  // the tokens after token i within this lane
#pragma unroll
            for (int i = 3; i >= 0; --i) {
                csv[i] = excl + cs[i];
                pl[i] = pexcl + cs[i];  // running sum from the piece's first token
                wv[i] = ex2_approx(suf + after) * dl[i];
                suf += al[i];
            }
            // piece k = lanes 4k..4k+3: its first token's sum sits in lane 4k, its last in 4k+3
            const float ref = __shfl_sync(0xffffffffu, pl[0], lane & ~3);
            const float span = ref - __shfl_sync(0xffffffffu, pl[3], lane | 3);
            const bool factored = fabsf(span) < kFactorSpan;
            float cf[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) cf[i] = factored ? ex2_approx(ref - pl[i]) * dl[i] : dl[i];
            *reinterpret_cast<float4*>(&s_w[4 * lane]) = make_float4(wv[0], wv[1], wv[2], wv[3]);
            *reinterpret_cast<float4*>(&s_cs[4 * lane]) = make_float4(csv[0], csv[1], csv[2], csv[3]);
            *reinterpret_cast<float4*>(&s_cf[4 * lane]) = make_float4(cf[0], cf[1], cf[2], cf[3]);
            if ((lane & 3) == 0) s_span[lane >> 2] = span;
            mbar_arrive(&bar_sums);
            dsum += incl;  // lane 31: the chunk's total
        }
        // the local-end pass: the segment's summed Delta*A*log2(e), for the fold
        if (ok && lane == 31 && sh_dsum) *sh_dsum = dsum;
        if (!ok) s_ok = 0;
    } else {
        // ---------------- 256 worker threads ----------------
        const float Dh = a.D ? a.D[h] : 0.f;
        const __nv_bfloat16* zp = static_cast<const __nv_bfloat16*>(a.z);
        Tout* yp = static_cast<Tout*>(a.y);
        bool ok = true;
        // z of this thread's outputs of chunk cc (row i = row, headdim 32*half..+31), loaded
        // ahead of the output step.
        uint4 z0 = make_uint4(0u, 0u, 0u, 0u), z1 = z0, z2 = z0, z3 = z0;
        auto load_z = [&](int cc) {
            const int64_t t_row = (int64_t)(t_base + cc * kQ + row);
            if (zp && t_row < L) {
                const uint4* zq = reinterpret_cast<const uint4*>(
                    zp + ((int64_t)b * L + t_row) * H * kHeadDim + (int64_t)h * kHeadDim + 32 * half);
                z0 = zq[0]; z1 = zq[1]; z2 = zq[2]; z3 = zq[3];
            }
        };
        // y of chunk cc = exp(cs_i) C S + M X + D x, times silu(z); e = exp(cs_i) of its row.
        auto output = [&](int cc, float e, bool with_state) {
            const int64_t t_row = (int64_t)(t_base + cc * kQ + row);
            const int64_t yoff = ((int64_t)b * L + t_row) * H * kHeadDim + (int64_t)h * kHeadDim + 32 * half;
            ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded(&bar_g2, (uint32_t)(cc & 1)));
            tc_fence_after_sync();
            if (ok) {
                const int in = kInTiles * (cc & 1);
                const uint32_t ccol = (cc & 1) ? kColCS1 : kColCS0;
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {  // 16 columns at a time
                    uint32_t mx[16], cs[16];
                    tmem_ld16_async(tmem + tlane + kColMX + 32 * half + 16 * hq, mx);
                    if (with_state) tmem_ld16_async(tmem + tlane + ccol + 32 * half + 16 * hq, cs);
                    tmem_wait_ld();
                    if (sh_store_y && t_row < L) {
                        float yd[16];
#pragma unroll
                        for (int qq = 0; qq < 2; ++qq) {
                            const int q = 2 * hq + qq;
                            float xv[8], zv[8];
                            unpack8(*reinterpret_cast<const uint4*>(tile(in + kInX) + sw128(row, 4 * half + q)), xv);
                            if (zp) unpack8(q == 0 ? z0 : q == 1 ? z1 : q == 2 ? z2 : z3, zv);
#pragma unroll
                            for (int i = 0; i < 8; i += 2) {  // pairs, packed
                                const int o = 8 * qq + i;
                                float2 y = __ffma2_rn(f2(Dh), make_float2(xv[i], xv[i + 1]),
                                                      make_float2(__uint_as_float(mx[o]), __uint_as_float(mx[o + 1])));
                                if (with_state)
                                    y = __ffma2_rn(f2(e), make_float2(__uint_as_float(cs[o]), __uint_as_float(cs[o + 1])), y);
                                if (zp) y = __fmul2_rn(y, silu2(make_float2(zv[i], zv[i + 1])));
                                yd[o] = y.x;
                                yd[o + 1] = y.y;
                            }
                        }
                        store16<Tout>(yp + yoff + 16 * hq, yd);
                    }
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&bar_y[cc & 1]);
        };

        float e_prev = 0.f;      // exp(cs_i) of the previous chunk (its output is pending)
        bool prev_state = false;
        if constexpr (kStateOnly) {
            for (int c = 0; c < nchunks; ++c) {
                const uint32_t par = (uint32_t)(c & 1);
                const int in = kInTiles * (c & 1);
                const bool had_state = c > 0 || init_state;
                ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded(&bar_sums, par));
                const float cs_last = s_cs[kQ - 1];
                ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded(&bar_tma[c & 1], (uint32_t)((c >> 1) & 1)));
                if (ok && half == 0) {  // w * X (hi / lo), row j = row
                    const float w = s_w[row];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        float v[8];
                        unpack8(*reinterpret_cast<const uint4*>(tile(in + kInX) + sw128(row, ch)), v);
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            const float2 p2 = __fmul2_rn(make_float2(v[e], v[e + 1]), f2(w));
                            v[e] = p2.x;
                            v[e + 1] = p2.y;
                        }
                        uint4 hi, lo;
                        split8(v, hi, lo);
                        *reinterpret_cast<uint4*>(tile(kTXH) + sw128(row, ch)) = hi;
                        *reinterpret_cast<uint4*>(tile(kTXL) + sw128(row, ch)) = lo;
                    }
                } else if (ok && had_state) {  // the carried state decays by exp(cs_last)
                    const float dec = ex2_approx(cs_last);
#pragma unroll 1
                    for (int part = 0; part < 2; ++part) {
                        float v[32];
                        tmem_ld32(tmem + tlane + kColS + 32 * part, v);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 d2 = __fmul2_rn(make_float2(v[i], v[i + 1]), f2(dec));
                            v[i] = d2.x;
                            v[i + 1] = d2.y;
                        }
                        tmem_st32(tmem + tlane + kColS + 32 * part, v);
                    }
                    tmem_wait_st();
                }
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&bar_x);
                mbar_arrive(&bar_free);  // this chunk's sums are no longer read
                // The state update has read w X and written S before either is touched again.
                ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded(&bar_g4, par));
                tc_fence_after_sync();
                if (!ok) break;
            }
        }
        for (int c = 0; c < (kStateOnly ? 0 : nchunks); ++c) {
            const int64_t t0 = (int64_t)(t_base + c * kQ);
            const uint32_t par = (uint32_t)(c & 1);
            const int in = kInTiles * (c & 1);
            const uint32_t gcol = (c & 1) ? kColG1 : kColG0;
            const bool had_state = c > 0 || init_state;
            ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded(&bar_sums, par));
            const float* const scs = s_cs;
            const float cs_last = scs[kQ - 1];

            // w * X (hi / lo) for the state update (warps 0-3, row j = row), and the decay of the
            // carried state by exp(cs_last) (warps 4-7, state row n = row).
            ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded(&bar_tma[c & 1], (uint32_t)((c >> 1) & 1)));
            if (ok && half == 0) {
                const float w = s_w[row];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float v[8];
                    unpack8(*reinterpret_cast<const uint4*>(tile(in + kInX) + sw128(row, ch)), v);
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const float2 p2 = __fmul2_rn(make_float2(v[e], v[e + 1]), f2(w));
                        v[e] = p2.x;
                        v[e + 1] = p2.y;
                    }
                    uint4 hi, lo;
                    split8(v, hi, lo);
                    *reinterpret_cast<uint4*>(tile(kTXH) + sw128(row, ch)) = hi;
                    *reinterpret_cast<uint4*>(tile(kTXL) + sw128(row, ch)) = lo;
                }
            } else if (ok && had_state) {
                const float dec = ex2_approx(cs_last);
#pragma unroll 1
                for (int part = 0; part < 2; ++part) {
                    float v[32];
                    tmem_ld32(tmem + tlane + kColS + 32 * part, v);
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float2 d2 = __fmul2_rn(make_float2(v[i], v[i + 1]), f2(dec));
                        v[i] = d2.x;
                        v[i + 1] = d2.y;
                    }
                    tmem_st32(tmem + tlane + kColS + 32 * part, v);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&bar_x);

            // The previous chunk's output, while this chunk's C B^T and C S run.
            if (c > 0) output(c - 1, e_prev, prev_state);

            // M = G * exp(cs_i - cs_j) * Delta_j (j <= i) as bf16 hi / lo pairs (row i = row,
            // columns 64*half..+63), written over the 16 columns of G they came from: columns
            // [16k, 16k+8) hold M hi of j = 16k..16k+15 (bf16 pairs), [16k+8, 16k+16) M lo.
            ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded(&bar_gg[c & 1], (uint32_t)((c >> 1) & 1)));
            tc_fence_after_sync();
            const float cs_i = scs[row];
            if (ok) {
                const bool live = t0 + row < L;
                const bool any = 64 * half <= quarter * 32 + 31;  // a column of this half is on or below the diagonal
#pragma unroll
                for (int piece = 0; piece < 4; ++piece) {  // 16 columns of G: j = 16k .. 16k+15
                    const int k = 4 * half + piece;
                    const uint32_t col = gcol + 16 * k;
                    const bool need = any && 16 * k <= quarter * 32 + 31;  // warp-uniform
                    uint32_t gp[16];
                    if (need) {
                        tmem_ld16_async(tmem + tlane + col, gp);
                        tmem_wait_ld();
                    }
                    uint32_t mh[8], ml[8];
                    // exp(cs_i - cs_j) Delta_j = 2^(cs_i - cs_16k) [2^(cs_16k - cs_j) Delta_j]: one
                    // exp per row and piece where the piece's decay span keeps both factors in
                    // range (rows decaying further make the first factor underflow to a
                    // negligible term); other pieces take the exp per element.
                    const bool factored = fabsf(s_span[k]) < kFactorSpan;  // warp-uniform
                    if (factored) {
                        const float rf = ex2_approx(cs_i - scs[16 * k]);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int j = 16 * k + 2 * e;
                            float2 m = make_float2(0.f, 0.f);
                            if (need && live && j <= row) {
                                const float2 gv = make_float2(__uint_as_float(gp[2 * e]), __uint_as_float(gp[2 * e + 1]));
                                const float2 cf = *reinterpret_cast<const float2*>(&s_cf[j]);
                                m = __fmul2_rn(__fmul2_rn(gv, cf), f2(rf));
                                if (j + 1 > row) m.y = 0.f;
                            }
                            split2(m, mh[e], ml[e]);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int j = 16 * k + 2 * e;
                            float2 m = make_float2(0.f, 0.f);
                            if (need && live && j <= row) {
                                const float2 cj = *reinterpret_cast<const float2*>(&scs[j]);
                                const float2 dj = *reinterpret_cast<const float2*>(&s_cf[j]);  // Delta here
                                const float2 dec = make_float2(ex2_approx(cs_i - cj.x),
                                                               j + 1 <= row ? ex2_approx(cs_i - cj.y) : 0.f);
                                const float2 gv = make_float2(__uint_as_float(gp[2 * e]), __uint_as_float(gp[2 * e + 1]));
                                m = __fmul2_rn(__fmul2_rn(gv, dec), dj);
                            }
                            split2(m, mh[e], ml[e]);
                        }
                    }
                    tmem_st8_async(tmem + tlane + col, mh);
                    tmem_st8_async(tmem + tlane + col + 8, ml);
                }
                tmem_wait_st();
            }
            tc_fence_before_sync();
            mbar_arrive(&bar_m);
            mbar_arrive(&bar_free);  // this chunk's sums are no longer read
            e_prev = ex2_approx(cs_i);
            prev_state = had_state;

            // The updated state -> hi / lo for the next chunk's C S (the wait on the state
            // update also covers this chunk's C S, issued before it).
            ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded(&bar_g4, par));
            tc_fence_after_sync();
            if (ok) {
                float sv[32];
                tmem_ld32(tmem + tlane + kColS + 32 * half, sv);
                put_state_split(sv);
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&bar_s);
            // z of this chunk's output (written in the next iteration; loaded here so that it
            // lands before the next proxy fence).
            load_z(c);
            if (!ok) break;
        }
        if (!kStateOnly && ok && nchunks > 0) output(nchunks - 1, e_prev, prev_state);

        float* const s_final = sh_final;
        if (ok && s_final) {  // S[n][p] -> final_state (p, n)
            float v[32];
            if (nchunks > 0 || init_state) {
                tmem_ld32(tmem + tlane + kColS + 32 * half, v);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.f;
            }
            float* dst = s_final + row;
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[(int64_t)(32 * half + i) * kSsdState] = v[i];
        }
        if (!ok) s_ok = 0;
    }
    // The whole chains, launched beside the local-end jobs: finish only after them, so that the
    // fold after this launch sees their end states.
    if (a.job_mode == 3) asm volatile("griddepcontrol.wait;" ::: "memory");
    tc_fence_before_sync();
    __syncthreads();
    if (tid == 0 && !s_ok) atomicOr(&g_ssd_status, 1u);
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// The initial states of segments 1..nseg-1 of the cut chains from the local-end pass: segment
// s+1 starts from 2^(dsum_s) times segment s's initial state plus segment s's end state from
// zero (the recurrence is linear in the state); segment 0's end state already started from the
// chain's initial state. One thread per (cut chain, state element), in segment order.
__global__ void ssd_fold_kernel(const SsdArgs a) {
    constexpr int64_t kStateElems = (int64_t)kHeadDim * kSsdState;
    constexpr int kBatch = 8;  // segments whose loads are issued together
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t tc = blockIdx.y;
    if (e >= kStateElems) return;
    const int64_t base = tc * (a.nseg - 1);
    const float* __restrict__ sloc = a.ws_sloc + base * kStateElems + e;
    const float* __restrict__ dsum = a.ws_dsum + base;
    float* __restrict__ sinit = a.ws_sinit + base * kStateElems + e;
    float v = 0.f;
    for (int s0 = 0; s0 < a.nseg - 1; s0 += kBatch) {
        float l[kBatch], d[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const bool in = s0 + i < a.nseg - 1;
            l[i] = in ? sloc[(int64_t)(s0 + i) * kStateElems] : 0.f;
            d[i] = in && s0 + i > 0 ? dsum[s0 + i] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            if (s0 + i >= a.nseg - 1) break;
            v = s0 + i == 0 ? l[i] : fmaf(exp2f(d[i]), v, l[i]);
            sinit[(int64_t)(s0 + i) * kStateElems] = v;
        }
    }
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
cudaError_t launch_ssd_typed(const SsdArgs& a0, void* workspace, size_t workspace_bytes, int sms,
                             cudaStream_t stream) {
    CUtensorMap mX{}, mB{}, mC{};
    if (a0.seqlen > 0) {
        cudaError_t e = make_ssd_map(&mX, a0.x, kHeadDim, a0.nheads, a0.seqlen, a0.batch);
        if (e == cudaSuccess) e = make_ssd_map(&mB, a0.B, kSsdState, a0.ngroups, a0.seqlen, a0.batch);
        if (e == cudaSuccess) e = make_ssd_map(&mC, a0.C, kSsdState, a0.ngroups, a0.seqlen, a0.batch);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaFuncSetAttribute(ssd_fwd_kernel<Tout, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSsdSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(ssd_fwd_kernel<Tout, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSsdSmemBytes);
    if (e != cudaSuccess) return e;
    SsdArgs a = a0;
    const SsdPlan plan = ssd_plan(a.batch, a.nheads, a.seqlen, sms);
    if (plan.n_cut == 0 || !workspace || workspace_bytes < plan.workspace_bytes) {
        a.job_mode = 0;  // one CTA per chain
        ssd_fwd_kernel<Tout, false><<<dim3((unsigned)a.nheads, (unsigned)a.batch), kSsdThreads,
                                      kSsdSmemBytes, stream>>>(a, mX, mB, mC);
        return cudaGetLastError();
    }
    // The balanced launch: the end states of the cut chains' segments 0..nseg-2 (state only),
    // with the whole chains starting on the SMs those leave free; their fold into initial
    // states; then every segment of the cut chains (the last wave).
    constexpr size_t kStateBytes = (size_t)kHeadDim * kSsdState * sizeof(float);
    const size_t nslots = (size_t)plan.n_cut * (size_t)(plan.nseg - 1);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.n_whole = plan.n_whole;
    a.nseg = plan.nseg;
    a.seg_chunks = plan.seg_chunks;
    a.ws_sloc = reinterpret_cast<float*>(ws);
    a.ws_sinit = reinterpret_cast<float*>(ws + nslots * kStateBytes);
    a.ws_dsum = reinterpret_cast<float*>(ws + 2 * nslots * kStateBytes);
    a.job_mode = 1;
    ssd_fwd_kernel<Tout, true><<<(unsigned)nslots, kSsdThreads, kSsdSmemBytes, stream>>>(a, mX, mB, mC);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    {
        SsdArgs w = a;
        w.job_mode = 3;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)plan.n_whole, 1, 1);
        cfg.blockDim = dim3(kSsdThreads, 1, 1);
        cfg.dynamicSmemBytes = kSsdSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, ssd_fwd_kernel<Tout, false>, w, mX, mB, mC);
        if (e != cudaSuccess) return e;
    }
    if (plan.nseg > 1) {
        ssd_fold_kernel<<<dim3((unsigned)((kHeadDim * kSsdState + 255) / 256), (unsigned)plan.n_cut),
                          256, 0, stream>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    a.job_mode = 2;
    const int64_t jobs = plan.n_cut * plan.nseg;
    ssd_fwd_kernel<Tout, false><<<(unsigned)jobs, kSsdThreads, kSsdSmemBytes, stream>>>(a, mX, mB, mC);
    return cudaGetLastError();
}

}  // namespace

// The chains (batch x heads, one CTA each, one CTA per SM) fill n full waves plus a remainder
// of r < sms chains that would run alone for a whole chain's time. Those r chains are cut into
// segments of seg_chunks chunks, as many as keep the r x nseg segments in one wave, at least two
// chunks each: the local-end pass and the segments' full pass then take about 2 seg_chunks
// chunk-times instead of nchunks. Not when the chains fit in one wave (nothing waits on a
// remainder) or the cut saves less than a third of that time.
SsdPlan ssd_plan(int64_t batch, int64_t nheads, int64_t seqlen, int sms) {
    SsdPlan p{batch * nheads, 0, 1, 0, 0};
    const int64_t chains = batch * nheads;
    const int64_t nchunks = (seqlen + kQ - 1) / kQ;
    if (sms <= 0 || chains <= sms || nchunks < 4) return p;
    const int64_t r = chains % sms;
    if (r == 0) return p;
    const int64_t nseg_target = std::min<int64_t>(sms / r, nchunks / 2);
    if (nseg_target < 2) return p;
    const int64_t seg_chunks = (nchunks + nseg_target - 1) / nseg_target;
    const int64_t nseg = (nchunks + seg_chunks - 1) / seg_chunks;
    if (nseg < 2 || 3 * (2 * seg_chunks) > 2 * nchunks) return p;
    constexpr size_t kStateBytes = (size_t)kHeadDim * kSsdState * sizeof(float);
    const size_t nslots = (size_t)r * (size_t)(nseg - 1);
    p.n_whole = chains - r;
    p.n_cut = r;
    p.nseg = (int)nseg;
    p.seg_chunks = (int)seg_chunks;
    p.workspace_bytes = 2 * nslots * kStateBytes + (nslots * sizeof(float) + 255) / 256 * 256;
    return p;
}

cudaError_t launch_ssd_fwd(const SsdArgs& a, bool out_bf16, void* workspace,
                           size_t workspace_bytes, int sms, cudaStream_t stream) {
    return out_bf16 ? launch_ssd_typed<__nv_bfloat16>(a, workspace, workspace_bytes, sms, stream)
                    : launch_ssd_typed<float>(a, workspace, workspace_bytes, sms, stream);
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
