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
// Layout as in the forward: a quad of 4 lanes per channel, lane g holding states 4g..4g+3; a CTA
// holds 32 channels of one batch. Lane g owns tokens 4g..4g+3 of each 16-token chunk (loads,
// per-token gradients); per-token values reach the quad by width-4 shuffles.
//
// dB and dC are sums over every channel of a batch and dA, dD, dbias over every batch: each
// CTA writes its partial sums (dB/dC per token after reducing its 32 channels, dA/dD/dbias per
// channel) to the workspace and a second kernel adds them in a fixed order, so the gradients
// are deterministic (no atomics).
#include "selscan_device.cuh"
#include "selscan_launch.h"

namespace selscan {

constexpr int kBChunk = 16;                 // tokens per chunk (and per checkpoint)
constexpr int kBWarps = 4;
constexpr int kBThreads = 32 * kBWarps;     // 128: 32 channels
constexpr int kBRows = 32;                  // channels per CTA
constexpr int kBSlots = 32;                 // dB[0..15], dC[0..15] per token

struct BwdSmem {
    float bc[kBChunk][32];                        // fp32 B | C of the chunk per token
    float4 H[kBWarps][kBChunk][32];               // recomputed states h_t of the chunk
    float X[kBWarps][8][kBSlots];                 // per-token transpose for the channel sums
    float P[kBWarps][kBChunk][kBSlots];           // warp sums of dB/dC per token
};

template <typename Tin>
__device__ __forceinline__ float ld1(const Tin* p) { return to_f32(*p); }

template <bool kPrecise>
__device__ __forceinline__ float sigmoid_f(float x) {
    return kPrecise ? 1.f / (1.f + expf(-x)) : rcp_approx(1.f + ex2_approx(-x * kLog2e));
}

template <typename Tin, typename Tg, bool kPrecise>
__global__ void __launch_bounds__(kBThreads) scan_bwd_kernel(const BwdArgs a) {
    __shared__ __align__(16) BwdSmem sm;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = lane >> 2, g = lane & 3;
    const int64_t b = blockIdx.y;
    const int64_t d_raw = (int64_t)blockIdx.x * kBRows + warp * 8 + quad;
    const bool active = d_raw < a.dim;
    const int64_t d = active ? d_raw : 0;
    const int64_t row = b * a.dim + d;
    const int64_t L = a.seqlen;
    const int nchunks = (int)((L + kBChunk - 1) / kBChunk);

    // Per-lane constants: A (natural units) and A*log2(e) for the SFU.
    const float4 An = *reinterpret_cast<const float4*>(a.A + d * kN + 4 * g);
    const float Av[4] = {An.x, An.y, An.z, An.w};
    float A2[4];
#pragma unroll
    for (int n = 0; n < 4; ++n) A2[n] = Av[n] * kLog2e;
    const float bias = a.delta_bias ? a.delta_bias[d] : 0.f;
    const float Dd = a.D ? a.D[d] : 0.f;

    const Tin* u_row = static_cast<const Tin*>(a.u) + row * L;
    const Tin* d_row = static_cast<const Tin*>(a.delta) + row * L;
    const Tin* z_row = a.z ? static_cast<const Tin*>(a.z) + row * L : nullptr;
    const Tg* o_row = static_cast<const Tg*>(a.dout) + row * L;
    const Tin* Bb = static_cast<const Tin*>(a.B) + b * kN * L;
    const Tin* Cb = static_cast<const Tin*>(a.C) + b * kN * L;
    float* ckpt = a.ws_ckpt + (row * nchunks) * kN + 4 * g;

    // Decay factor of state n over a step with Delta: exp(Delta*A).
    auto decay = [&](float dt, int n) -> float {
        return kPrecise ? expf(dt * Av[n]) : ex2_approx(dt * A2[n]);
    };
    auto delta_of = [&](float x) -> float {
        if (!a.softplus) return x;
        return kPrecise ? softplus_f<true>(x) : softplus2(make_float2(x, x)).x;
    };
    // Stage B (and C) of chunk c as fp32 rows per token: thread -> (token, 4 states of B|C).
    auto stage_bc = [&](int c, bool withC) {
        const int64_t t0 = (int64_t)c * kBChunk;
        for (int item = tid; item < kBChunk * 8; item += kBThreads) {
            const int tt = item % kBChunk, ch = item / kBChunk;  // ch 0..3: B quads, 4..7: C quads
            if (ch >= 4 && !withC) continue;
            const Tin* src = ch >= 4 ? Cb : Bb;
            const int q = ch & 3;
            const int64_t t = t0 + tt;
            const bool ok = t < L;
            float4 v;
            v.x = ok ? ld1(src + (4 * q + 0) * L + t) : 0.f;
            v.y = ok ? ld1(src + (4 * q + 1) * L + t) : 0.f;
            v.z = ok ? ld1(src + (4 * q + 2) * L + t) : 0.f;
            v.w = ok ? ld1(src + (4 * q + 3) * L + t) : 0.f;
            *reinterpret_cast<float4*>(&sm.bc[tt][4 * ch]) = v;
        }
    };

    // ---- checkpoint pass: the forward state before every chunk ----
    float h[4];
    {
        float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.initial_state) s0 = *reinterpret_cast<const float4*>(a.initial_state + row * kN + 4 * g);
        h[0] = s0.x; h[1] = s0.y; h[2] = s0.z; h[3] = s0.w;
    }
    for (int c = 0; c < nchunks; ++c) {
        if (active) *reinterpret_cast<float4*>(ckpt + (int64_t)c * kN) = make_float4(h[0], h[1], h[2], h[3]);
        __syncthreads();
        stage_bc(c, false);
        const int64_t tl = (int64_t)c * kBChunk + 4 * g;
        float dl[4], kl[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool ok = active && tl + i < L;
            const float dt = ok ? delta_of(ld1(d_row + tl + i) + bias) : 0.f;
            dl[i] = dt;
            kl[i] = ok ? dt * ld1(u_row + tl + i) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int t = 0; t < kBChunk; ++t) {
            const float dt = __shfl_sync(0xffffffffu, dl[t & 3], t >> 2, 4);
            const float k = __shfl_sync(0xffffffffu, kl[t & 3], t >> 2, 4);
            const float4 Bv = *reinterpret_cast<const float4*>(&sm.bc[t][4 * g]);
            const float Bs[4] = {Bv.x, Bv.y, Bv.z, Bv.w};
#pragma unroll
            for (int n = 0; n < 4; ++n) h[n] = fmaf(decay(dt, n), h[n], k * Bs[n]);
        }
    }

    // ---- reverse pass ----
    float gad[4];  // adjoint of the state
    {
        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.dfinal_state && active)
            f = *reinterpret_cast<const float4*>(a.dfinal_state + row * kN + 4 * g);
        gad[0] = f.x; gad[1] = f.y; gad[2] = f.z; gad[3] = f.w;
    }
    float dA_acc[4] = {0.f, 0.f, 0.f, 0.f};
    float dD_acc = 0.f, db_acc = 0.f;
    Tg* du_row = static_cast<Tg*>(a.du) + row * L;
    Tg* dd_row = static_cast<Tg*>(a.ddelta) + row * L;
    Tg* dz_row = a.dz ? static_cast<Tg*>(a.dz) + row * L : nullptr;
    float* part = a.ws_part + ((int64_t)blockIdx.x * a.batch + b) * kBSlots * L;  // [slot][t]

    for (int c = nchunks - 1; c >= 0; --c) {
        __syncthreads();  // the previous chunk's readers of bc / P are done
        stage_bc(c, true);
        const int64_t t0 = (int64_t)c * kBChunk;
        const int64_t tl = t0 + 4 * g;
        // Owned tokens: inputs and per-token values.
        float dl[4], kl[4], ul[4], xl[4], zl[4], ol[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool ok = active && tl + i < L;
            xl[i] = ok ? ld1(d_row + tl + i) + bias : 0.f;
            ul[i] = ok ? ld1(u_row + tl + i) : 0.f;
            zl[i] = ok && z_row ? ld1(z_row + tl + i) : 0.f;
            ol[i] = ok ? to_f32(o_row[tl + i]) : 0.f;
            dl[i] = ok ? delta_of(xl[i]) : 0.f;
            kl[i] = dl[i] * ul[i];
        }
        float hk[4];
        {
            // Rows past dim never wrote a checkpoint: they run on zeros.
            float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (active) s0 = *reinterpret_cast<const float4*>(ckpt + (int64_t)c * kN);
            hk[0] = s0.x; hk[1] = s0.y; hk[2] = s0.z; hk[3] = s0.w;
        }
        __syncthreads();
        // Recompute the chunk's states (kept in shared memory) and the readouts s_t.
        float sl[4] = {0.f, 0.f, 0.f, 0.f};
        {
            float hh[4] = {hk[0], hk[1], hk[2], hk[3]};
#pragma unroll
            for (int t = 0; t < kBChunk; ++t) {
                const float dt = __shfl_sync(0xffffffffu, dl[t & 3], t >> 2, 4);
                const float k = __shfl_sync(0xffffffffu, kl[t & 3], t >> 2, 4);
                const float4 Bv = *reinterpret_cast<const float4*>(&sm.bc[t][4 * g]);
                const float4 Cv = *reinterpret_cast<const float4*>(&sm.bc[t][16 + 4 * g]);
                const float Bs[4] = {Bv.x, Bv.y, Bv.z, Bv.w}, Cs[4] = {Cv.x, Cv.y, Cv.z, Cv.w};
                float y = 0.f;
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    hh[n] = fmaf(decay(dt, n), hh[n], k * Bs[n]);
                    y = fmaf(Cs[n], hh[n], y);
                }
                sm.H[warp][t][lane] = make_float4(hh[0], hh[1], hh[2], hh[3]);
                y += __shfl_xor_sync(0xffffffffu, y, 1);
                y += __shfl_xor_sync(0xffffffffu, y, 2);
                if (g == (t >> 2)) sl[t & 3] = y;  // the owner keeps s_t - D u_t
            }
        }
        // Owner: ds and dz of its tokens.
        float dsl[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float s = sl[i] + Dd * ul[i];
            if (z_row) {
                const float sig = sigmoid_f<kPrecise>(zl[i]);
                dsl[i] = ol[i] * zl[i] * sig;
                const float dzv = ol[i] * s * sig * (1.f + zl[i] * (1.f - sig));
                if (active && tl + i < L) dz_row[tl + i] = from_f32<Tg>(dzv);
            } else {
                dsl[i] = ol[i];
            }
        }
        __syncwarp();
        // Adjoint recurrence, last token of the chunk first.
        float dkl[4], dal[4];  // owner: dk_t and the Abar part of dDelta_t
#pragma unroll
        for (int t = kBChunk - 1; t >= 0; --t) {
            const float dt = __shfl_sync(0xffffffffu, dl[t & 3], t >> 2, 4);
            const float k = __shfl_sync(0xffffffffu, kl[t & 3], t >> 2, 4);
            const float ds = __shfl_sync(0xffffffffu, dsl[t & 3], t >> 2, 4);
            const float4 Bv = *reinterpret_cast<const float4*>(&sm.bc[t][4 * g]);
            const float4 Cv = *reinterpret_cast<const float4*>(&sm.bc[t][16 + 4 * g]);
            const float Bs[4] = {Bv.x, Bv.y, Bv.z, Bv.w}, Cs[4] = {Cv.x, Cv.y, Cv.z, Cv.w};
            const float4 ht = sm.H[warp][t][lane];
            float4 hp;
            if (t > 0) hp = sm.H[warp][t - 1][lane];
            else hp = make_float4(hk[0], hk[1], hk[2], hk[3]);
            const float hts[4] = {ht.x, ht.y, ht.z, ht.w}, hps[4] = {hp.x, hp.y, hp.z, hp.w};
            float dk = 0.f, da = 0.f, cdb[4], cdc[4];
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                gad[n] = fmaf(ds, Cs[n], gad[n]);
                cdc[n] = ds * hts[n];
                cdb[n] = gad[n] * k;
                dk = fmaf(gad[n], Bs[n], dk);
                const float ab = decay(dt, n);
                const float w = gad[n] * hps[n] * ab;  // dAbar * Abar
                da = fmaf(w, Av[n], da);
                dA_acc[n] = fmaf(w, dt, dA_acc[n]);
                gad[n] *= ab;
            }
            dk += __shfl_xor_sync(0xffffffffu, dk, 1);
            dk += __shfl_xor_sync(0xffffffffu, dk, 2);
            da += __shfl_xor_sync(0xffffffffu, da, 1);
            da += __shfl_xor_sync(0xffffffffu, da, 2);
            if (g == (t >> 2)) { dkl[t & 3] = dk; dal[t & 3] = da; }
            // Channel sums of this warp's 8 rows for dB_t, dC_t: transpose through shared memory.
            *reinterpret_cast<float4*>(&sm.X[warp][quad][4 * g]) = make_float4(cdb[0], cdb[1], cdb[2], cdb[3]);
            *reinterpret_cast<float4*>(&sm.X[warp][quad][16 + 4 * g]) = make_float4(cdc[0], cdc[1], cdc[2], cdc[3]);
            __syncwarp();
            float s = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q) s += sm.X[warp][q][lane];
            sm.P[warp][t][lane] = s;
            __syncwarp();
        }
        // Owner: per-token gradients of its tokens.
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool ok = active && tl + i < L;
            const float du = fmaf(dkl[i], dl[i], dsl[i] * Dd);
            const float dDelta = fmaf(dkl[i], ul[i], dal[i]);
            const float ddv = a.softplus ? dDelta * sigmoid_f<kPrecise>(xl[i]) : dDelta;
            if (ok) {
                du_row[tl + i] = from_f32<Tg>(du);
                dd_row[tl + i] = from_f32<Tg>(ddv);
                dD_acc = fmaf(dsl[i], ul[i], dD_acc);
                db_acc += ddv;
            }
        }
        __syncthreads();
        // CTA sums of dB_t / dC_t over its 4 warps -> partials [slot][t] of this CTA.
        for (int item = tid; item < kBSlots * kBChunk; item += kBThreads) {
            const int slot = item / kBChunk, tt = item % kBChunk;
            const int64_t t = t0 + tt;
            if (t < L) {
                float s = 0.f;
#pragma unroll
                for (int w = 0; w < kBWarps; ++w) s += sm.P[w][tt][slot];
                part[(int64_t)slot * L + t] = s;
            }
        }
    }

    // ---- per-channel partials (summed over batches by the reduction kernel) ----
    if (active) {
        if (a.dinitial_state)
            *reinterpret_cast<float4*>(a.dinitial_state + row * kN + 4 * g) =
                make_float4(gad[0], gad[1], gad[2], gad[3]);
        *reinterpret_cast<float4*>(a.ws_dA + row * kN + 4 * g) =
            make_float4(dA_acc[0], dA_acc[1], dA_acc[2], dA_acc[3]);
    }
    dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, 1);
    dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, 2);
    db_acc += __shfl_xor_sync(0xffffffffu, db_acc, 1);
    db_acc += __shfl_xor_sync(0xffffffffu, db_acc, 2);
    if (active && g == 0) {
        a.ws_dD[row] = dD_acc;
        a.ws_db[row] = db_acc;
    }
}

// Adds the per-CTA / per-row partials in a fixed order: dB, dC over channel blocks; dA, dD,
// dbias over batches.
__global__ void scan_bwd_reduce_kernel(const BwdArgs a, int64_t nblk) {
    const int64_t L = a.seqlen;
    const int64_t nbc = a.batch * kBSlots * L;            // dB and dC entries
    const int64_t nda = a.dim * kN;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nbc + nda + 2 * a.dim;
         i += stride) {
        if (i < nbc) {
            const int64_t t = i % L, slot = (i / L) % kBSlots, b = i / (L * kBSlots);
            float s = 0.f;
            for (int64_t k = 0; k < nblk; ++k) s += a.ws_part[((k * a.batch + b) * kBSlots + slot) * L + t];
            float* dst = slot < kN ? a.dB : a.dC;
            dst[(b * kN + (slot % kN)) * L + t] = s;
        } else if (i < nbc + nda) {
            const int64_t j = i - nbc;  // d*16 + n
            float s = 0.f;
            for (int64_t b = 0; b < a.batch; ++b) s += a.ws_dA[b * nda + j];
            a.dA[j] = s;
        } else {
            const int64_t j = i - nbc - nda;
            const int64_t dd = j % a.dim;
            const bool isD = j < a.dim;
            float s = 0.f;
            for (int64_t b = 0; b < a.batch; ++b) s += (isD ? a.ws_dD : a.ws_db)[b * a.dim + dd];
            if (isD && a.dD) a.dD[dd] = s;
            if (!isD && a.ddelta_bias) a.ddelta_bias[dd] = s;
        }
    }
}

template <typename Tin, typename Tg, bool kPrecise>
static cudaError_t launch_bwd_typed(const BwdArgs& a, cudaStream_t stream) {
    const unsigned gx = (unsigned)((a.dim + kBRows - 1) / kBRows);
    scan_bwd_kernel<Tin, Tg, kPrecise><<<dim3(gx, (unsigned)a.batch), kBThreads, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
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

size_t scan_bwd_workspace_floats(int64_t batch, int64_t dim, int64_t seqlen, int64_t* off_part,
                                 int64_t* off_dA, int64_t* off_dD, int64_t* off_db) {
    const int64_t rows = batch * dim;
    const int64_t nchunks = (seqlen + kBChunk - 1) / kBChunk;
    const int64_t nblk = (dim + kBRows - 1) / kBRows;
    auto up = [](int64_t x) { return (x + 63) / 64 * 64; };  // 256-byte alignment
    const int64_t ckpt = up(rows * nchunks * kN);
    const int64_t part = up(nblk * batch * kBSlots * seqlen);
    const int64_t dA = up(rows * kN);
    const int64_t dD = up(rows), db = up(rows);
    if (off_part) *off_part = ckpt;
    if (off_dA) *off_dA = ckpt + part;
    if (off_dD) *off_dD = ckpt + part + dA;
    if (off_db) *off_db = ckpt + part + dA + dD;
    return (size_t)(ckpt + part + dA + dD + db);
}

}  // namespace selscan
