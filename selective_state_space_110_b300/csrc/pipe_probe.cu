// Pipe-rate microbenchmarks behind the scan's arithmetic ceiling (libselscan_probe.so).
//
// The selective scan is bounded by arithmetic, not by HBM, on a B300: every (token, state)
// pair needs one exp2 on the SFU and four fp32 lane-operations on the FMA pipe, and every
// value a lane needs from another lane (shared memory, shuffles) passes the L1 data pipe. The
// ceiling the benchmark reports rests on three rates, measured here rather than assumed:
//   - ex2.approx results per clock per SM (SFU);
//   - fp32 FMA lane-operations per clock per SM, scalar and as packed f32x2 instructions;
//   - shared-memory words delivered to lanes per clock per SM (32-bit and 128-bit loads) and
//     shuffles per clock per SM.
// (lg2 and rcp, used by softplus and silu, are measured too.)
//
// Method: one CTA of 1,024 threads per SM (enough warps to cover every latency), each thread
// running 16 independent dependency chains (or 8 independent loads) for a fixed number of
// iterations; thread 0 reads clock64 before and after, around a __syncthreads on each side.
// Rate per SM = operations of the CTA / elapsed SM clocks, independent of the clock frequency.
// Every chain stays bounded (fixed points below), every shared-memory index is masked into the
// array, and every loop has a fixed trip count.
#include <cuda_runtime.h>
#include <stdint.h>

#define PROBE_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr int kThreads = 1024;
constexpr int kChains = 16;

__device__ __forceinline__ float ex2a(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2a(float x) {
    float y;
    asm volatile("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcpa(float x) {
    float y;
    asm volatile("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Elapsed clocks of the CTA's loop, written by thread 0; `sink` keeps the results alive.
struct Out {
    long long* cycles;  // one per CTA
    float* sink;        // one per thread of the grid
};

template <int kOp>
__global__ void __launch_bounds__(kThreads, 1) arith_kernel(Out o, int iters) {
    float v[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) v[i] = 0.01f * (threadIdx.x & 7) + 0.1f * i;
    __syncthreads();
    long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) {
            if (kOp == 0) v[i] = ex2a(v[i]) - 1.5f;          // fixed point near -0.93
            if (kOp == 1) v[i] = fmaf(v[i], 0.999f, 0.001f);  // fixed point 1
            if (kOp == 2) v[i] = lg2a(v[i] + 3.f);            // stays in [1.5, 2.4]
            if (kOp == 3) v[i] = rcpa(v[i] + 1.f);            // stays in [0.5, 1]
        }
    }
    __syncthreads();
    long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += v[i];
    o.sink[blockIdx.x * kThreads + threadIdx.x] = s;
    if (threadIdx.x == 0) o.cycles[blockIdx.x] = t1 - t0;
}

// Packed f32x2 FMA: 8 chains of pairs = 16 lanes of work per thread per iteration.
__global__ void __launch_bounds__(kThreads, 1) ffma2_kernel(Out o, int iters) {
    float2 v[kChains / 2];
#pragma unroll
    for (int i = 0; i < kChains / 2; ++i) v[i] = make_float2(0.1f * i, 0.05f * i);
    const float2 a = make_float2(0.999f, 0.998f), b = make_float2(0.001f, 0.002f);
    __syncthreads();
    long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains / 2; ++i) v[i] = __ffma2_rn(v[i], a, b);
    }
    __syncthreads();
    long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains / 2; ++i) s += v[i].x + v[i].y;
    o.sink[blockIdx.x * kThreads + threadIdx.x] = s;
    if (threadIdx.x == 0) o.cycles[blockIdx.x] = t1 - t0;
}

// Shared-memory loads (kVec = 1: 32-bit, 4: 128-bit) and shuffles (kVec = 0). Each thread
// keeps 8 independent loads in flight per iteration from conflict-free addresses (lane-linear
// within a warp); the index moves each iteration and is masked into the 16 KiB array.
template <int kVec>
__global__ void __launch_bounds__(kThreads, 1) l1_kernel(Out o, int iters) {
    __shared__ __align__(16) float smem[4096];
    for (int i = threadIdx.x; i < 4096; i += kThreads) smem[i] = 0.001f * (i & 63);
    const int lane = threadIdx.x & 31;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    __syncthreads();
    long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (kVec == 0) {
                acc[j] = __shfl_xor_sync(0xffffffffu, acc[j], (j & 3) + 1) + 1.f;
            } else if (kVec == 1) {
                const int idx = ((it * 8 + j) * 32 + lane) & 4095;
                acc[j] += smem[idx];
            } else {
                const int idx = (((it * 8 + j) * 32 + lane) * 4) & 4095;
                const float4 q = *reinterpret_cast<const float4*>(&smem[idx]);
                acc[j] += (q.x + q.y) + (q.z + q.w);
            }
        }
    }
    __syncthreads();
    long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += acc[j];
    o.sink[blockIdx.x * kThreads + threadIdx.x] = s;
    if (threadIdx.x == 0) o.cycles[blockIdx.x] = t1 - t0;
}

}  // namespace

// Runs probe `which` on `ctas` CTAs of 1,024 threads for `iters` iterations and returns, per
// SM-resident CTA, the operations per clock (averaged over CTAs), or a negative value on a CUDA
// error. cycles: device buffer of `ctas` int64; sink: device buffer of ctas*1024 floats.
//   which 0 ex2, 1 fp32 FMA (lane-ops), 2 lg2, 3 rcp, 4 f32x2 FMA (lane-ops),
//         5 shuffles (thread-shuffles), 6 32-bit shared loads (words), 7 128-bit shared loads
//         (words).
PROBE_EXPORT double selscan_probe_rate(int which, int ctas, int iters, long long* cycles,
                                       float* sink) {
    if (ctas <= 0 || iters <= 0 || iters > (1 << 20) || !cycles || !sink) return -1.0;
    Out o{cycles, sink};
    double per_thread_per_iter = 0;
    switch (which) {
        case 0: arith_kernel<0><<<ctas, kThreads>>>(o, iters); per_thread_per_iter = kChains; break;
        case 1: arith_kernel<1><<<ctas, kThreads>>>(o, iters); per_thread_per_iter = kChains; break;
        case 2: arith_kernel<2><<<ctas, kThreads>>>(o, iters); per_thread_per_iter = kChains; break;
        case 3: arith_kernel<3><<<ctas, kThreads>>>(o, iters); per_thread_per_iter = kChains; break;
        case 4: ffma2_kernel<<<ctas, kThreads>>>(o, iters); per_thread_per_iter = kChains; break;
        case 5: l1_kernel<0><<<ctas, kThreads>>>(o, iters); per_thread_per_iter = 8; break;
        case 6: l1_kernel<1><<<ctas, kThreads>>>(o, iters); per_thread_per_iter = 8; break;
        case 7: l1_kernel<4><<<ctas, kThreads>>>(o, iters); per_thread_per_iter = 32; break;
        default: return -1.0;
    }
    if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return -2.0;
    }
    long long host[1024];
    const int n = ctas < 1024 ? ctas : 1024;
    if (cudaMemcpy(host, cycles, sizeof(long long) * n, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return -3.0;
    }
    double sum = 0;
    for (int i = 0; i < n; ++i) sum += (double)host[i];
    const double mean_cycles = sum / n;
    return per_thread_per_iter * kThreads * (double)iters / mean_cycles;
}
