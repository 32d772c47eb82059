// ssm_scan_fwd_no_alloc: the selective scan for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory: code embedded in a host program whose
// framework owns every device allocation and exposes no allocator hook, or a latency-critical
// loop that must not call cudaMalloc (which can synchronise the device). For them this entry
// point takes the time-split scratch of the scan from a fixed array that the library itself
// declares in device memory, instead of from a caller-provided workspace. It allocates
// nothing and calls no allocating routine; every computation is the one of ssm_scan_fwd.
//
// The array is a file-scope static __device__ object: every GPU that loads the library keeps
// kNoAllocScratchBytes of it until the process exits. Host code cannot use its name as an
// address (on the host the name is only a stand-in), so its device address is looked up once
// per device with cudaGetSymbolAddress, with that device current, on the first call made on
// that device.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/selscan.h"
#include "selscan_launch.h"

#define SELSCAN_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kNoAllocScratchBytes = SELSCAN_NO_ALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Shared by every call on a device; holds the per-segment end states and Delta sums.
static __device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up on first use.
selscan_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return SELSCAN_ERR_CUDA; }
    if (dev < 0 || dev >= kMaxDevices) return SELSCAN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return SELSCAN_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SELSCAN_OK;
}

}  // namespace

SELSCAN_EXPORT selscan_status ssm_scan_fwd_no_alloc(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus, void* out,
    float* final_state, int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    selscan_dtype in_dtype, selscan_dtype out_dtype, const float* initial_state,
    selscan_stream_t stream) {
    // The scratch this shape cannot do without on the current device; 0 also for invalid
    // shapes, which ssm_scan_fwd then reports with its own status. A shape whose time split
    // only balances the GPU takes it when it fits the array and runs unsplit otherwise.
    if (dstate == 16 && selscan::scan_required_workspace(batch, dim, seqlen) > kNoAllocScratchBytes)
        return SELSCAN_ERR_SCRATCH_LIMIT;
    const size_t want = ssm_scan_workspace_size(batch, dim, dstate, seqlen);
    void* scratch = nullptr;
    if (want > 0) {
        // The array's address is the current device's: a stream of another device would run
        // the kernels there with a pointer into this device's memory.
        if (stream) {
            int cur = 0, sdev = 0;
            if (cudaGetDevice(&cur) != cudaSuccess ||
                cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) {
                cudaGetLastError();
                return SELSCAN_ERR_CUDA;
            }
            if (sdev != cur) return SELSCAN_ERR_INVALID_ARG;
        }
        const selscan_status s = scratch_address(&scratch);
        if (s != SELSCAN_OK) return s;
    }
    // No part of the scratch needs to start at zero: the first kernel of a call writes every
    // entry that the second kernel reads.
    return ssm_scan_fwd(u, delta, A, B, C, D, z, delta_bias, delta_softplus, out, final_state,
                        batch, dim, dstate, seqlen, in_dtype, out_dtype, initial_state,
                        want > 0 ? scratch : nullptr, want > 0 ? kNoAllocScratchBytes : 0,
                        stream);
}
