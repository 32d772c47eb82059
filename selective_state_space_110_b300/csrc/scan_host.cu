// ssm_scan_fwd_host: the selective scan on host buffers, copies overlapped with the scan.
//
// A caller whose activations live in host memory pays for the host-device copies, which on a
// PCIe link take longer than the scan itself. This entry point cuts the batch into slices of one
// sequence and pipelines them over three streams: the upload of slice i+1 and the download of
// slice i-1 run while slice i is scanned. Every computation is the one of ssm_scan_fwd (it is
// called once per slice on the caller's stream); the copies are plain cudaMemcpyAsync calls on
// two streams the library creates once per device, ordered by events.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/selscan.h"

#define SELSCAN_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr int kMaxDevices = 64;
constexpr int kSlots = 2;  // device buffers for two slices in flight
constexpr size_t kAlign = 256;

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
size_t esize(selscan_dtype t) { return t == SELSCAN_BF16 ? 2 : 4; }

// Copy-in and copy-out streams and the events that order the pipeline, per device.
struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t entry = nullptr, in_done[kSlots] = {}, scan_done[kSlots] = {}, out_done[kSlots] = {};
};
std::mutex g_pipe_mutex;
HostPipe g_pipe[kMaxDevices];
bool g_pipe_ready[kMaxDevices] = {};

selscan_status get_pipe(HostPipe** p) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return SELSCAN_ERR_CUDA; }
    if (dev < 0 || dev >= kMaxDevices) return SELSCAN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    HostPipe& h = g_pipe[dev];
    if (!g_pipe_ready[dev]) {
        bool ok = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.entry, cudaEventDisableTiming) == cudaSuccess;
        for (int s = 0; ok && s < kSlots; ++s)
            ok = cudaEventCreateWithFlags(&h.in_done[s], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h.scan_done[s], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h.out_done[s], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) { cudaGetLastError(); return SELSCAN_ERR_CUDA; }
        g_pipe_ready[dev] = true;
    }
    *p = &h;
    return SELSCAN_OK;
}

// Byte offsets of one slot's buffers and of the per-channel parameters in the workspace.
struct HostLayout {
    size_t u, delta, z, B, C, out, fin, init, scan_ws, slot_bytes;
    size_t A, D, bias, total;
};
HostLayout host_layout(int64_t dim, int64_t seqlen, size_t ein, size_t eout, size_t scan_ws) {
    HostLayout l{};
    const size_t act = (size_t)dim * (size_t)seqlen;
    size_t o = 0;
    l.u = o; o += up(act * ein);
    l.delta = o; o += up(act * ein);
    l.z = o; o += up(act * ein);
    l.B = o; o += up((size_t)16 * seqlen * ein);
    l.C = o; o += up((size_t)16 * seqlen * ein);
    l.out = o; o += up(act * eout);
    l.fin = o; o += up((size_t)dim * 16 * 4);
    l.init = o; o += up((size_t)dim * 16 * 4);
    l.scan_ws = o; o += up(scan_ws);
    l.slot_bytes = o;
    o *= kSlots;
    l.A = o; o += up((size_t)dim * 16 * 4);
    l.D = o; o += up((size_t)dim * 4);
    l.bias = o; o += up((size_t)dim * 4);
    l.total = o;
    return l;
}

}  // namespace

SELSCAN_EXPORT size_t ssm_scan_fwd_host_workspace_size(int64_t batch, int64_t dim, int64_t dstate,
                                                       int64_t seqlen, selscan_dtype in_dtype,
                                                       selscan_dtype out_dtype) {
    if (batch < 1 || dim < 1 || seqlen < 0 || dstate != 16) return 0;
    if ((in_dtype != SELSCAN_F32 && in_dtype != SELSCAN_BF16) ||
        (out_dtype != SELSCAN_F32 && out_dtype != SELSCAN_BF16))
        return 0;
    const size_t scan_ws = ssm_scan_workspace_size(1, dim, dstate, seqlen);
    return host_layout(dim, seqlen, esize(in_dtype), esize(out_dtype), scan_ws).total;
}

SELSCAN_EXPORT selscan_status ssm_scan_fwd_host(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus, void* out,
    float* final_state, int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    selscan_dtype in_dtype, selscan_dtype out_dtype, const float* initial_state,
    void* workspace, size_t workspace_bytes, selscan_stream_t stream) {
    if (dstate != 16) return SELSCAN_ERR_UNSUPPORTED;
    if ((in_dtype != SELSCAN_F32 && in_dtype != SELSCAN_BF16) ||
        (out_dtype != SELSCAN_F32 && out_dtype != SELSCAN_BF16))
        return SELSCAN_ERR_UNSUPPORTED;
    if (batch < 1 || batch > 65535 || dim < 1 || seqlen < 0) return SELSCAN_ERR_INVALID_ARG;
    const bool has_tokens = seqlen > 0;
    if (!A || (has_tokens && (!u || !delta || !B || !C || !out))) return SELSCAN_ERR_INVALID_ARG;
    const size_t need = ssm_scan_fwd_host_workspace_size(batch, dim, dstate, seqlen, in_dtype, out_dtype);
    if (!workspace || workspace_bytes < need) return SELSCAN_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return SELSCAN_ERR_ALIGNMENT;

    HostPipe* pipe = nullptr;
    selscan_status st = get_pipe(&pipe);
    if (st != SELSCAN_OK) return st;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const size_t ein = esize(in_dtype), eout = esize(out_dtype);
    const size_t scan_ws = ssm_scan_workspace_size(1, dim, dstate, seqlen);
    const HostLayout l = host_layout(dim, seqlen, ein, eout, scan_ws);
    char* ws = static_cast<char*>(workspace);
    const size_t act = (size_t)dim * (size_t)seqlen;
    const size_t bc = (size_t)16 * (size_t)seqlen;
    const size_t stb = (size_t)dim * 16 * 4;
    auto fail = [] { cudaGetLastError(); return SELSCAN_ERR_CUDA; };
    auto h2d = [&](size_t off, const void* src, size_t bytes) {
        return bytes == 0 || cudaMemcpyAsync(ws + off, src, bytes, cudaMemcpyHostToDevice, pipe->in) == cudaSuccess;
    };
    auto d2h = [&](void* dst, size_t off, size_t bytes) {
        return bytes == 0 || cudaMemcpyAsync(dst, ws + off, bytes, cudaMemcpyDeviceToHost, pipe->out) == cudaSuccess;
    };

    // Work already queued on the caller's stream (which may use the workspace) comes first.
    if (cudaEventRecord(pipe->entry, cs) != cudaSuccess ||
        cudaStreamWaitEvent(pipe->in, pipe->entry, 0) != cudaSuccess ||
        cudaStreamWaitEvent(pipe->out, pipe->entry, 0) != cudaSuccess)
        return fail();
    if (!h2d(l.A, A, (size_t)dim * 16 * 4) || (D && !h2d(l.D, D, (size_t)dim * 4)) ||
        (delta_bias && !h2d(l.bias, delta_bias, (size_t)dim * 4)))
        return fail();

    for (int64_t i = 0; i < batch; ++i) {
        const int s = (int)(i % kSlots);
        const size_t base = (size_t)s * l.slot_bytes;
        // The slot is free once slice i-2 has been copied out (which followed its scan).
        if (i >= kSlots && cudaStreamWaitEvent(pipe->in, pipe->out_done[s], 0) != cudaSuccess) return fail();
        const char* uh = static_cast<const char*>(u) + (size_t)i * act * ein;
        const char* dh = static_cast<const char*>(delta) + (size_t)i * act * ein;
        const char* bh = static_cast<const char*>(B) + (size_t)i * bc * ein;
        const char* ch = static_cast<const char*>(C) + (size_t)i * bc * ein;
        bool ok = !has_tokens || (h2d(base + l.u, uh, act * ein) && h2d(base + l.delta, dh, act * ein) &&
                                  h2d(base + l.B, bh, bc * ein) && h2d(base + l.C, ch, bc * ein));
        if (ok && z && has_tokens) ok = h2d(base + l.z, static_cast<const char*>(z) + (size_t)i * act * ein, act * ein);
        if (ok && initial_state) ok = h2d(base + l.init, initial_state + (size_t)i * dim * 16, stb);
        if (!ok || cudaEventRecord(pipe->in_done[s], pipe->in) != cudaSuccess) return fail();

        if (cudaStreamWaitEvent(cs, pipe->in_done[s], 0) != cudaSuccess) return fail();
        st = ssm_scan_fwd(has_tokens ? ws + base + l.u : nullptr, has_tokens ? ws + base + l.delta : nullptr,
                          reinterpret_cast<const float*>(ws + l.A), has_tokens ? ws + base + l.B : nullptr,
                          has_tokens ? ws + base + l.C : nullptr,
                          D ? reinterpret_cast<const float*>(ws + l.D) : nullptr,
                          (z && has_tokens) ? ws + base + l.z : nullptr,
                          delta_bias ? reinterpret_cast<const float*>(ws + l.bias) : nullptr,
                          delta_softplus, has_tokens ? ws + base + l.out : nullptr,
                          final_state ? reinterpret_cast<float*>(ws + base + l.fin) : nullptr, 1, dim,
                          dstate, seqlen, in_dtype, out_dtype,
                          initial_state ? reinterpret_cast<const float*>(ws + base + l.init) : nullptr,
                          scan_ws ? ws + base + l.scan_ws : nullptr, scan_ws, stream);
        if (st != SELSCAN_OK) return st;
        if (cudaEventRecord(pipe->scan_done[s], cs) != cudaSuccess) return fail();

        if (cudaStreamWaitEvent(pipe->out, pipe->scan_done[s], 0) != cudaSuccess) return fail();
        ok = !has_tokens || d2h(static_cast<char*>(out) + (size_t)i * act * eout, base + l.out, act * eout);
        if (ok && final_state) ok = d2h(final_state + (size_t)i * dim * 16, base + l.fin, stb);
        if (!ok || cudaEventRecord(pipe->out_done[s], pipe->out) != cudaSuccess) return fail();
    }
    // The caller's stream completes after the last download.
    for (int s = 0; s < kSlots && s < batch; ++s)
        if (cudaStreamWaitEvent(cs, pipe->out_done[s], 0) != cudaSuccess) return fail();
    return SELSCAN_OK;
}
