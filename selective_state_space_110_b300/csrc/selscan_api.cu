// C-ABI entry points of libselscan: argument checks, time-segment planning, launches.
// The declarations and the contract (layouts, ownership, errors) are in include/selscan.h.
#include <cuda_runtime.h>

#include <algorithm>

#include "../../include/selscan.h"
#include "selscan_launch.h"

#define SELSCAN_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr int64_t kStateN = 16;
constexpr int64_t kMinSegTokens = 4096;  // shortest time segment worth a split for parallelism
constexpr int64_t kMinBalanceSegTokens = 64;  // shortest segment of the balanced plan's tail
constexpr int64_t kTwoRowsMinRows = 16384;  // rows from which two rows per lane pay off
constexpr int kKnownFlags = SELSCAN_FLAG_SOFTPLUS | SELSCAN_FLAG_ZOH;
constexpr int64_t kConvTaps = 4;  // width of the block's short convolution
constexpr size_t kWsAlign = 256;

size_t dtype_size(selscan_dtype t) { return t == SELSCAN_BF16 ? 2 : 4; }
bool dtype_ok(selscan_dtype t) { return t == SELSCAN_F32 || t == SELSCAN_BF16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};
Range range_of(const void* p, size_t bytes) {
    uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return {lo, lo + bytes};
}
bool overlaps(Range a, Range b) {
    return a.lo != a.hi && b.lo != b.hi && a.lo < b.hi && b.lo < a.hi;
}

// Current device's SM count; UNSUPPORTED unless it is compute capability 10.3 (sm_103).
selscan_status device_sms(int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return SELSCAN_ERR_CUDA; }
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return SELSCAN_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return SELSCAN_ERR_UNSUPPORTED;
    return SELSCAN_OK;
}

struct Plan {
    int rows_per_lane;
    int64_t gx;        // blocks of 32 channels per batch
    int64_t nfull;     // blocks run whole
    int64_t nsplit;    // blocks cut into time segments
    int nseg;          // segments per split block
    int64_t seg_len;
    bool wide;         // balanced plan: wide CTAs (128 channels), one per SM
    bool optional;     // the split only balances the GPU: without workspace, run unsplit
    size_t hloc_bytes, dsum_bytes, ws_bytes;
};

// Cost of a launch in units of one whole block's time at two warps per scheduler, with the
// measured per-scheduler throughput of the scan kernel at 1, 2 and 3+ resident warps (B300:
// 0.116, 0.154, 0.166 elements per clock): a scheduler with w warps of total work W blocks
// takes W * 0.154 / rate(w) units, since the warps share its issue slots.
double sched_time(double blocks_of_work, int warps) {
    const double rate = warps <= 1 ? 0.116 : warps == 2 ? 0.154 : 0.166;
    return blocks_of_work * 0.154 / rate;
}

void set_workspace(Plan& p, int64_t rows_split) {
    p.hloc_bytes = p.dsum_bytes = 0;
    if (p.nsplit > 0 && p.nseg > 1) {
        p.hloc_bytes = round_up((size_t)rows_split * (size_t)(p.nseg - 1) * kStateN * sizeof(float), kWsAlign);
        p.dsum_bytes = round_up((size_t)rows_split * (size_t)(p.nseg - 1) * sizeof(float), kWsAlign);
    }
    p.ws_bytes = p.hloc_bytes + p.dsum_bytes;
}

// The launch of one scan, in blocks of 32 consecutive channels of one batch (one CTA each).
//  - Few blocks for the GPU (they fill at most half of its CTA slots): every block is cut into
//    time segments, as many as fit every segment of the full pass into one wave. Each extra
//    segment costs a second pass over it (the local-end pass), so segments are used only when
//    the rows alone leave the GPU idle. The workspace is required.
//  - More blocks than two warps per scheduler hold (slots): a wave of whole blocks leaves the
//    remainder r = blocks mod slots for a last, partial wave in which most schedulers idle.
//    The balanced plan uses the wide CTA (128 channels, 8 warps), which its registers keep to
//    one per SM: q = blocks / SMs whole blocks per SM, and the r remainder blocks (the last r
//    blocks of the last batch) cut into as many time segments as there are SMs per remainder
//    block, so every SM gets the same work up to one segment. The segments run in a launch of
//    their own after the whole blocks.
//    It is taken when the cost model says it is faster than letting the hardware stack the
//    blocks unevenly, and only with a workspace (else the unsplit launch runs).
Plan make_plan(int64_t batch, int64_t dim, int64_t seqlen, int sms, bool fast) {
    const int64_t chunk = selscan::scan_chunk_tokens();
    const int64_t rows = batch * dim;
    const int64_t rpc = selscan::scan_rows_per_cta();
    Plan p{};
    p.gx = (dim + rpc - 1) / rpc;
    const int64_t blocks = batch * p.gx;
    p.nfull = blocks;
    p.nsplit = 0;
    p.nseg = 1;
    p.seg_len = std::max<int64_t>(seqlen, 1);
    p.rows_per_lane = rows >= kTwoRowsMinRows ? 2 : 1;

    // Few rows: time segments on every block.
    const int64_t slots6 = (int64_t)sms * selscan::scan_ctas_per_sm(2);
    if (2 * blocks <= slots6) {
        int64_t n = slots6 / blocks;
        n = std::min<int64_t>(n, seqlen / kMinSegTokens);
        n = std::max<int64_t>(n, 1);
        n = std::min<int64_t>(n, 65535);
        int64_t seg_len = (std::max<int64_t>(seqlen, 1) + n - 1) / n;
        seg_len = (seg_len + chunk - 1) / chunk * chunk;
        n = std::max<int64_t>(1, (seqlen + seg_len - 1) / seg_len);
        if (n > 1) {
            p.rows_per_lane = 2;
            p.nfull = 0;
            p.nsplit = blocks;
            p.nseg = (int)n;
            p.seg_len = seg_len;
        }
        set_workspace(p, p.nsplit * rpc);
        return p;
    }

    // Many rows: balance the last wave, with the wide CTA (128 channels, 8 warps: one per SM by
    // its registers) of the fast bf16 path.
    const int64_t wrpc = selscan::scan_wide_rows_per_cta();
    const int64_t wgx = (dim + wrpc - 1) / wrpc;
    const int64_t wblocks = batch * wgx;
    const int64_t q = wblocks / sms, r = wblocks % sms;
    // (The cut blocks are the last r blocks of the last batch, so r must not exceed its blocks.)
    if (fast && p.rows_per_lane == 2 && q >= 1 && r > 0 && r <= wgx &&
        seqlen >= 2 * kMinBalanceSegTokens) {
        int64_t n = std::min<int64_t>(sms / r, seqlen / kMinBalanceSegTokens);
        int64_t seg_len = (seqlen + n - 1) / n;
        seg_len = (seg_len + chunk - 1) / chunk * chunk;
        n = (seqlen + seg_len - 1) / seg_len;
        // Unsplit: the hardware spreads the 32-channel blocks over the SMs, and the busiest
        // scheduler holds ceil(blocks / sms) CTAs' worth of warps (two warps a CTA).
        const int64_t per_sm = (blocks + sms - 1) / sms;
        const int warps_sched = (int)((per_sm * 2 + 3) / 4);
        const double t_unsplit = sched_time((double)warps_sched, warps_sched);
        // Balanced: two warps per scheduler, q whole wide blocks plus one segment each, after
        // the local-end pass over the cut blocks' first n-1 segments (about 0.6 of a full pass).
        const double seg = (double)seg_len / (double)seqlen;
        const double t_split = sched_time(2.0 * ((double)q + seg), 2) + sched_time(2.0 * 0.6 * seg, 2);
        if (n >= 2 && t_split < t_unsplit) {
            p.gx = wgx;
            p.nfull = wblocks - r;
            p.nsplit = r;
            p.nseg = (int)n;
            p.seg_len = seg_len;
            p.wide = true;
            p.optional = true;
            set_workspace(p, p.nsplit * wrpc);
            return p;
        }
    }
    set_workspace(p, p.nsplit * rpc);
    return p;
}

// The plan to run with `ws_bytes` of workspace: the balanced split is dropped (unsplit launch)
// when the workspace cannot hold it.
// `fast`: the call takes the bf16 vector path without the zero-order hold (the only path with
// the wide CTA); the balanced split is dropped otherwise, or when the workspace cannot hold it.
Plan plan_for_workspace(int64_t batch, int64_t dim, int64_t seqlen, int sms, size_t ws_bytes,
                        bool fast) {
    Plan p = make_plan(batch, dim, seqlen, sms, fast);
    if (p.optional && ws_bytes < p.ws_bytes) p = make_plan(batch, dim, seqlen, sms, false);
    return p;
}

// The bf16 vector path without the zero-order hold: the one the balanced plan's wide CTA has.
bool fast_path(selscan_dtype in_dtype, int64_t seqlen, int flags) {
    return in_dtype == SELSCAN_BF16 && seqlen % 8 == 0 && !(flags & SELSCAN_FLAG_ZOH);
}

bool shape_ok(int64_t batch, int64_t dim, int64_t seqlen) {
    return batch >= 1 && dim >= 1 && seqlen >= 0 && batch <= 65535 &&
           dim <= (int64_t(1) << 40) && seqlen <= (int64_t(1) << 40);
}

}  // namespace

SELSCAN_EXPORT const char* selscan_status_string(selscan_status s) {
    switch (s) {
        case SELSCAN_OK: return "SELSCAN_OK";
        case SELSCAN_ERR_INVALID_ARG: return "SELSCAN_ERR_INVALID_ARG: null pointer, bad size or overlapping output";
        case SELSCAN_ERR_UNSUPPORTED: return "SELSCAN_ERR_UNSUPPORTED: dstate must be 16, dtype f32/bf16, device sm_103";
        case SELSCAN_ERR_ALIGNMENT: return "SELSCAN_ERR_ALIGNMENT: every pointer must be 16-byte aligned";
        case SELSCAN_ERR_WORKSPACE: return "SELSCAN_ERR_WORKSPACE: workspace missing or smaller than ssm_scan_workspace_size()";
        case SELSCAN_ERR_CUDA: return "SELSCAN_ERR_CUDA: the CUDA runtime reported an error";
        case SELSCAN_ERR_DEVICE_TIMEOUT: return "SELSCAN_ERR_DEVICE_TIMEOUT: a kernel gave up a bounded wait on the device (results of that launch are invalid)";
        case SELSCAN_ERR_SCRATCH_LIMIT: return "SELSCAN_ERR_SCRATCH_LIMIT: this shape needs more scratch than ssm_scan_fwd_no_alloc's static array (SELSCAN_NO_ALLOC_SCRATCH_BYTES); call ssm_scan_fwd with a workspace";
    }
    return "SELSCAN_ERR_UNKNOWN";
}

SELSCAN_EXPORT size_t ssm_scan_workspace_size(int64_t batch, int64_t dim, int64_t dstate,
                                              int64_t seqlen) {
    if (!shape_ok(batch, dim, seqlen) || dstate != kStateN) return 0;
    int sms = 0;
    if (device_sms(&sms) != SELSCAN_OK) return 0;
    return make_plan(batch, dim, seqlen, sms, true).ws_bytes;
}

SELSCAN_EXPORT selscan_status ssm_scan_plan(int64_t batch, int64_t dim, int64_t dstate,
                                            int64_t seqlen, selscan_dtype in_dtype, int flags,
                                            size_t workspace_bytes, int sms, int64_t* info) {
    if (!info || sms < 0 || sms > 4096) return SELSCAN_ERR_INVALID_ARG;
    if (dstate != kStateN || !dtype_ok(in_dtype)) return SELSCAN_ERR_UNSUPPORTED;
    if (!shape_ok(batch, dim, seqlen) || (flags & ~kKnownFlags)) return SELSCAN_ERR_INVALID_ARG;
    if (sms == 0) {
        const selscan_status s = device_sms(&sms);
        if (s != SELSCAN_OK) return s;
    }
    const Plan p = plan_for_workspace(batch, dim, seqlen, sms, workspace_bytes,
                                      fast_path(in_dtype, seqlen, flags));
    info[0] = p.rows_per_lane;
    info[1] = p.nfull;
    info[2] = p.nsplit;
    info[3] = p.nseg;
    info[4] = p.nsplit > 0 ? p.seg_len : seqlen;
    info[5] = p.wide ? selscan::scan_wide_rows_per_cta() : selscan::scan_rows_per_cta();
    info[6] = (int64_t)p.ws_bytes;
    info[7] = p.optional ? 0 : (int64_t)p.ws_bytes;
    return SELSCAN_OK;
}

namespace selscan {
size_t scan_required_workspace(int64_t batch, int64_t dim, int64_t seqlen) {
    if (!shape_ok(batch, dim, seqlen)) return 0;
    int sms = 0;
    if (device_sms(&sms) != SELSCAN_OK) return 0;
    const Plan p = make_plan(batch, dim, seqlen, sms, true);
    return p.optional ? 0 : p.ws_bytes;
}
}  // namespace selscan

namespace {
selscan_status scan_fwd_impl(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus, void* out,
    float* final_state, int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    selscan_dtype in_dtype, selscan_dtype out_dtype, const float* initial_state,
    void* workspace, size_t workspace_bytes, float* ckpt, selscan_stream_t stream) {
    // ---- checks that need no device ----
    if (dstate != kStateN || !dtype_ok(in_dtype) || !dtype_ok(out_dtype))
        return SELSCAN_ERR_UNSUPPORTED;
    if (!shape_ok(batch, dim, seqlen) || (delta_softplus & ~kKnownFlags)) return SELSCAN_ERR_INVALID_ARG;
    const bool has_tokens = seqlen > 0;
    if (!A || (has_tokens && (!u || !delta || !B || !C || !out))) return SELSCAN_ERR_INVALID_ARG;
    if (ckpt && (delta_softplus & SELSCAN_FLAG_ZOH)) return SELSCAN_ERR_UNSUPPORTED;
    const void* ptrs[] = {u, delta, A, B, C, D, z, delta_bias, out, final_state, initial_state, workspace, ckpt};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SELSCAN_ERR_ALIGNMENT;

    const size_t ein = dtype_size(in_dtype), eout = dtype_size(out_dtype);
    const size_t act = (size_t)batch * (size_t)dim * (size_t)seqlen;
    const size_t bc = (size_t)batch * kStateN * (size_t)seqlen;
    const size_t st = (size_t)batch * (size_t)dim * kStateN * sizeof(float);
    const size_t ck = (size_t)batch * (size_t)dim * (size_t)((seqlen + 15) / 16) * kStateN * sizeof(float);
    const Range in_r[] = {range_of(u, act * ein), range_of(delta, act * ein),
                          range_of(A, (size_t)dim * kStateN * 4), range_of(B, bc * ein),
                          range_of(C, bc * ein), range_of(D, D ? (size_t)dim * 4 : 0),
                          range_of(z, z ? act * ein : 0),
                          range_of(delta_bias, delta_bias ? (size_t)dim * 4 : 0),
                          range_of(initial_state, initial_state ? st : 0)};
    const Range out_r = range_of(out, has_tokens ? act * eout : 0);
    const Range fin_r = range_of(final_state, final_state ? st : 0);
    const Range ck_r = range_of(ckpt, ckpt ? ck : 0);
    for (const Range& r : in_r)
        if (overlaps(out_r, r) || overlaps(fin_r, r) || overlaps(ck_r, r)) return SELSCAN_ERR_INVALID_ARG;
    if (overlaps(out_r, fin_r) || overlaps(ck_r, out_r) || overlaps(ck_r, fin_r)) return SELSCAN_ERR_INVALID_ARG;

    // ---- device and plan ----
    int sms = 0;
    selscan_status s = device_sms(&sms);
    if (s != SELSCAN_OK) return s;
    const Plan plan = plan_for_workspace(batch, dim, seqlen, sms, workspace ? workspace_bytes : 0,
                                         fast_path(in_dtype, seqlen, delta_softplus));
    if (plan.ws_bytes > 0) {
        if (!workspace || workspace_bytes < plan.ws_bytes) return SELSCAN_ERR_WORKSPACE;
        const Range ws_r = range_of(workspace, plan.ws_bytes);
        for (const Range& r : in_r)
            if (overlaps(ws_r, r)) return SELSCAN_ERR_INVALID_ARG;
        if (overlaps(ws_r, out_r) || overlaps(ws_r, fin_r) || overlaps(ws_r, ck_r))
            return SELSCAN_ERR_INVALID_ARG;
    }

    selscan::ScanArgs a{};
    a.u = u; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z;
    a.delta_bias = delta_bias; a.out = out; a.final_state = final_state;
    a.initial_state = initial_state;
    a.ws_hloc = plan.ws_bytes ? static_cast<float*>(workspace) : nullptr;
    a.ws_dsum = plan.ws_bytes ? reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.hloc_bytes) : nullptr;
    a.dim = dim; a.seqlen = seqlen; a.seg_len = plan.seg_len; a.nseg = plan.nseg;
    a.nfull = plan.nfull; a.nsplit = plan.nsplit; a.wide = plan.wide ? 1 : 0;
    a.softplus = (delta_softplus & SELSCAN_FLAG_SOFTPLUS) ? 1 : 0;
    a.zoh = (delta_softplus & SELSCAN_FLAG_ZOH) ? 1 : 0;
    a.ckpt = ckpt;
    // Two rows per lane halves the shared-memory traffic of B and C but also the warps: worth it
    // once the rows alone give about two warps per scheduler, or when time segments supply
    // the parallelism.
    a.rows_per_lane = plan.rows_per_lane;
    // 128-bit loads of 8 tokens and TMA tiles of B / C need seqlen % 8 == 0 (16-byte row
    // strides) and 32-bit token coordinates.
    const bool vec = (seqlen % 8) == 0 && seqlen < (int64_t(1) << 31) - 64;
    const bool precise = in_dtype == SELSCAN_F32;
    cudaError_t e = selscan::launch_scan_fwd(a, batch, in_dtype == SELSCAN_BF16,
                                             out_dtype == SELSCAN_BF16, vec, precise,
                                             reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SELSCAN_OK : SELSCAN_ERR_CUDA;
}
}  // namespace

SELSCAN_EXPORT selscan_status ssm_scan_fwd(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus, void* out,
    float* final_state, int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    selscan_dtype in_dtype, selscan_dtype out_dtype, const float* initial_state,
    void* workspace, size_t workspace_bytes, selscan_stream_t stream) {
    return scan_fwd_impl(u, delta, A, B, C, D, z, delta_bias, delta_softplus, out, final_state,
                         batch, dim, dstate, seqlen, in_dtype, out_dtype, initial_state, workspace,
                         workspace_bytes, nullptr, stream);
}

SELSCAN_EXPORT selscan_status ssm_scan_fwd_ckpt(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus, void* out,
    float* final_state, int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    selscan_dtype in_dtype, selscan_dtype out_dtype, const float* initial_state,
    void* workspace, size_t workspace_bytes, float* checkpoints, selscan_stream_t stream) {
    if (!checkpoints && seqlen > 0) return SELSCAN_ERR_INVALID_ARG;
    return scan_fwd_impl(u, delta, A, B, C, D, z, delta_bias, delta_softplus, out, final_state,
                         batch, dim, dstate, seqlen, in_dtype, out_dtype, initial_state, workspace,
                         workspace_bytes, seqlen > 0 ? checkpoints : nullptr, stream);
}

SELSCAN_EXPORT selscan_status ssm_state_update(float* state, const void* x, const void* dt,
                                               const float* A, const void* B, const void* C,
                                               const float* D, const void* z, void* out,
                                               const float* dt_bias, int dt_softplus,
                                               int64_t batch, int64_t dim, int64_t dstate,
                                               selscan_dtype in_dtype, selscan_dtype out_dtype,
                                               selscan_stream_t stream) {
    if (dstate != kStateN || !dtype_ok(in_dtype) || !dtype_ok(out_dtype))
        return SELSCAN_ERR_UNSUPPORTED;
    if (!shape_ok(batch, dim, 0) || (dt_softplus & ~kKnownFlags)) return SELSCAN_ERR_INVALID_ARG;
    if (!state || !x || !dt || !A || !B || !C || !out) return SELSCAN_ERR_INVALID_ARG;
    const void* ptrs[] = {state, x, dt, A, B, C, D, z, out, dt_bias};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SELSCAN_ERR_ALIGNMENT;
    const size_t ein = dtype_size(in_dtype), eout = dtype_size(out_dtype);
    const size_t rows = (size_t)batch * (size_t)dim;
    const Range in_r[] = {range_of(x, rows * ein), range_of(dt, rows * ein),
                          range_of(A, (size_t)dim * kStateN * 4),
                          range_of(B, (size_t)batch * kStateN * ein),
                          range_of(C, (size_t)batch * kStateN * ein),
                          range_of(D, D ? (size_t)dim * 4 : 0), range_of(z, z ? rows * ein : 0),
                          range_of(dt_bias, dt_bias ? (size_t)dim * 4 : 0)};
    const Range st_r = range_of(state, rows * kStateN * sizeof(float));
    const Range out_r = range_of(out, rows * eout);
    for (const Range& r : in_r)
        if (overlaps(out_r, r) || overlaps(st_r, r)) return SELSCAN_ERR_INVALID_ARG;
    if (overlaps(out_r, st_r)) return SELSCAN_ERR_INVALID_ARG;

    int sms = 0;
    selscan_status s = device_sms(&sms);
    if (s != SELSCAN_OK) return s;
    selscan::UpdateArgs a{};
    a.state = state; a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z;
    a.out = out; a.dt_bias = dt_bias; a.dim = dim; a.rows = (int64_t)rows; a.sms = sms;
    a.softplus = (dt_softplus & SELSCAN_FLAG_SOFTPLUS) ? 1 : 0;
    a.zoh = (dt_softplus & SELSCAN_FLAG_ZOH) ? 1 : 0;
    cudaError_t e = selscan::launch_state_update(a, in_dtype == SELSCAN_BF16,
                                                 out_dtype == SELSCAN_BF16,
                                                 reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SELSCAN_OK : SELSCAN_ERR_CUDA;
}

SELSCAN_EXPORT selscan_status selscan_device_status(int reset, selscan_stream_t stream) {
    unsigned int bits = 0, ssd_bits = 0;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (selscan::read_device_status(&bits, reset != 0, s) != cudaSuccess ||
        selscan::read_ssd_status(&ssd_bits, reset != 0, s) != cudaSuccess) {
        cudaGetLastError();
        return SELSCAN_ERR_CUDA;
    }
    return (bits | ssd_bits) ? SELSCAN_ERR_DEVICE_TIMEOUT : SELSCAN_OK;
}

SELSCAN_EXPORT selscan_status selscan_selftest_wait_timeout(int64_t limit_cycles,
                                                            selscan_stream_t stream) {
    if (limit_cycles <= 0 || limit_cycles > (int64_t(1) << 32)) return SELSCAN_ERR_INVALID_ARG;
    int sms = 0;
    selscan_status s = device_sms(&sms);
    if (s != SELSCAN_OK) return s;
    return selscan::launch_wait_selftest(limit_cycles, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? SELSCAN_OK
               : SELSCAN_ERR_CUDA;
}

SELSCAN_EXPORT selscan_status ssm_conv_state_update(
    void* conv_state, const void* x, const float* conv_weight, const float* conv_bias,
    int conv_silu, int64_t conv_width, void* conv_out, float* state, const void* dt,
    const float* A, const void* B, const void* C, const float* D, const void* z, void* out,
    const float* dt_bias, int dt_flags, int64_t batch, int64_t dim, int64_t dstate,
    selscan_dtype in_dtype, selscan_dtype out_dtype, selscan_stream_t stream) {
    const bool ssm = state != nullptr;
    if (conv_width != kConvTaps || !dtype_ok(in_dtype) || (ssm && !dtype_ok(out_dtype)) ||
        (ssm && dstate != kStateN))
        return SELSCAN_ERR_UNSUPPORTED;
    if (!shape_ok(batch, dim, 0) || (dt_flags & ~kKnownFlags)) return SELSCAN_ERR_INVALID_ARG;
    if (!conv_state || !x || !conv_weight) return SELSCAN_ERR_INVALID_ARG;
    if (ssm ? (!dt || !A || !B || !C || !out) : !conv_out) return SELSCAN_ERR_INVALID_ARG;
    const void* ptrs[] = {conv_state, x, conv_weight, conv_bias, conv_out, state, dt, A, B, C,
                          D, z, out, dt_bias};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SELSCAN_ERR_ALIGNMENT;
    const size_t ein = dtype_size(in_dtype), eout = dtype_size(out_dtype);
    const size_t rows = (size_t)batch * (size_t)dim;
    const Range in_r[] = {range_of(x, rows * ein), range_of(conv_weight, (size_t)dim * kConvTaps * 4),
                          range_of(conv_bias, conv_bias ? (size_t)dim * 4 : 0),
                          range_of(dt, ssm ? rows * ein : 0),
                          range_of(A, ssm ? (size_t)dim * kStateN * 4 : 0),
                          range_of(B, ssm ? (size_t)batch * kStateN * ein : 0),
                          range_of(C, ssm ? (size_t)batch * kStateN * ein : 0),
                          range_of(D, ssm && D ? (size_t)dim * 4 : 0),
                          range_of(z, ssm && z ? rows * ein : 0),
                          range_of(dt_bias, ssm && dt_bias ? (size_t)dim * 4 : 0)};
    const Range out_r[] = {range_of(conv_state, rows * kConvTaps * ein),
                           range_of(conv_out, conv_out ? rows * ein : 0),
                           range_of(state, ssm ? rows * kStateN * sizeof(float) : 0),
                           range_of(out, ssm ? rows * eout : 0)};
    for (size_t i = 0; i < 4; ++i) {
        for (const Range& r : in_r)
            if (overlaps(out_r[i], r)) return SELSCAN_ERR_INVALID_ARG;
        for (size_t j = i + 1; j < 4; ++j)
            if (overlaps(out_r[i], out_r[j])) return SELSCAN_ERR_INVALID_ARG;
    }

    int sms = 0;
    selscan_status st = device_sms(&sms);
    if (st != SELSCAN_OK) return st;
    selscan::UpdateArgs a{};
    a.state = state; a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z;
    a.out = out; a.dt_bias = dt_bias; a.dim = dim; a.rows = (int64_t)rows; a.sms = sms;
    a.softplus = (dt_flags & SELSCAN_FLAG_SOFTPLUS) ? 1 : 0;
    a.zoh = (dt_flags & SELSCAN_FLAG_ZOH) ? 1 : 0;
    a.conv_state = conv_state; a.conv_weight = conv_weight; a.conv_bias = conv_bias;
    a.conv_silu = conv_silu ? 1 : 0; a.conv_out = conv_out;
    cudaError_t e = selscan::launch_state_update(a, in_dtype == SELSCAN_BF16,
                                                 out_dtype == SELSCAN_BF16,
                                                 reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SELSCAN_OK : SELSCAN_ERR_CUDA;
}

namespace {
// Time segments of the backward: split only when the rows alone fill less than half of the CTA
// slots (as the forward does). Of the segment counts that fit one wave (segments of at least
// kMinSegTokens), take the one with the least estimated time: with n segments the grid holds
// ctas * n CTAs, the most loaded SM p = ceil(ctas * n / sms) of them, each seqlen / n tokens
// long, and an SM's throughput depends on p. Measured on B300 (CTAs of 48 channels, 2,048
// tokens, one wave): 1, 2 and 3 CTAs per SM process 22.6, 33.9 and 31.2 G elements/s per
// SM-load, so the time is taken as p * kBwdSmCost[p] / n; ties go to fewer segments. 32 blocks on
// 148 SMs: 9 segments (2 CTAs per SM) rather than the 13 that fill the slots (3 per SM),
// 73.3 -> 69.1 ms for a million tokens.
constexpr int64_t kBwdSmCost[4] = {0, 150, 100, 109};  // 1 / relative throughput, x 100
struct BwdPlan {
    int nseg;
    int64_t seg_len;
};
BwdPlan make_bwd_plan(int64_t batch, int64_t dim, int64_t seqlen, int sms) {
    const int64_t chunk = selscan::scan_bwd_chunk_tokens();
    const int64_t rows_per_cta = selscan::scan_bwd_rows_per_cta();
    const int64_t ctas = batch * ((dim + rows_per_cta - 1) / rows_per_cta);
    const int ctas_per_sm = selscan::scan_bwd_ctas_per_sm();
    const int64_t slots = (int64_t)sms * ctas_per_sm;
    int64_t n = 1;
    if (2 * ctas <= slots) {
        int64_t nmax = slots / ctas;
        nmax = std::min<int64_t>(nmax, seqlen / kMinSegTokens);
        nmax = std::max<int64_t>(nmax, 1);
        nmax = std::min<int64_t>(nmax, 65535);
        // minimise cost(k) / k, compared as cost(k) * n < cost(n) * k
        int64_t best_cost = -1;
        for (int64_t k = 1; k <= nmax; ++k) {
            const int64_t per_sm = std::min<int64_t>((ctas * k + sms - 1) / sms, ctas_per_sm);
            const int64_t cost = per_sm * kBwdSmCost[std::min<int64_t>(per_sm, 3)];
            if (best_cost < 0 || cost * n < best_cost * k) {
                n = k;
                best_cost = cost;
            }
        }
    }
    int64_t seg_len = (std::max<int64_t>(seqlen, 1) + n - 1) / n;
    seg_len = (seg_len + chunk - 1) / chunk * chunk;
    n = std::max<int64_t>(1, (seqlen + seg_len - 1) / seg_len);
    return BwdPlan{(int)n, seg_len};
}
size_t bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int sms, bool ckpt_given) {
    const BwdPlan p = make_bwd_plan(batch, dim, seqlen, sms);
    return (size_t)selscan::scan_bwd_workspace(batch, dim, seqlen, p.nseg, !ckpt_given).total *
           sizeof(float);
}
}  // namespace

SELSCAN_EXPORT size_t ssm_scan_bwd_workspace_size(int64_t batch, int64_t dim, int64_t dstate,
                                                  int64_t seqlen, int checkpoints_given) {
    if (!shape_ok(batch, dim, seqlen) || dstate != kStateN) return 0;
    int sms = 0;
    if (device_sms(&sms) != SELSCAN_OK) return 0;
    return bwd_workspace_bytes(batch, dim, seqlen, sms, checkpoints_given != 0);
}

SELSCAN_EXPORT selscan_status ssm_scan_bwd_plan(int64_t batch, int64_t dim, int64_t dstate,
                                                int64_t seqlen, int checkpoints_given, int sms,
                                                int64_t* info) {
    if (!info || !shape_ok(batch, dim, seqlen) || dstate != kStateN || sms < 0 || sms > 4096)
        return SELSCAN_ERR_INVALID_ARG;
    if (sms == 0) {
        const selscan_status s = device_sms(&sms);
        if (s != SELSCAN_OK) return s;
    }
    const BwdPlan p = make_bwd_plan(batch, dim, seqlen, sms);
    const int64_t rows_per_cta = selscan::scan_bwd_rows_per_cta();
    const int64_t ctas = batch * ((dim + rows_per_cta - 1) / rows_per_cta) * p.nseg;
    info[0] = p.nseg;
    info[1] = p.seg_len;
    info[2] = rows_per_cta;
    info[3] = ctas;
    const int roomy = selscan::scan_bwd_ctas_per_sm_roomy();
    info[4] = ctas <= (int64_t)sms * roomy ? roomy : selscan::scan_bwd_ctas_per_sm();
    info[5] = (int64_t)bwd_workspace_bytes(batch, dim, seqlen, sms, checkpoints_given != 0);
    return SELSCAN_OK;
}

SELSCAN_EXPORT selscan_status ssm_scan_bwd(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    const float* initial_state, const void* dout, const float* dfinal_state, void* du,
    void* ddelta, float* dA, float* dB, float* dC, float* dD, void* dz, float* ddelta_bias,
    float* dinitial_state, int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    selscan_dtype in_dtype, selscan_dtype grad_dtype, const float* checkpoints,
    void* workspace, size_t workspace_bytes, selscan_stream_t stream) {
    if (dstate != kStateN || !dtype_ok(in_dtype) || !dtype_ok(grad_dtype))
        return SELSCAN_ERR_UNSUPPORTED;
    if (delta_softplus & SELSCAN_FLAG_ZOH) return SELSCAN_ERR_UNSUPPORTED;
    if (!shape_ok(batch, dim, seqlen) || (delta_softplus & ~kKnownFlags)) return SELSCAN_ERR_INVALID_ARG;
    const bool has_tokens = seqlen > 0;
    if (!A || !dA) return SELSCAN_ERR_INVALID_ARG;
    if (has_tokens && (!u || !delta || !B || !C || !dout || !du || !ddelta || !dB || !dC))
        return SELSCAN_ERR_INVALID_ARG;
    if (has_tokens && (z != nullptr) != (dz != nullptr)) return SELSCAN_ERR_INVALID_ARG;
    const void* ptrs[] = {u, delta, A, B, C, D, z, delta_bias, initial_state, dout,
                          dfinal_state, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias,
                          dinitial_state, workspace, checkpoints};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SELSCAN_ERR_ALIGNMENT;

    const size_t ein = dtype_size(in_dtype), eg = dtype_size(grad_dtype);
    const size_t act = (size_t)batch * (size_t)dim * (size_t)seqlen;
    const size_t bc = (size_t)batch * kStateN * (size_t)seqlen;
    const size_t st = (size_t)batch * (size_t)dim * kStateN * sizeof(float);
    const size_t dvec = (size_t)dim * 4;
    const Range in_r[] = {range_of(u, act * ein), range_of(delta, act * ein),
                          range_of(A, (size_t)dim * kStateN * 4), range_of(B, bc * ein),
                          range_of(C, bc * ein), range_of(D, D ? dvec : 0),
                          range_of(z, z ? act * ein : 0),
                          range_of(delta_bias, delta_bias ? dvec : 0),
                          range_of(initial_state, initial_state ? st : 0),
                          range_of(dout, act * eg),
                          range_of(dfinal_state, dfinal_state ? st : 0),
                          range_of(checkpoints, checkpoints ? (size_t)batch * dim * ((seqlen + 15) / 16) * kStateN * 4 : 0)};
    const Range out_r[] = {range_of(du, has_tokens ? act * eg : 0),
                           range_of(ddelta, has_tokens ? act * eg : 0),
                           range_of(dz, dz && has_tokens ? act * eg : 0),
                           range_of(dA, (size_t)dim * kStateN * 4),
                           range_of(dB, has_tokens ? bc * 4 : 0),
                           range_of(dC, has_tokens ? bc * 4 : 0),
                           range_of(dD, dD ? dvec : 0),
                           range_of(ddelta_bias, ddelta_bias ? dvec : 0),
                           range_of(dinitial_state, dinitial_state ? st : 0)};
    constexpr size_t kOuts = sizeof(out_r) / sizeof(out_r[0]);
    for (size_t i = 0; i < kOuts; ++i) {
        for (const Range& r : in_r)
            if (overlaps(out_r[i], r)) return SELSCAN_ERR_INVALID_ARG;
        for (size_t j = i + 1; j < kOuts; ++j)
            if (overlaps(out_r[i], out_r[j])) return SELSCAN_ERR_INVALID_ARG;
    }
    if (!workspace || workspace_bytes == 0) return SELSCAN_ERR_WORKSPACE;  // always needed

    // The time-segment plan (and so the workspace size) depends on the device's SM count.
    int sms = 0;
    selscan_status s = device_sms(&sms);
    if (s != SELSCAN_OK) return s;
    const BwdPlan plan = make_bwd_plan(batch, dim, seqlen, sms);
    const selscan::BwdWorkspace wl =
        selscan::scan_bwd_workspace(batch, dim, seqlen, plan.nseg, checkpoints == nullptr);
    const size_t ws_need = (size_t)wl.total * sizeof(float);
    if (workspace_bytes < ws_need) return SELSCAN_ERR_WORKSPACE;
    const Range ws_r = range_of(workspace, ws_need);
    for (const Range& r : in_r)
        if (overlaps(ws_r, r)) return SELSCAN_ERR_INVALID_ARG;
    for (const Range& r : out_r)
        if (overlaps(ws_r, r)) return SELSCAN_ERR_INVALID_ARG;

    float* ws = static_cast<float*>(workspace);
    selscan::BwdArgs a{};
    a.u = u; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z;
    a.delta_bias = delta_bias; a.initial_state = initial_state; a.dout = dout;
    a.dfinal_state = dfinal_state; a.du = du; a.ddelta = ddelta; a.dz = z ? dz : nullptr;
    a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD; a.ddelta_bias = ddelta_bias;
    a.dinitial_state = dinitial_state;
    a.ws_ckpt = checkpoints ? const_cast<float*>(checkpoints) : ws + wl.ckpt;
    a.ckpt_given = checkpoints ? 1 : 0;
    a.ws_part = ws + wl.part; a.ws_dA = ws + wl.dA;
    a.ws_dD = ws + wl.dD; a.ws_db = ws + wl.db; a.ws_hloc = ws + wl.hloc;
    a.ws_fsum = ws + wl.fsum; a.ws_gloc = ws + wl.gloc; a.ws_bsum = ws + wl.bsum;
    a.batch = batch; a.dim = dim; a.seqlen = seqlen;
    a.nseg = plan.nseg; a.seg_len = plan.seg_len; a.sms = sms;
    a.softplus = (delta_softplus & SELSCAN_FLAG_SOFTPLUS) ? 1 : 0;
    cudaError_t e = selscan::launch_scan_bwd(a, in_dtype == SELSCAN_BF16,
                                             grad_dtype == SELSCAN_BF16,
                                             reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SELSCAN_OK : SELSCAN_ERR_CUDA;
}

SELSCAN_EXPORT size_t ssd_chunk_scan_workspace_size(int64_t batch, int64_t seqlen,
                                                    int64_t nheads) {
    int sms = 0;
    if (batch < 1 || nheads < 1 || seqlen < 0 || device_sms(&sms) != SELSCAN_OK) return 0;
    return selscan::ssd_plan(batch, nheads, seqlen, sms).workspace_bytes;
}

SELSCAN_EXPORT selscan_status ssd_chunk_scan_plan(int64_t batch, int64_t seqlen, int64_t nheads,
                                                  int sms, int64_t* info) {
    if (!info || batch < 1 || nheads < 1 || seqlen < 0 || sms < 0 || sms > 4096)
        return SELSCAN_ERR_INVALID_ARG;
    if (sms == 0) {
        const selscan_status s = device_sms(&sms);
        if (s != SELSCAN_OK) return s;
    }
    const selscan::SsdPlan p = selscan::ssd_plan(batch, nheads, seqlen, sms);
    info[0] = p.n_whole;
    info[1] = p.n_cut;
    info[2] = p.nseg;
    info[3] = p.seg_chunks;
    info[4] = (int64_t)p.workspace_bytes;
    return SELSCAN_OK;
}

SELSCAN_EXPORT selscan_status ssd_chunk_scan_fwd(
    const void* x, const void* dt, const float* A, const void* B, const void* C, const float* D,
    const void* z, const float* dt_bias, int dt_softplus, void* y, float* final_state,
    const float* initial_state, int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
    int64_t ngroups, int64_t dstate, selscan_dtype in_dtype, selscan_dtype out_dtype,
    void* workspace, size_t workspace_bytes, selscan_stream_t stream) {
    if (headdim != 64 || dstate != 128 || in_dtype != SELSCAN_BF16 || !dtype_ok(out_dtype))
        return SELSCAN_ERR_UNSUPPORTED;
    if (batch < 1 || batch > 65535 || nheads < 1 || nheads > 65535 || ngroups < 1 ||
        nheads % ngroups != 0 || seqlen < 0 || seqlen > (int64_t(1) << 31) - 256 ||
        (dt_softplus & ~SELSCAN_FLAG_SOFTPLUS))
        return SELSCAN_ERR_INVALID_ARG;
    const bool has_tokens = seqlen > 0;
    if (!A || (has_tokens && (!x || !dt || !B || !C || !y))) return SELSCAN_ERR_INVALID_ARG;
    const void* ptrs[] = {x, dt, A, B, C, D, z, dt_bias, y, final_state, initial_state, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SELSCAN_ERR_ALIGNMENT;
    const size_t eout = dtype_size(out_dtype);
    const size_t act = (size_t)batch * (size_t)seqlen * (size_t)nheads * 64;
    const size_t bc = (size_t)batch * (size_t)seqlen * (size_t)ngroups * 128 * 2;
    const size_t st = (size_t)batch * (size_t)nheads * 64 * 128 * sizeof(float);
    const size_t hv = (size_t)nheads * 4;
    const Range in_r[] = {range_of(x, act * 2), range_of(dt, (size_t)batch * seqlen * nheads * 2),
                          range_of(A, hv), range_of(B, bc), range_of(C, bc),
                          range_of(D, D ? hv : 0), range_of(z, z ? act * 2 : 0),
                          range_of(dt_bias, dt_bias ? hv : 0),
                          range_of(initial_state, initial_state ? st : 0)};
    const Range y_r = range_of(y, has_tokens ? act * eout : 0);
    const Range fin_r = range_of(final_state, final_state ? st : 0);
    for (const Range& r : in_r)
        if (overlaps(y_r, r) || overlaps(fin_r, r)) return SELSCAN_ERR_INVALID_ARG;
    if (overlaps(y_r, fin_r)) return SELSCAN_ERR_INVALID_ARG;

    int sms = 0;
    selscan_status s = device_sms(&sms);
    if (s != SELSCAN_OK) return s;
    // The workspace only balances the last wave: without enough of it the chains run unsplit.
    const size_t ws_need = selscan::ssd_plan(batch, nheads, seqlen, sms).workspace_bytes;
    if (!workspace || workspace_bytes < ws_need) workspace = nullptr;
    if (workspace && ws_need) {
        const Range ws_r = range_of(workspace, ws_need);
        for (const Range& r : in_r)
            if (overlaps(ws_r, r)) return SELSCAN_ERR_INVALID_ARG;
        if (overlaps(ws_r, y_r) || overlaps(ws_r, fin_r)) return SELSCAN_ERR_INVALID_ARG;
    }
    selscan::SsdArgs a{};
    a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.dt_bias = dt_bias;
    a.y = y; a.final_state = final_state; a.initial_state = initial_state;
    a.batch = batch; a.seqlen = seqlen; a.nheads = nheads; a.ngroups = ngroups;
    a.softplus = (dt_softplus & SELSCAN_FLAG_SOFTPLUS) ? 1 : 0;
    cudaError_t e = selscan::launch_ssd_fwd(a, out_dtype == SELSCAN_BF16, workspace,
                                            workspace ? workspace_bytes : 0, sms,
                                            reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SELSCAN_ERR_CUDA;
    }
    return SELSCAN_OK;
}
