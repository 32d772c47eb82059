// Internal interface between the C-ABI entry points (selscan_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace selscan {

struct ScanArgs {
    const void* u;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* delta_bias;
    void* out;
    float* final_state;
    const float* initial_state;
    // Work of a scan, in blocks of consecutive channels of one batch (32, or 128 with `wide`):
    // nfull blocks run whole;
    // nsplit blocks are cut into nseg time segments of seg_len tokens (all blocks when nfull is
    // 0; else the last nsplit blocks of the last batch). Per launch, a CTA's block is
    // (b0 + blockIdx.z, bx0 + blockIdx.x) and its segment blockIdx.y; a whole-block launch
    // skips the blocks (skip_b, bx >= skip_bx0) that are cut (skip_bx0 = -1: none).
    float* ws_hloc;  // (cut blocks * 32, nseg-1, 16): local end state of segments 0..nseg-2
    float* ws_dsum;  // (cut blocks * 32, nseg-1): sum of Delta over those segments
    int64_t dim;
    int64_t seqlen;
    int64_t nfull;
    int64_t nsplit;
    int64_t seg_len;  // tokens per time segment, a multiple of the chunk length
    int nseg;         // time segments (1 = no split)
    int64_t bx0, b0;
    int64_t skip_bx0, skip_b;
    int wide;         // balanced plan: CTAs of 8 warps (128 channels), one per SM
    // Programmatic dependent launch of the balanced plan's three launches (wide CTA only):
    // bit 0 lets the next launch in the stream start its CTAs now, bit 1 waits for the earlier
    // grids before anything else, bit 2 waits for them before the CTA exits.
    int pdl;
    int softplus;
    int rows_per_lane;  // 1 or 2 (2 only honoured on the bf16 vector path)
    int zoh;            // zero-order-hold discretisation of B instead of Euler
    float* ckpt;        // (batch*dim, ceil(seqlen/16), 16): the state before every 16th token, or NULL
};

// Launches the local-end pass (nseg > 1) and the full pass on `stream`.
cudaError_t launch_scan_fwd(const ScanArgs& a, int64_t batch, bool in_bf16, bool out_bf16,
                            bool vec, bool precise, cudaStream_t stream);
int scan_chunk_tokens();  // time segments are multiples of this
// Workspace bytes without which a scan of this shape cannot run on the current device (its
// time split is needed for parallelism); a split that only balances the GPU is not counted.
size_t scan_required_workspace(int64_t batch, int64_t dim, int64_t seqlen);
int scan_rows_per_cta();
int scan_ctas_per_sm(int rows_per_lane);  // CTAs per SM the scan kernels are built to fit
int scan_wide_rows_per_cta();  // channels per CTA of the balanced plan's wide CTA

// Copies the device error bits raised by kernels of this library (synchronises `stream`);
// with `reset`, clears them afterwards.
cudaError_t read_device_status(unsigned int* status, bool reset, cudaStream_t stream);
// Launches one CTA that waits on an mbarrier no one arrives at, for at most `limit_cycles`
// SM clocks, and then raises the timeout bit exactly as a scan kernel would.
cudaError_t launch_wait_selftest(long long limit_cycles, cudaStream_t stream);

struct UpdateArgs {
    float* state;
    const void* x;
    const void* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    void* out;
    const float* dt_bias;
    int64_t dim;
    int64_t rows;  // batch*dim
    int softplus;
    int zoh;
    int sms;            // SMs of the device (sizes the launch)
    int early_trigger;  // set by the launcher: let the next grid start before this one's wait
    // Short causal convolution before the update (conv_state NULL = none); state NULL with a
    // conv_state runs the convolution step alone.
    void* conv_state;          // (rows, 4), input dtype, rolled in place
    const float* conv_weight;  // (dim, 4)
    const float* conv_bias;    // (dim) or NULL
    int conv_silu;
    void* conv_out;            // (rows), input dtype, or NULL
};

cudaError_t launch_state_update(const UpdateArgs& a, bool in_bf16, bool out_bf16,
                                cudaStream_t stream);

struct BwdArgs {
    const void* u;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* delta_bias;
    const float* initial_state;
    const void* dout;           // gradient dtype
    const float* dfinal_state;  // NULL = 0
    void* du;                   // gradient dtype
    void* ddelta;
    void* dz;                   // NULL iff z is NULL
    float* dA;
    float* dB;
    float* dC;
    float* dD;                  // NULL = not written
    float* ddelta_bias;         // NULL = not written
    float* dinitial_state;      // NULL = not written
    float* ws_ckpt;  // (batch*dim, chunks, 16): the state before every chunk
    int ckpt_given;  // ws_ckpt holds the forward's checkpoints (no checkpoint pass)
    float* ws_part;  // (channel blocks, batch, 32, seqlen): per-CTA sums of dB | dC
    float* ws_dA;    // (batch*dim, nseg, 16) per-row, per-segment sums
    float* ws_dD;    // (batch*dim, nseg)
    float* ws_db;    // (batch*dim, nseg)
    float* ws_hloc;  // (batch*dim, nseg-1, 16): local end states of segments 0..nseg-2
    float* ws_fsum;  // (batch*dim, nseg-1): their summed Delta
    float* ws_gloc;  // (batch*dim, nseg-1, 16): local start adjoints of segments 1..nseg-1
    float* ws_bsum;  // (batch*dim, nseg-1): their summed Delta
    int64_t batch;
    int64_t dim;
    int64_t seqlen;
    int64_t seg_len;  // tokens per time segment, a multiple of 16
    int nseg;         // time segments (1 = no split)
    int softplus;
    int sms;          // SMs of the device (launch shape)
};

// Workspace of the backward, in floats from its start.
struct BwdWorkspace {
    int64_t ckpt, part, dA, dD, db, hloc, fsum, gloc, bsum, total;
};
BwdWorkspace scan_bwd_workspace(int64_t batch, int64_t dim, int64_t seqlen, int nseg,
                                bool with_ckpt);
int scan_bwd_chunk_tokens();   // time segments are multiples of this
int scan_bwd_rows_per_cta();
int scan_bwd_ctas_per_sm();
int scan_bwd_ctas_per_sm_roomy();  // the instantiation a grid of at most sms x this many CTAs takes
// Launches the backward kernel and the reduction of its partial sums on `stream`.
cudaError_t launch_scan_bwd(const BwdArgs& a, bool in_bf16, bool grad_bf16, cudaStream_t stream);

// Mamba-2 SSD layer (bf16 inputs, headdim 64, dstate 128).
struct SsdArgs {
    const void* x;        // (batch, seqlen, nheads, 64) bf16
    const void* dt;       // (batch, seqlen, nheads) bf16
    const float* A;       // (nheads)
    const void* B;        // (batch, seqlen, ngroups, 128) bf16
    const void* C;
    const float* D;       // (nheads) or NULL
    const void* z;        // like x, or NULL
    const float* dt_bias; // (nheads) or NULL
    void* y;              // like x, output dtype
    float* final_state;   // (batch, nheads, 64, 128) or NULL
    const float* initial_state;
    int64_t batch;
    int64_t seqlen;
    int64_t nheads;
    int64_t ngroups;
    int softplus;
    // Balanced launch (set by launch_ssd_fwd): the first n_whole (batch, head) chains run whole,
    // the others are cut into nseg segments of seg_chunks chunks. job_mode 0: one CTA per chain
    // on a (nheads, batch) grid; 1: the local end states of segments 0..nseg-2 of the cut
    // chains (the state-only kernel); 2: every segment of the cut chains; 3: the whole chains.
    int job_mode;
    int64_t n_whole;
    int nseg;
    int seg_chunks;
    float* ws_sloc;   // (cut chains, nseg - 1, 64, 128): end states of segments from zero
    float* ws_sinit;  // (cut chains, nseg - 1, 64, 128): initial states of segments 1..nseg-1
    float* ws_dsum;   // (cut chains, nseg - 1): summed Delta*A*log2(e) of segments 0..nseg-2
};
// The balanced launch of an SSD call: cut chains, segments, chunks per segment and the
// workspace bytes it needs (all 0 / 1 when it does not pay).
struct SsdPlan {
    int64_t n_whole, n_cut;
    int nseg, seg_chunks;
    size_t workspace_bytes;
};
SsdPlan ssd_plan(int64_t batch, int64_t nheads, int64_t seqlen, int sms);
cudaError_t launch_ssd_fwd(const SsdArgs& a, bool out_bf16, void* workspace,
                           size_t workspace_bytes, int sms, cudaStream_t stream);
// Error bits raised by the SSD kernel (timeouts of its bounded waits); see read_device_status.
cudaError_t read_ssd_status(unsigned int* status, bool reset, cudaStream_t stream);

}  // namespace selscan
