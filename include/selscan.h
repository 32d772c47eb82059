/*
 * libselscan: the selective state-space (S6) recurrence of Mamba on one B300 GPU.
 *
 * Two entry points compute the method; two more size and describe.
 *
 * The method ("Mamba and State Space Models", world.lapla.si):
 *   - section "A State of Fixed Size": every token updates a state of fixed size once,
 *     h <- Abar*h + Bbar*x, and the output is read from the updated state, y = C*h;
 *   - section "Chosen by the Token": Delta, B and C are computed from each token, A is
 *     fixed, and the retained fraction is Abar = exp(Delta*A);
 *   - section "A Scan on the Chip": Delta, A, B, C are read into on-chip memory,
 *     discretised and run through the recurrence there; only the output is written back,
 *     never the per-token state.
 * Per batch b, channel d, state index n and token t this library computes
 *     Delta   = softplus(delta[b,d,t] + delta_bias[d])     (no softplus if the flag is 0)
 *     h[n]    = exp(Delta*A[d,n]) * h[n] + Delta*B[b,n,t]*u[b,d,t]
 *     y       = (sum_n C[b,n,t]*h[n] + D[d]*u[b,d,t]) * silu(z[b,d,t]),  silu(z) = z/(1+e^-z)
 * with Euler discretisation of B, in fp32 arithmetic, for dstate = 16.
 *
 * Conventions shared by every entry point:
 *   - Pointers are device memory (or memory the device can address) owned by the caller.
 *     The library allocates nothing on a call's path and keeps no pointer after the call
 *     returns. Its only state, created once per device and kept until the process exits:
 *       * one device-side error word per device, which any kernel of the library that gives
 *         up a bounded wait sets, and which selscan_device_status reads and clears; it is
 *         shared by every stream and every call on that device, so a timeout raised on one
 *         stream is seen (and, with reset, cleared) by a reader on any other;
 *       * the fixed scratch array of ssm_scan_fwd_no_alloc;
 *       * the two copy streams and their events of ssm_scan_fwd_host.
 *     Apart from these, calls on different streams with different buffers are independent.
 *   - All work is enqueued asynchronously on `stream` (NULL = the legacy default stream).
 *     The returned status covers argument checks and the launch itself. A non-OK status
 *     means nothing was launched and no output was written (SELSCAN_ERR_CUDA excepted:
 *     the launch was attempted and the CUDA runtime reported an error).
 *   - Every pointer must be 16-byte aligned (SELSCAN_ERR_ALIGNMENT otherwise).
 *   - Outputs must not overlap inputs (SELSCAN_ERR_INVALID_ARG), except `state` of
 *     ssm_state_update, which is updated in place by design.
 *   - NaN and Inf in inputs propagate; they are not checked.
 */
#ifndef SELSCAN_H
#define SELSCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st* selscan_stream_t;

typedef enum {
    SELSCAN_F32 = 0,  /* IEEE fp32 */
    SELSCAN_BF16 = 1  /* bfloat16 */
} selscan_dtype;

/* Bits of the `delta_softplus` / `dt_softplus` argument. Other bits are rejected. */
enum {
    SELSCAN_FLAG_SOFTPLUS = 1, /* Delta = softplus(delta + bias); else Delta = delta + bias */
    SELSCAN_FLAG_ZOH = 2       /* zero-order hold: Bbar = ((exp(Delta*A) - 1)/A) * B instead of
                                  the Euler Bbar = Delta*B (the limit Delta*B where A = 0) */
};

typedef enum {
    SELSCAN_OK = 0,
    SELSCAN_ERR_INVALID_ARG = 1,  /* NULL required pointer, bad size, overlapping output */
    SELSCAN_ERR_UNSUPPORTED = 2,  /* dstate != 16, unknown dtype, no sm_103 device */
    SELSCAN_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned */
    SELSCAN_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than ssm_scan_workspace_size() */
    SELSCAN_ERR_CUDA = 5,         /* the CUDA runtime reported an error at launch */
    SELSCAN_ERR_SCRATCH_LIMIT = 6, /* ssm_scan_fwd_no_alloc: the shape needs more scratch than
                                      SELSCAN_NO_ALLOC_SCRATCH_BYTES */
    SELSCAN_ERR_DEVICE_TIMEOUT = 7 /* selscan_device_status: a kernel gave up a bounded wait */
} selscan_status;

/*
 * ssm_scan_fwd: the selective scan over a whole sequence (prefill / training forward).
 *
 * Layouts (contiguous, row-major, last index fastest):
 *   u, delta, z, out      (batch, dim, seqlen)       dtype in_dtype (out: out_dtype)
 *   B, C                  (batch, dstate, seqlen)    dtype in_dtype
 *   A                     (dim, dstate)              fp32, the fixed (negative) A
 *   D, delta_bias         (dim)                      fp32
 *   initial_state         (batch, dim, dstate)       fp32, NULL = zeros
 *   final_state           (batch, dim, dstate)       fp32, the state after token seqlen-1
 * Optional pointers: D (NULL = no skip term), z (NULL = no gate), delta_bias (NULL = 0),
 * initial_state, final_state (NULL = not written).
 * delta_softplus: flag bits. SELSCAN_FLAG_SOFTPLUS applies softplus to delta + delta_bias
 * (without it Delta = delta + delta_bias as is); SELSCAN_FLAG_ZOH selects the zero-order-hold
 * discretisation of B. With the zero-order hold and a single state number (A = -1, B = C = 1)
 * the update is the recurrent gate h <- (1 - g) h + g x, g = sigmoid(delta + delta_bias),
 * that "Chosen by the Token" describes. Unknown bits: SELSCAN_ERR_INVALID_ARG.
 * dstate must be 16. batch, dim >= 1; seqlen >= 0 (seqlen = 0 writes final_state only).
 * in_dtype applies to u, delta, z, B and C; out_dtype to out. Arithmetic is fp32.
 *
 * workspace / workspace_bytes: scratch device memory of ssm_scan_workspace_size(batch, dim,
 * dstate, seqlen) bytes (NULL/0 when that is 0). Some channel blocks (32 channels, or 128 in
 * the wide CTA of the balanced case below) are cut into time segments that run in parallel;
 * the workspace holds each segment's local end state and its summed Delta. Two cases (ssm_scan_plan reports which one a shape takes):
 *   - long sequences with few (batch, channel) rows are split for parallelism; the workspace
 *     is then required (SELSCAN_ERR_WORKSPACE without it);
 *   - shapes with more channel blocks than the GPU runs at once (bf16 inputs, seqlen % 8 == 0,
 *     no zero-order hold) have their last, partial wave cut into segments so every SM gets
 *     the same work; with a smaller workspace (or none) such a shape runs unsplit, correct but
 *     with an unbalanced last wave.
 * Its contents on entry do not matter. Two calls running at the same time need two
 * workspaces. The plan (and so the workspace size) is made for the current device: pass a
 * `stream` of that device.
 */
selscan_status ssm_scan_fwd(const void* u, const void* delta, const float* A, const void* B,
                            const void* C, const float* D, const void* z,
                            const float* delta_bias, int delta_softplus, void* out,
                            float* final_state, int64_t batch, int64_t dim, int64_t dstate,
                            int64_t seqlen, selscan_dtype in_dtype, selscan_dtype out_dtype,
                            const float* initial_state, void* workspace, size_t workspace_bytes,
                            selscan_stream_t stream);

/*
 * ssm_scan_fwd_ckpt: ssm_scan_fwd that also writes the state before every 16th token, for a
 * backward pass (ssm_scan_bwd) that then does not recompute it. The paper has no counterpart:
 * "A Scan on the Chip" recomputes the states in the backward pass; this trades 4 bytes per
 * (b, d, token) of memory for that pass.
 *   checkpoints  (batch, dim, ceil(seqlen/16), 16) fp32, device: entry [b, d, c, n] is state n
 *                before token 16*c (entry c = 0 is the initial state).
 * Everything else as ssm_scan_fwd. The zero-order hold is SELSCAN_ERR_UNSUPPORTED here (the
 * backward does not cover it); checkpoints must not overlap any other argument.
 */
selscan_status ssm_scan_fwd_ckpt(const void* u, const void* delta, const float* A, const void* B,
                                 const void* C, const float* D, const void* z,
                                 const float* delta_bias, int delta_softplus, void* out,
                                 float* final_state, int64_t batch, int64_t dim, int64_t dstate,
                                 int64_t seqlen, selscan_dtype in_dtype, selscan_dtype out_dtype,
                                 const float* initial_state, void* workspace,
                                 size_t workspace_bytes, float* checkpoints,
                                 selscan_stream_t stream);

/*
 * Workspace bytes ssm_scan_fwd uses for this shape on the CURRENT device (the time split
 * depends on its SM count), including a split that only balances the GPU (taken by bf16 inputs
 * with seqlen % 8 == 0 and no zero-order hold; other inputs use less of it). 0 means no
 * workspace is used. Returns 0 for invalid shapes (ssm_scan_fwd then reports the error).
 */
size_t ssm_scan_workspace_size(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen);

/*
 * ssm_scan_plan: how ssm_scan_fwd will launch this shape for inputs of `in_dtype`, flag bits
 * `flags` (as delta_softplus) and `workspace_bytes` of workspace, on a GPU of `sms` SMs (0 =
 * the current device; a positive count plans for that many SMs without touching any device).
 * The paper has no counterpart; it describes the launch for callers that size buffers or report
 * performance. info[0..7] (int64, host memory):
 *   [0] rows per lane (1 or 2)        [1] blocks of channels run whole
 *   [2] blocks cut into time segments [3] segments per cut block (1 = none)
 *   [4] tokens per segment            [5] channels per block (CTA)
 *   [6] workspace bytes this plan uses [7] workspace bytes the shape requires (the rest only
 *       balances the GPU)
 * Returns SELSCAN_ERR_INVALID_ARG for a NULL info, bad sizes, unknown flags or sms outside
 * 0..4096, SELSCAN_ERR_UNSUPPORTED for dstate != 16, an unknown dtype or (sms 0) a current
 * device that is not sm_103.
 */
selscan_status ssm_scan_plan(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                             selscan_dtype in_dtype, int flags, size_t workspace_bytes, int sms,
                             int64_t* info);

/*
 * ssm_state_update: one generated token ("Taken Apart": the head reads one token, computes
 * Delta, B and C, and the state moves once). The same update as one step of ssm_scan_fwd.
 *
 *   state                 (batch, dim, dstate)  fp32, read and overwritten in place
 *   x, dt, z, out         (batch, dim)          dtype in_dtype (out: out_dtype)
 *   B, C                  (batch, dstate)       dtype in_dtype
 *   A                     (dim, dstate)         fp32
 *   D, dt_bias            (dim)                 fp32, NULL = 0
 * z NULL = no gate. dt_softplus: the flag bits of delta_softplus above. dstate must be 16.
 * out must not overlap state or any input.
 */
selscan_status ssm_state_update(float* state, const void* x, const void* dt, const float* A,
                                const void* B, const void* C, const float* D, const void* z,
                                void* out, const float* dt_bias, int dt_softplus, int64_t batch,
                                int64_t dim, int64_t dstate, selscan_dtype in_dtype,
                                selscan_dtype out_dtype, selscan_stream_t stream);

/*
 * ssm_conv_state_update: the decode step of one layer's two fixed-size states. "A State of
 * Fixed Size" gives each channel its 16 state numbers "plus a short convolution that holds the
 * last 4 inputs"; this call moves both once per generated token in one kernel:
 *   1. the convolution window of each (b, d) drops its oldest input and takes x[b,d];
 *      u = sum_k conv_weight[d,k] * window[k] + conv_bias[d], then silu(u) if conv_silu;
 *   2. the state update of ssm_state_update with u as its input x (dt, B, C, z as given).
 *
 *   conv_state   (batch, dim, conv_width)  in_dtype, oldest input first, rolled in place
 *   x            (batch, dim)              in_dtype, the new input to the convolution
 *   conv_weight  (dim, conv_width) fp32;   conv_bias (dim) fp32, NULL = 0
 *   conv_out     (batch, dim)              in_dtype, u, NULL = not written
 *   state, dt, A, B, C, D, z, out, dt_bias, dt_flags: as ssm_state_update.
 * conv_width must be 4. With state == NULL only step 1 runs (conv_out is then required and the
 * state-update arguments are ignored): in a Mamba-1 block dt, B and C are projected from u by a
 * dense layer, so the caller runs step 1, the projection, then ssm_state_update. The fused
 * form fits blocks whose dt, B and C do not depend on u. Outputs must not overlap inputs or one
 * another (SELSCAN_ERR_INVALID_ARG); every pointer 16-byte aligned.
 */
selscan_status ssm_conv_state_update(void* conv_state, const void* x, const float* conv_weight,
                                     const float* conv_bias, int conv_silu, int64_t conv_width,
                                     void* conv_out, float* state, const void* dt, const float* A,
                                     const void* B, const void* C, const float* D, const void* z,
                                     void* out, const float* dt_bias, int dt_flags, int64_t batch,
                                     int64_t dim, int64_t dstate, selscan_dtype in_dtype,
                                     selscan_dtype out_dtype, selscan_stream_t stream);

/*
 * ssm_scan_fwd_no_alloc: ssm_scan_fwd for callers that cannot allocate device memory.
 *
 * The paper has no counterpart to this entry point; it exists for callers that have no way to
 * obtain scratch memory, such as code inside a host program whose framework owns every device
 * allocation and offers no allocator hook, or a latency-critical loop that must not call
 * cudaMalloc because it can synchronise the device. Arguments, layouts, results and errors are
 * those of ssm_scan_fwd without workspace / workspace_bytes: the time-split scratch is taken
 * from a fixed array of SELSCAN_NO_ALLOC_SCRATCH_BYTES bytes that the library declares in the
 * device memory of every GPU that loads it, held until the process exits. The call allocates
 * nothing and calls no allocating routine.
 *
 *   - Shapes whose required workspace (ssm_scan_plan info[7]) exceeds
 *     SELSCAN_NO_ALLOC_SCRATCH_BYTES are rejected with SELSCAN_ERR_SCRATCH_LIMIT before
 *     anything is launched; use ssm_scan_fwd with a workspace for them. A shape whose time
 *     split only balances the GPU uses it when it fits the array and runs unsplit otherwise.
 *     This size check comes before every other argument check: a shape beyond the array gets
 *     SELSCAN_ERR_SCRATCH_LIMIT even if a pointer is also NULL, misaligned or overlapping (no
 *     pointer is dereferenced or checked at that point).
 *   - `stream` must belong to the current device (cudaSetDevice): the array's address is the
 *     current device's, and a stream of another device is refused with
 *     SELSCAN_ERR_INVALID_ARG.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 *     once per device, with that device current). Make that first call before any stream
 *     capture on that device.
 *   - Every call on a device shares the one array, and the array keeps what the last call
 *     left in it (no part of it needs to start at zero). Calls that can overlap on the GPU
 *     (other streams, other host threads) race on it: serialise them, or use ssm_scan_fwd
 *     with one workspace per concurrent call.
 */
#define SELSCAN_NO_ALLOC_SCRATCH_BYTES ((size_t)524288) /* 512 KiB per device */

selscan_status ssm_scan_fwd_no_alloc(const void* u, const void* delta, const float* A,
                                     const void* B, const void* C, const float* D,
                                     const void* z, const float* delta_bias, int delta_softplus,
                                     void* out, float* final_state, int64_t batch, int64_t dim,
                                     int64_t dstate, int64_t seqlen, selscan_dtype in_dtype,
                                     selscan_dtype out_dtype, const float* initial_state,
                                     selscan_stream_t stream);

/*
 * ssm_scan_fwd_host: ssm_scan_fwd on HOST buffers. The paper has no counterpart; it serves
 * callers whose activations live in host memory. Arguments, layouts and results are those of
 * ssm_scan_fwd, except that u, delta, A, B, C, D, z, delta_bias, initial_state, out and
 * final_state are host pointers (pinned memory, e.g. cudaHostAlloc, lets the copies overlap the
 * scan; pageable memory works but serialises them). The batch is cut into slices of one
 * sequence: each slice is uploaded, scanned by ssm_scan_fwd on `stream` and downloaded, with the
 * upload of the next slice and the download of the previous one running during the scan on two
 * copy streams the library creates once per device. When the call returns the work is queued;
 * the host outputs are valid once `stream` has completed. Calls on one device must not overlap
 * (they share those streams and their events).
 *
 * workspace: device memory, 256-byte aligned, of at least ssm_scan_fwd_host_workspace_size()
 * bytes (two slices of inputs and outputs plus A, D, delta_bias); SELSCAN_ERR_WORKSPACE
 * otherwise. Its contents on entry do not matter.
 */
selscan_status ssm_scan_fwd_host(const void* u, const void* delta, const float* A, const void* B,
                                 const void* C, const float* D, const void* z,
                                 const float* delta_bias, int delta_softplus, void* out,
                                 float* final_state, int64_t batch, int64_t dim, int64_t dstate,
                                 int64_t seqlen, selscan_dtype in_dtype, selscan_dtype out_dtype,
                                 const float* initial_state, void* workspace,
                                 size_t workspace_bytes, selscan_stream_t stream);

/* Device workspace bytes ssm_scan_fwd_host needs (0 for invalid arguments). */
size_t ssm_scan_fwd_host_workspace_size(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                                        selscan_dtype in_dtype, selscan_dtype out_dtype);

/*
 * ssm_scan_bwd: gradients of the selective scan (Euler), for training. "A Scan on the Chip"
 * (world.lapla.si) keeps the expanded state out of main memory in the forward pass and computes
 * it again in the backward pass ("recomputation"); this call does the same: it stores the state
 * only every 16 tokens (in the workspace), recomputes each 16-token chunk's states on chip and
 * runs the adjoint recurrence of the scan backwards through them.
 *
 * With out, final_state the results of ssm_scan_fwd on the same inputs (Euler, no ZOH), it
 * returns the gradients of  sum(dout * out) + sum(dfinal_state * final_state)  with respect to
 * every input:
 *   du, ddelta, dz        (batch, dim, seqlen)     grad_dtype (like dout)
 *   dA                    (dim, dstate)            fp32, summed over batch and tokens
 *   dB, dC                (batch, dstate, seqlen)  fp32, summed over channels
 *   dD, ddelta_bias       (dim)                    fp32, NULL = not computed
 *   dinitial_state        (batch, dim, dstate)     fp32, NULL = not computed
 * Inputs u, delta, A, B, C, D, z, delta_bias, initial_state, delta_softplus: as ssm_scan_fwd
 * (in_dtype). dout (batch, dim, seqlen) in grad_dtype; dfinal_state (batch, dim, dstate) fp32,
 * NULL = zeros. dz is required exactly when z is given. Every output is overwritten (nothing is
 * accumulated into); the sums over channels and batches are taken in a fixed order, so results
 * are bitwise repeatable. SELSCAN_FLAG_ZOH: SELSCAN_ERR_UNSUPPORTED. Outputs must not overlap
 * inputs, one another or the workspace (SELSCAN_ERR_INVALID_ARG); every pointer 16-byte aligned.
 *
 * checkpoints: NULL, or the states written by ssm_scan_fwd_ckpt on the same inputs; the backward
 * then reads them instead of running its own forward pass.
 *
 * workspace: at least ssm_scan_bwd_workspace_size(..., checkpoints != NULL) bytes on the CURRENT
 * device (always > 0: without checkpoints the state every 16 tokens, 4 bytes per (b, d, token);
 * per-block partial sums of dB and dC, 4*batch*32*seqlen bytes per block of 48 channels;
 * per-row sums;
 * and, for long sequences with few rows, which are split into time segments as in the forward,
 * each segment's local end state and start adjoint). Its contents on entry do not matter.
 */
selscan_status ssm_scan_bwd(const void* u, const void* delta, const float* A, const void* B,
                            const void* C, const float* D, const void* z,
                            const float* delta_bias, int delta_softplus,
                            const float* initial_state, const void* dout,
                            const float* dfinal_state, void* du, void* ddelta, float* dA,
                            float* dB, float* dC, float* dD, void* dz, float* ddelta_bias,
                            float* dinitial_state, int64_t batch, int64_t dim, int64_t dstate,
                            int64_t seqlen, selscan_dtype in_dtype, selscan_dtype grad_dtype,
                            const float* checkpoints, void* workspace, size_t workspace_bytes,
                            selscan_stream_t stream);

/* Workspace bytes ssm_scan_bwd needs for this shape on the current device, with or without
 * checkpoints from ssm_scan_fwd_ckpt (0 for invalid shapes or no device). */
size_t ssm_scan_bwd_workspace_size(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                                   int checkpoints_given);

/*
 * ssm_scan_bwd_plan: the launch plan of ssm_scan_bwd for a shape on a GPU of `sms` SMs (0 = the
 * current device; a positive count touches no device). Rows are taken in CTAs of 48 channels;
 * when they fill less than half of the CTA slots, the sequence is cut into time segments
 * (each at least 4,096 tokens), as many as give the least work on the most loaded SM, weighted
 * by the measured throughput of an SM holding 1, 2 or 3 of these CTAs. info[0..5] (int64, host
 * memory): [0] time segments, [1] tokens per segment (a multiple of 16), [2] channels per CTA,
 * [3] CTAs of the full pass (channel blocks x batch x segments), [4] CTAs per SM its
 * instantiation is built for (2: 168 registers, dB / dC by per-chunk contractions; 3: 96
 * registers, by per-token shuffles), [5] workspace bytes (as ssm_scan_bwd_workspace_size with
 * checkpoints_given). SELSCAN_ERR_INVALID_ARG for a NULL info, bad sizes, dstate != 16 or sms
 * outside 0..4096.
 */
selscan_status ssm_scan_bwd_plan(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                                 int checkpoints_given, int sms, int64_t* info);

/*
 * ssd_chunk_scan_fwd: the Mamba-2 layer core, state space duality (SSD). "Mamba and State Space
 * Models" (world.lapla.si), section "Mamba-2": A is one number per head times the identity, so
 * the layer is one lower-triangular matrix per head (entry i, j = C_i . B_j times the decay
 * between j and i), computed in chunks: matrix products inside each chunk on the tensor cores,
 * only the state passed between chunks. Per batch b, head h (group g = h / (nheads/ngroups)):
 *   Delta_t  = softplus(dt[b,t,h] + dt_bias[h])   (dt + dt_bias without SELSCAN_FLAG_SOFTPLUS)
 *   H_t[p,n] = exp(Delta_t A[h]) H_{t-1}[p,n] + Delta_t x[b,t,h,p] B[b,t,g,n]
 *   y[b,t,h,p] = (sum_n C[b,t,g,n] H_t[p,n] + D[h] x[b,t,h,p]) * silu(z[b,t,h,p])
 * Layouts (contiguous, row-major):
 *   x, z, y          (batch, seqlen, nheads, headdim)   bf16 (y: out_dtype)
 *   dt               (batch, seqlen, nheads)            bf16
 *   B, C             (batch, seqlen, ngroups, dstate)   bf16
 *   A, D, dt_bias    (nheads)                           fp32; D, dt_bias NULL = 0
 *   initial_state, final_state  (batch, nheads, headdim, dstate)  fp32, NULL = zeros / not written
 * z NULL = no gate. headdim must be 64 and dstate 128 (the released Mamba-2 models' sizes),
 * in_dtype bf16, else SELSCAN_ERR_UNSUPPORTED; nheads % ngroups == 0. dt_softplus takes only
 * SELSCAN_FLAG_SOFTPLUS. Arithmetic: fp32 accumulation on the tensor cores; the products the
 * layer derives (the masked decay matrix, the decayed inputs, the state) enter as the sum of two
 * bf16 parts, which keeps about 16 significand bits. The state of each (b, h) stays on chip for
 * the whole sequence; nothing but y and the final state is written to the outputs.
 *
 * workspace (device, 16-byte aligned, owned by the caller, not read before it is written):
 * optional. One CTA per SM takes one (b, h) chain; when the chains fill whole waves of SMs and a
 * remainder, the remainder's chains are cut into time segments run in parallel (their end
 * states from zero in a first pass, folded into each segment's initial state, then the whole
 * chains and the segments), which needs ssd_chunk_scan_workspace_size() bytes. With NULL or
 * fewer bytes the chains run unsplit; the results agree to rounding. The workspace must not
 * overlap any input or output (SELSCAN_ERR_INVALID_ARG).
 */
selscan_status ssd_chunk_scan_fwd(const void* x, const void* dt, const float* A, const void* B,
                                  const void* C, const float* D, const void* z,
                                  const float* dt_bias, int dt_softplus, void* y,
                                  float* final_state, const float* initial_state, int64_t batch,
                                  int64_t seqlen, int64_t nheads, int64_t headdim,
                                  int64_t ngroups, int64_t dstate, selscan_dtype in_dtype,
                                  selscan_dtype out_dtype, void* workspace,
                                  size_t workspace_bytes, selscan_stream_t stream);

/*
 * ssd_chunk_scan_workspace_size: bytes of workspace ssd_chunk_scan_fwd uses to balance the
 * last wave of (batch x nheads) chains of seqlen tokens on the current device (0 = the chains
 * run unsplit: they fit one wave, fill whole waves, or are too short to cut; also 0 for
 * invalid shapes or without a device).
 */
size_t ssd_chunk_scan_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads);

/*
 * ssd_chunk_scan_plan: the balanced launch of ssd_chunk_scan_fwd for (batch x nheads) chains of
 * seqlen tokens on a GPU of `sms` SMs (0 = the current device; a positive count touches no
 * device). info[0..4] (int64, host memory): [0] chains run whole, [1] chains cut into time
 * segments (0 = none), [2] segments per cut chain, [3] chunks of 128 tokens per segment,
 * [4] workspace bytes. SELSCAN_ERR_INVALID_ARG for a NULL info, bad sizes or sms outside
 * 0..4096.
 */
selscan_status ssd_chunk_scan_plan(int64_t batch, int64_t seqlen, int64_t nheads, int sms,
                                   int64_t* info);

/*
 * selscan_device_status: errors that kernels of this library detected on the device.
 *
 * Every wait inside a kernel (for a TMA copy of B / C to land in shared memory) is bounded
 * (about two seconds of SM clock); a kernel that gives up records it in a device-side flag of
 * the library, leaves its outputs incomplete and exits normally, so the GPU and the context
 * stay usable. This call synchronises `stream`, then returns SELSCAN_ERR_DEVICE_TIMEOUT if the
 * flag is set on the current device (SELSCAN_OK otherwise); with `reset` nonzero it also clears
 * the flag. The flag is one word per device, shared by every stream and call of the library on
 * that device: a timeout raised by a launch on one stream is reported by a query on any stream,
 * and a reset from any stream clears it for all. Callers that need to know which call timed out
 * query right after that call, with no other call of the library in flight on the device.
 */
selscan_status selscan_device_status(int reset, selscan_stream_t stream);

/*
 * selscan_selftest_wait_timeout: test hook for the bounded waits. Launches one CTA that waits
 * on an mbarrier nothing arrives at, gives up after `limit_cycles` SM clocks (1 .. 2^32) and
 * sets the flag that selscan_device_status reports, as a scan kernel would. Nothing faults.
 */
selscan_status selscan_selftest_wait_timeout(int64_t limit_cycles, selscan_stream_t stream);

/* Static, human-readable name of a status code. */
const char* selscan_status_string(selscan_status status);

#ifdef __cplusplus
}
#endif

#endif /* SELSCAN_H */
