/*
 * ssm_gb300.h -- C ABI of the GB300 (sm_103a) Mamba-1 selective-scan library.
 *
 * The library computes the hot path of the Mamba-1 (S6) block described by the
 * CPU reference src/training/mamba1_cpu.ts (page "@seanhogg/builderforce-memory-
 * engine 2026.7.12 -> 2026.9.27"): the selective scan forward (mamba1CpuForward
 * steps 8-9) and backward (mamba1CpuBackward steps 9-8), and the causal
 * depthwise conv1d + SiLU (forward steps 4-5, backward steps 5-4), plus the
 * primitives of src/training/cpu_ops.ts they use (softplus, silu, sigmoid);
 * the whole block (steps 1-11 and their backward) with its projections on
 * the tensor cores; and single-token decode (the same recurrences one
 * position at a time from caller-held states).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Layout (the pages' "Layout conventions"): activations are row-major
 *    (M, width) with M = batch*seqlen and row r = b*seqlen + t.  Every
 *    activation tensor has its own row stride (ld_*, in ELEMENTS), so column
 *    slices of a wider projection (x | z of in_proj, dt | B | C of x_proj) are
 *    passed as base pointer + row stride, without a copy.  A stride of 0 means
 *    "packed" (dinner for (M, dinner) tensors, dstate for (M, dstate) tensors).
 *  - Ownership: the caller allocates and owns every buffer (inputs, outputs,
 *    saved context, workspace).  The library never allocates or frees memory.
 *    All pointers are DEVICE pointers unless stated otherwise.
 *  - Asynchrony: every call validates its arguments on the host, then enqueues
 *    its kernels on `stream` and returns; results are ready when the stream
 *    reaches that point.  Calls on one stream are ordered.
 *  - Errors: arguments are validated on the host before anything is launched;
 *    any status other than SSM_OK means NOTHING was enqueued, except
 *    SSM_ERR_LAUNCH, which reports a failed launch (cudaGetLastError) and may
 *    leave outputs partially written.  No kernel traps or asserts.
 *  - Outputs and gradients are WRITTEN, not accumulated.  (The pages add
 *    parameter gradients into a caller-owned accumulator; adding is the
 *    caller's job here.)
 *  - Alignment: every pointer to an (M, dinner) activation must be 16-byte
 *    aligned and its row stride times the element size must be a multiple of
 *    16 bytes; otherwise SSM_ERR_ALIGN.  B/C (and dB/dC) and the fp32
 *    parameter vectors need only natural alignment.
 *  - Arithmetic: fp32 state and accumulation in every case; SSM_BF16 changes
 *    only the storage type of the activations and their gradients (rounded to
 *    nearest even from fp32).
 */
#ifndef SSM_GB300_H
#define SSM_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSM_GB300_ABI_VERSION 1
#define SSM_MAX_DSTATE 16

typedef enum ssm_status {
    SSM_OK = 0,
    SSM_ERR_NULL = 1,       /* a required pointer is NULL */
    SSM_ERR_SHAPE = 2,      /* a size or stride is out of range */
    SSM_ERR_ALIGN = 3,      /* a pointer or row stride breaks the alignment rule */
    SSM_ERR_DTYPE = 4,      /* unknown dtype or discretisation */
    SSM_ERR_WORKSPACE = 5,  /* context or workspace smaller than required */
    SSM_ERR_LAUNCH = 6,     /* a kernel launch failed (see ssm_last_cuda_error) */
    SSM_ERR_DEVICE = 7      /* the current device is not an sm_103 GPU */
} ssm_status;

/* Storage type of the activations and their gradients. */
typedef enum ssm_dtype { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

/* Discretisation of B (the input matrix).
 *  SSM_DISC_EULER: beta = delta * B          -> h_t = exp(delta A) h_{t-1} + delta B_t u_t
 *  SSM_DISC_ZOH:   beta = (exp(delta A) - 1) / A * B, as mamba1_cpu.ts step 8
 *                  writes it (evaluated without cancellation for small delta*A). */
typedef enum ssm_disc { SSM_DISC_EULER = 0, SSM_DISC_ZOH = 1 } ssm_disc;

/* Shape, types and row strides of one selective-scan problem.
 *   u, delta_raw, z, out, dout, du, ddelta_raw, dz : (M, dinner), dtype
 *   B, C, dB, dC                                   : (M, dstate), dtype
 *   A_log : (dinner, dstate) fp32, packed;  D : (dinner) fp32
 * 0 <= dstate <= 16; batch <= 65535.  batch, seqlen or dinner may be 0 (empty
 * problem). */
typedef struct ssm_scan_desc {
    int32_t batch, seqlen, dinner, dstate;
    int32_t dtype;  /* ssm_dtype */
    int32_t disc;   /* ssm_disc  */
    int64_t ld_u, ld_delta, ld_z, ld_B, ld_C, ld_out;
    int64_t ld_dout, ld_du, ld_ddelta, ld_dz, ld_dB, ld_dC;
} ssm_scan_desc;

/* Bytes of the saved context that ssm_scan_fwd writes for ssm_scan_bwd: the
 * fp32 scan state h at every chunk boundary (the backward recomputes h inside
 * each chunk instead of reading an (M, dinner, dstate) history). */
size_t ssm_scan_ctx_bytes(const ssm_scan_desc* desc);

/* Bytes of device scratch that ssm_scan_fwd / ssm_scan_bwd need.  The
 * forward needs none unless the problem has few channels for its length
 * (batch * ceil(dinner/32) < 304 and seqlen >= 512): it then scans time
 * segments in parallel and keeps per-segment states (about
 * 2 * batch * segments * 16 * dinner floats). */
size_t ssm_scan_fwd_workspace_bytes(const ssm_scan_desc* desc);
size_t ssm_scan_bwd_workspace_bytes(const ssm_scan_desc* desc);

/* Selective scan forward (mamba1_cpu.ts mamba1CpuForward steps 8-9):
 *   delta = softplus(delta_raw)                        (cpu_ops.ts softplus)
 *   A     = -exp(clamp(A_log, -10, 5))                 (A_LOG_CLAMP_LO/HI)
 *   h_t   = exp(delta_t A) * h_{t-1} + beta_t * u_t,   h_{-1} = 0 per batch row
 *   y_t   = sum_n C_t[n] h_t[n] + D * u_t
 *   out_t = y_t * silu(z_t)     (or y_t when z == NULL: no gate)
 * D may be NULL (no skip term).  ctx may be NULL (inference: nothing saved);
 * otherwise it must hold ssm_scan_ctx_bytes(desc) bytes and is read by
 * ssm_scan_bwd.  workspace must hold ssm_scan_fwd_workspace_bytes(desc)
 * (may be NULL when that is 0). */
ssm_status ssm_scan_fwd(const ssm_scan_desc* desc,
                        const void* u, const void* delta_raw, const float* A_log,
                        const void* B, const void* C, const float* D, const void* z,
                        void* out, void* ctx, size_t ctx_bytes,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Selective scan backward (mamba1_cpu.ts mamba1CpuBackward steps 9-8), given
 * dout = dL/dout and the context of the matching ssm_scan_fwd call (same
 * inputs).  Writes
 *   du, ddelta_raw, dz (M, dinner) dtype;  dB, dC (M, dstate) dtype;
 *   dA_log (dinner, dstate) fp32 -- exactly 0 where A_log <= -10 or >= 5;
 *   dD (dinner) fp32 (may be NULL: not written).
 * dz is required iff z != NULL.  workspace must hold
 * ssm_scan_bwd_workspace_bytes(desc) bytes. */
ssm_status ssm_scan_bwd(const ssm_scan_desc* desc,
                        const void* u, const void* delta_raw, const float* A_log,
                        const void* B, const void* C, const float* D, const void* z,
                        const void* dout, const void* ctx, size_t ctx_bytes,
                        void* du, void* ddelta_raw, float* dA_log, void* dB, void* dC,
                        float* dD, void* dz,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Causal depthwise conv1d + SiLU (mamba1_cpu.ts forward steps 4-5):
 *   out[r, d] = silu(bias[d] + sum_{k < kconv, t >= k} w[d*kconv + k] * x[r - k, d])
 * x and out are (M, dinner) fp32 with row strides ld_x, ld_out (0 = packed);
 * w is (dinner, kconv) fp32 with tap k = 0 on the CURRENT step (the reverse of
 * torch.nn.Conv1d's weight order); bias (dinner) fp32 may be NULL.
 * 1 <= kconv <= 8.  out must not overlap x (a thread reads rows that another
 * thread's run writes). */
ssm_status ssm_conv1d_silu(int32_t batch, int32_t seqlen, int32_t dinner, int32_t kconv,
                           const float* x, int64_t ld_x, const float* w, const float* bias,
                           float* out, int64_t ld_out, cudaStream_t stream);

/* Backward of ssm_conv1d_silu (mamba1_cpu.ts backward steps 5-4): given
 * dout = dL/d(out) (ld_dout), writes dx (ld_dx), dw (dinner, kconv) and dbias
 * (dinner; may be NULL).  dx must not overlap x or dout.  workspace must hold
 * ssm_conv1d_silu_bwd_workspace_bytes(...) bytes. */
size_t ssm_conv1d_silu_bwd_workspace_bytes(int32_t batch, int32_t seqlen, int32_t dinner,
                                           int32_t kconv);
ssm_status ssm_conv1d_silu_bwd(int32_t batch, int32_t seqlen, int32_t dinner, int32_t kconv,
                               const float* x, int64_t ld_x, const float* w, const float* bias,
                               const float* dout, int64_t ld_dout,
                               float* dx, int64_t ld_dx, float* dw, float* dbias,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Linear layer (cpu_ops.ts linearForward): Y (M, N) = X (M, K) W^T + bias
 * (+ R), fp32, on the tensor cores as three TF32 products of hi/lo splits
 * that the GEMM forms from the fp32 tiles itself, with the partial sums
 * drained to fp32 every 128 K (about fp32 accuracy).  W is (N, K) as
 * torch.nn.Linear stores it; row strides ldx, ldw, ldr, ldy in elements
 * (0 = packed); bias (N) and R (M, N) may be NULL; R may alias Y.  X and W
 * are read in place when 16-byte aligned with a row stride that is a multiple
 * of 4 elements, else copied into the workspace first.  workspace (16-byte
 * aligned) must hold ssm_linear_workspace_bytes(M, N, K) bytes.  K = 0 is
 * rejected (SSM_ERR_SHAPE). */
size_t ssm_linear_workspace_bytes(int32_t M, int32_t N, int32_t K);
ssm_status ssm_linear_fwd(int32_t M, int32_t N, int32_t K, const float* X, int64_t ldx,
                          const float* W, int64_t ldw, const float* bias, const float* R,
                          int64_t ldr, float* Y, int64_t ldy,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---- The whole Mamba-1 block (mamba1_cpu.ts mamba1CpuForward /
 * mamba1CpuBackward, with the linear and RMSNorm primitives of cpu_ops.ts):
 *   xn   = rmsnorm(x) * norm_w            inv = 1/sqrt(mean(x^2) + 1e-6)
 *   xz   = xn in_proj_w^T + in_proj_b      (M, 2 dinner) -> x_in | z
 *   u    = silu(conv1d(x_in))              causal depthwise, kconv taps
 *   xd   = u x_proj_w^T + x_proj_b         (M, dtrank + 2 dstate) -> dt | B | C
 *   draw = dt dt_proj_w^T + dt_proj_b      (M, dinner): the scan's delta_raw
 *   g    = scan(u, draw, A_log, B, C, D) * silu(z)
 *   out  = g out_proj_w^T + out_proj_b + x
 * Every tensor is fp32, row-major and packed; weights are (out, in) as
 * torch.nn.Linear stores them, conv_w is (dinner, kconv) with tap 0 on the
 * current step.  The projections run on the tensor cores as three TF32
 * products of hi/lo splits (about fp32 accuracy); the scan is ssm_scan_fwd /
 * ssm_scan_bwd.  dmodel, dinner, dtrank and dstate must be multiples of 4
 * (else SSM_ERR_ALIGN); 1 <= dstate <= 16; 1 <= kconv <= 8; dtrank >= 1. */
typedef struct ssm_block_desc {
    int32_t batch, seqlen, dmodel, dinner, dstate, dtrank, dconv;
    int32_t disc;  /* ssm_disc */
} ssm_block_desc;

/* The 13 block parameters, in the pages' order (Mamba1CpuWeights). */
typedef struct ssm_block_weights {
    const float *in_proj_w, *in_proj_b, *conv_w, *conv_b, *x_proj_w, *x_proj_b,
                *dt_proj_w, *dt_proj_b, *A_log, *D, *out_proj_w, *out_proj_b, *norm_w;
} ssm_block_weights;
/* Their gradients (same shapes), written by ssm_block_bwd. */
typedef struct ssm_block_grads {
    float *in_proj_w, *in_proj_b, *conv_w, *conv_b, *x_proj_w, *x_proj_b,
          *dt_proj_w, *dt_proj_b, *A_log, *D, *out_proj_w, *out_proj_b, *norm_w;
} ssm_block_grads;

/* Bytes of the activations ssm_block_fwd saves for ssm_block_bwd (xn, inv,
 * xz, u, xd, draw, g and the scan context), and of the device scratch either
 * call needs.  0 for an invalid descriptor. */
size_t ssm_block_ctx_bytes(const ssm_block_desc* desc);
size_t ssm_block_workspace_bytes(const ssm_block_desc* desc);

/* Block forward: x, out (M, dmodel).  ctx (required, 16-byte aligned) must
 * hold ssm_block_ctx_bytes and workspace ssm_block_workspace_bytes bytes;
 * out may not alias x.  Every weight pointer is required. */
ssm_status ssm_block_fwd(const ssm_block_desc* desc, const float* x,
                         const ssm_block_weights* weights, float* out,
                         void* ctx, size_t ctx_bytes,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Block backward, given dout = dL/d(out) (M, dmodel) and the ctx written by
 * ssm_block_fwd for the same x and weights: writes dx (M, dmodel) and every
 * gradient in *grads (all required). */
ssm_status ssm_block_bwd(const ssm_block_desc* desc, const float* x,
                         const ssm_block_weights* weights, const float* dout,
                         const void* ctx, size_t ctx_bytes, float* dx,
                         const ssm_block_grads* grads,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---- A stack of blocks with activation checkpointing (the model of the
 * pages "@seanhogg/builderforce-memory-engine 2026.7.14 -> 2026.9.28",
 * src/training/model_cpu.js: forwardInternal runs the layers one after
 * another; cpuModelBackward walks them last to first and, with activation
 * checkpointing, recomputes each layer's forward from that layer's saved
 * input before its backward -- the same gradients as keeping every
 * activation).  Here: hidden_0 = x, hidden_{i+1} = block_i(hidden_i) for
 * i < layers (each block with its own residual), out = hidden_layers.
 *  - weights / grads: arrays of `layers` structs, one per layer, as for
 *    ssm_block_fwd / ssm_block_bwd (all pointers required).
 *  - ctx (ssm_stack_ctx_bytes, 16-byte aligned; may be NULL for one layer)
 *    keeps only the layer inputs hidden_1 .. hidden_{layers-1}, (layers-1) x
 *    batch*seqlen x dmodel fp32 -- not the per-layer block contexts.
 *  - workspace (ssm_stack_workspace_bytes, 16-byte aligned) holds one block
 *    context and one block workspace that every layer reuses, plus three
 *    (batch*seqlen, dmodel) buffers for the backward.
 *  - ssm_stack_bwd recomputes each layer's forward once (one extra block
 *    forward per layer), then runs its backward; dx and every layer's
 *    gradients are written.  x, weights and ctx must be those of the
 *    matching ssm_stack_fwd call.
 * Other rules as ssm_block_fwd / ssm_block_bwd; layers < 1 is SSM_ERR_SHAPE;
 * 0 for an invalid descriptor from the size queries. */
size_t ssm_stack_ctx_bytes(const ssm_block_desc* desc, int32_t layers);
size_t ssm_stack_workspace_bytes(const ssm_block_desc* desc, int32_t layers);
ssm_status ssm_stack_fwd(const ssm_block_desc* desc, int32_t layers, const float* x,
                         const ssm_block_weights* weights, float* out, void* ctx, size_t ctx_bytes,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);
ssm_status ssm_stack_bwd(const ssm_block_desc* desc, int32_t layers, const float* x,
                         const ssm_block_weights* weights, const float* dout, const void* ctx,
                         size_t ctx_bytes, float* dx, const ssm_block_grads* grads,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ssm_conv1d_silu_bwd without a workspace argument: the same result as
 * ssm_conv1d_silu_bwd, but the per-run dw/dbias partial sums live in scratch
 * that the library reserves once, as a fixed 8 MiB array in the device image,
 * instead of in caller memory.  (The pages have no counterpart; this is an
 * interface convenience.)  It is meant for callers that cannot give the
 * library any scratch: a runtime or plugin interface that owns every device
 * buffer and offers kernels none, or a loop where a cudaMalloc -- which may
 * synchronise the device -- is not allowed.  The function itself allocates
 * nothing.
 *  - Capacity: ceil(seqlen / 64) * batch * dinner * (kconv + 1) floats must not
 *    exceed 2^21 (8 MiB); larger problems return SSM_ERR_WORKSPACE and launch
 *    nothing.
 *  - The first call on a device looks up the scratch's device address (once per
 *    device and CUDA context, with that device current); make that first call
 *    before any stream capture.  A call after the context was destroyed and
 *    made again (cudaDeviceReset, or the primary context released and
 *    retained anew) looks the address up again, since the array may have moved.
 *  - Every call on a device shares the one scratch array, and it keeps the
 *    last call's contents; each call writes every partial it reads, so nothing
 *    has to start at zero.  Calls that overlap on the GPU (for example on two
 *    streams at once) race on the scratch and must not be issued.
 * Other arguments, layouts and errors as ssm_conv1d_silu_bwd. */
ssm_status ssm_conv1d_silu_bwd_noalloc(int32_t batch, int32_t seqlen, int32_t dinner,
                                       int32_t kconv, const float* x, int64_t ld_x,
                                       const float* w, const float* bias, const float* dout,
                                       int64_t ld_dout, float* dx, int64_t ld_dx, float* dw,
                                       float* dbias, cudaStream_t stream);

/* ---- Single-token decode (inference) ----------------------------------
 * The same recurrence one position at a time, for serving: the scan state of
 * a batch of sequences is kept by the caller between calls.
 *   h    : (batch, dstate, dinner) fp32, element (b, n, d) at
 *          h[(b*dstate + n)*dinner + d]; 16-byte aligned.
 *   conv_state : (batch, kconv-1, dinner) fp32, the conv1d's previous inputs:
 *          slot j holds the input kconv-1-j steps back, element (b, j, d) at
 *          conv_state[(b*(kconv-1) + j)*dinner + d]; 16-byte aligned.  A new
 *          sequence starts from zeros (no input before position 0); each step
 *          shifts the slots by one, so a decode step takes no position and the
 *          same call can be replayed (e.g. from a CUDA graph) at every position. */

/* Scan forward from a carried state and/or returning the final state (prefill):
 * ssm_scan_fwd without a saved context, plus
 *   h_init : state before the first step of every batch row (NULL = zero);
 *   h_last : receives the state after the last step (may be NULL).
 * Both (batch, dstate, dinner) as above, 4-byte aligned, and they must not
 * overlap (SSM_ERR_SHAPE).  seqlen = 0 copies h_init (or zero) to h_last.
 * There is no backward for a non-zero h_init.  workspace as ssm_scan_fwd. */
ssm_status ssm_scan_fwd_state(const ssm_scan_desc* desc,
                              const void* u, const void* delta_raw, const float* A_log,
                              const void* B, const void* C, const float* D, const void* z,
                              void* out, const float* h_init, float* h_last,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* One decode step of the scan (mamba1_cpu.ts mamba1CpuForward steps 8-9 at a
 * single position): desc->seqlen must be 1 and row b of every activation
 * belongs to batch row b.  For every (b, d):
 *   delta = softplus(delta_raw);  h[b,n,d] <- exp(delta A[d,n]) h[b,n,d] + beta u
 *   out = (sum_n C[b,n] h[b,n,d] + D[d] u) * silu(z)     (no gate when z == NULL)
 * h is read and overwritten in place.  D may be NULL.  Activation types,
 * strides and alignment as ssm_scan_fwd. */
ssm_status ssm_scan_step(const ssm_scan_desc* desc,
                         const void* u, const void* delta_raw, const float* A_log,
                         const void* B, const void* C, const float* D, const void* z,
                         float* h, void* out, cudaStream_t stream);

/* One decode step of the causal depthwise conv1d + SiLU (mamba1_cpu.ts
 * forward steps 4-5 at one position):
 *   out[b,d] = silu(bias[d] + w[d,0] x[b,d] + sum_{1<=k<kconv} w[d,k] conv_state[b, kconv-1-k, d])
 * then conv_state[b, j] <- conv_state[b, j+1] and conv_state[b, kconv-2] <- x.
 * x, out: (batch, dinner) fp32 with row strides ld_x, ld_out (0 = packed);
 * w (dinner, kconv), tap 0 on the current input; bias may be NULL.
 * dinner, ld_x, ld_out multiples of 4 and x, out, conv_state, bias 16-byte
 * aligned (else SSM_ERR_ALIGN); 1 <= kconv <= 8 (kconv = 1: no state, may be
 * NULL). */
ssm_status ssm_conv1d_silu_step(int32_t batch, int32_t dinner, int32_t kconv,
                                const float* x, int64_t ld_x, const float* w, const float* bias,
                                float* conv_state, float* out, int64_t ld_out, cudaStream_t stream);

/* The conv_state that continues a prompt x (batch*seqlen, dinner) fp32 (row
 * stride ld_x) at position seqlen: slot j <- the input at position
 * seqlen-(kconv-1)+j, or zero where that is before 0.  Alignment as
 * ssm_conv1d_silu_step. */
ssm_status ssm_conv1d_state_from_prompt(int32_t batch, int32_t seqlen, int32_t dinner,
                                        int32_t kconv, const float* x, int64_t ld_x,
                                        float* conv_state, cudaStream_t stream);

/* ssm_block_fwd that also leaves, for every batch row, the states after the
 * last position (prefill before ssm_block_step): conv_state (batch, dconv-1,
 * dinner) and h (batch, dstate, dinner), each 16-byte aligned and may be NULL
 * (not written).  The forward starts from zero states (new sequences).
 * seqlen = 0 writes zero states.  Other arguments as ssm_block_fwd. */
ssm_status ssm_block_fwd_state(const ssm_block_desc* desc, const float* x,
                               const ssm_block_weights* weights, float* out,
                               void* ctx, size_t ctx_bytes, float* conv_state, float* h,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* One decode step of the whole block (mamba1_cpu.ts mamba1CpuForward steps
 * 1-11 at a single position): desc->seqlen must be 1 (SSM_ERR_SHAPE) and x,
 * out are (batch, dmodel) fp32, row b = the next token of sequence b.  The
 * conv1d and the scan continue from conv_state (batch, dconv-1, dinner) and
 * h (batch, dstate, dinner), laid out as for ssm_conv1d_silu_step and
 * ssm_scan_step and updated in place (zeros for new sequences).  The
 * projections run as in ssm_block_fwd (with batch rows); weights_split, if
 * not NULL, holds the copies made by ssm_block_split_weights for these
 * weights (else the weights are read in place, or copied into the workspace
 * when not 16-byte aligned).  workspace (16-byte aligned)
 * must hold ssm_block_step_workspace_bytes(desc) bytes (0 for an invalid
 * descriptor).  Other rules as ssm_block_fwd. */
size_t ssm_block_step_workspace_bytes(const ssm_block_desc* desc);
ssm_status ssm_block_step(const ssm_block_desc* desc, const float* x,
                          const ssm_block_weights* weights, const void* weights_split,
                          float* conv_state, float* h, float* out, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream);

/* The four projection weights as the GEMM reads them (16-byte aligned copies,
 * rows padded to a multiple of 4 floats), made once for many ssm_block_step
 * calls with the same weights (decode): split (16-byte aligned) must hold
 * ssm_block_weights_split_bytes(desc) bytes; batch and seqlen of desc do not
 * matter.  (The GEMM forms the TF32 hi/lo halves itself.) */
size_t ssm_block_weights_split_bytes(const ssm_block_desc* desc);
ssm_status ssm_block_split_weights(const ssm_block_desc* desc, const ssm_block_weights* weights,
                                   void* split, size_t split_bytes, cudaStream_t stream);

/* ---- Measurement helper (no counterpart in the pages) ------------------
 * Throughput probe of one arithmetic pipe, used by the benchmark to measure
 * the rates its roofline divides by: kind 0 = MUFU ex2 (ex2.approx.ftz.f32),
 * 1 = scalar fp32 FFMA, 2 = packed f32x2 FFMA2.  Launches `blocks` CTAs of
 * 256 threads; each thread runs 8 independent dependency chains (4 packed
 * pairs for kind 2) of `iters` steps, i.e. blocks*256*iters*8 lane-operations,
 * and writes one float per thread to sink (blocks*256 floats, device).  The
 * caller times the launch (CUDA events) and reads the SM clock.  Kinds 3 and
 * 4 are for counting instructions, not rates: 4 packed chains whose FFMA2
 * multiplier is a scalar broadcast to both halves (3) or a pair (4).
 * Returns SSM_ERR_SHAPE for a kind outside 0..4 or non-positive sizes,
 * SSM_ERR_NULL for a NULL sink, SSM_ERR_LAUNCH if the launch fails. */
ssm_status ssm_probe_pipe(int32_t kind, int32_t blocks, int32_t iters, float* sink,
                          cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char* ssm_status_string(ssm_status status);

/* The cudaError_t of the most recent SSM_ERR_LAUNCH / SSM_ERR_DEVICE on the
 * calling thread (cudaSuccess if none). */
int ssm_last_cuda_error(void);

/* SSM_GB300_ABI_VERSION of the built library. */
int ssm_abi_version(void);

/* Fault bits recorded by the kernels since the last call, then cleared:
 * every wait of a kernel on an asynchronous copy is bounded, and a wait that
 * gives up sets a bit here (1: forward copy wait, 2: backward copy wait,
 * 4: drain after a failed wait, 8: block GEMM pipeline wait, 16: the
 * self-test below) instead of hanging; that call's outputs are
 * then invalid.  Synchronous: call it after the work has completed.  Returns
 * 0 when no sm_103 device is current. */
unsigned ssm_device_faults(void);

/* Self-test of the bounded waits (no counterpart in the pages): launches one
 * CTA that arms an mbarrier for a 16-byte copy that is never issued and waits
 * on it with at most poll_limit polls (1 <= poll_limit <= 2^20, else
 * SSM_ERR_SHAPE).  The wait gives up, the kernel returns, and the next
 * ssm_device_faults() reports bit 16 -- the path every kernel's waits take
 * when a copy does not arrive, without faulting or hanging the GPU. */
ssm_status ssm_selftest_bounded_wait(uint32_t poll_limit, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SSM_GB300_H */
