/*
 * ssm.h -- C ABI of libssm.so, the selective state-space (S6, "Mamba-1")
 * hot path on NVIDIA B300 (sm_103a).
 *
 * What the library computes (notation of the pages on the selective state
 * space model; b = batch index, d = channel, t = time step, n = state index):
 *
 *   delta_t = softplus(dt_t + bias_d)            (or dt_t + bias_d)
 *   Abar    = exp(delta_t * A[d,n])
 *   Bbar    = (exp(delta_t*A[d,n]) - 1)/A[d,n] * B[b,n,t]   zero-order hold
 *           = delta_t * B[b,n,t]                           simplified rule
 *   h[n]    = Abar * h[n] + Bbar * u_t                     (fp32 state)
 *   y_t     = sum_n C[b,n,t] h[n] + D[d] u_t
 *   out_t   = y_t * silu(z_t)                              (or y_t)
 *
 * Sources: "Mamba 模型" (gaos6e.github.io), the block flowchart's softplus,
 * discretise, selective-scan, readout and gate nodes and the decode section
 * ("为什么 Mamba 推理更省"); "Mamba 与状态空间模型" (world.lapla.si),
 * section 07 (fused on-chip scan, the (B,D,L,N) state never written out,
 * recompute in the backward) and section "模型省略了什么" (the simplified
 * Bbar = Delta*B); mhpn.cn section 3.1 (Bbar = (Abar - I) A^-1 B).
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library never allocates, frees or retains device memory.  Where an
 *    entry point needs scratch space it says so and the caller passes a
 *    workspace of at least the size the matching *_workspace_size() returns.
 *  - Calls are asynchronous on the given stream (NULL = legacy default
 *    stream).  Arguments are validated on the host before anything is
 *    launched; a failed validation launches nothing and returns a negative
 *    ssm_status.  Kernel launch errors are returned as SSM_ERR_CUDA.  The
 *    library never aborts, traps or exits.  ssm_last_error() gives a
 *    thread-local message for the last failure of the calling thread.
 *  - Sequence tensors are (batch, rows, seqlen) with the seqlen stride equal
 *    to 1; their batch and row strides are given in ELEMENTS.  Vectorised
 *    (16-byte) access is used when the base pointer and both strides keep
 *    every row 16-byte aligned; otherwise a slower scalar path runs.  No
 *    other layout is accepted.
 *  - Floating-point parameters (A, D, biases, weights) and recurrent states
 *    are float32.  Activations are float32 or bfloat16 (ssm_dtype).
 *  - Outputs are written, never accumulated into.
 */
#ifndef SSM_H
#define SSM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so that this header does not
 * need the CUDA headers. */
typedef struct CUstream_st* ssm_stream_t;

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = -1, /* a NULL required pointer, a negative size, ... */
    SSM_ERR_UNSUPPORTED = -2, /* a valid request this library does not implement */
    SSM_ERR_MISALIGNED = -3,  /* a pointer that must be aligned (workspace, checkpoints) is not */
    SSM_ERR_WORKSPACE = -4,   /* workspace missing or smaller than required */
    SSM_ERR_CUDA = -5,        /* a CUDA runtime error (see ssm_last_error) */
    SSM_ERR_TIMEOUT = -6      /* a bounded device-side wait gave up (ssm_device_status) */
} ssm_status;

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

/* Bbar rule: zero-order hold, or the simplified Bbar = delta * B. */
typedef enum { SSM_BBAR_ZOH = 0, SSM_BBAR_SIMPLE = 1 } ssm_bbar_mode;

/* Element strides of the two outer axes of a (batch, rows, seqlen) tensor. */
typedef struct {
    int64_t batch;
    int64_t row;
} ssm_strides;

/* ------------------------------------------------------------------------
 * Selective scan, forward (fused discretisation + recurrence + readout +
 * gate; the per-step state never leaves the chip).
 * "Mamba 模型", flowchart nodes softplus .. gate; world.lapla.si section 07.
 *
 *   u, delta, z, out : (batch, dim, seqlen)   in_dtype (out: out_dtype)
 *   B, C             : (batch, dstate, seqlen) in_dtype, shared by all d
 *   A                : (dim, dstate) float32, contiguous
 *   D, delta_bias    : (dim) float32 or NULL (= 0)
 *   z                : NULL = no gate
 *   h0               : (batch, dim, dstate) float32 contiguous or NULL (= 0)
 *   final_state      : (batch, dim, dstate) float32 contiguous or NULL
 *   checkpoints      : (batch, ceil(seqlen/K), ceil(dstate/2), dim, 2)
 *                      float32 contiguous, 16-byte aligned, or NULL; entry
 *                      [b, k, p, d, q] holds state 2p+q of channel (b, d)
 *                      before step k*K (k = 0: h0); the state pairs of
 *                      neighbouring channels are adjacent so that the kernels'
 *                      accesses coalesce (the partner of a last odd state is
 *                      0).  K = checkpoint_every must be a positive multiple
 *                      of 4 when checkpoints != NULL.
 *                      ssm_scan_bwd can take these instead of recomputing.
 * dstate: 1..64 (above 16 the state runs as groups of 16 states, one pass
 * each, the readout summed across them in an fp32 workspace buffer).  dim,
 * batch >= 1; seqlen >= 0 (seqlen 0 only copies h0
 * to final_state).
 * Workspace: ssm_scan_fwd_workspace_size() bytes (0 for many shapes; the
 * long-sequence schedule stores per-segment carries there).  Pointer
 * must be 256-byte aligned when the size is non-zero.
 * Accuracy: bfloat16 inputs use the SFU fast exponentials; float32
 * inputs use correctly-rounded-class library exp/expm1/log1p.  A value
 * A[d,n] == 0 is handled as the limit Bbar = delta * B. */
typedef struct {
    int64_t batch, dim, seqlen, dstate;
    ssm_dtype in_dtype;
    ssm_dtype out_dtype;
    int bbar_mode;      /* ssm_bbar_mode */
    int delta_softplus; /* 1: delta = softplus(dt + bias); 0: dt + bias */
    const void* u;     ssm_strides u_strides;
    const void* delta; ssm_strides delta_strides;
    const void* z;     ssm_strides z_strides;
    const void* B;     ssm_strides B_strides;
    const void* C;     ssm_strides C_strides;
    void* out;         ssm_strides out_strides;
    const float* A;
    const float* D;
    const float* delta_bias;
    const float* h0;
    float* final_state;
    float* checkpoints;
    int64_t checkpoint_every;
    /* B/C groups: channel d reads B, C of group d / (dim / ngroups); B is then
     * (batch, ngroups, dstate, L) with group stride B_group_stride elements
     * (C likewise).  0 or 1 = one group shared by all channels.  With more than
     * one group, dim / ngroups must be a multiple of 128. */
    int64_t ngroups;
    int64_t B_group_stride, C_group_stride;
} ssm_scan_fwd_params;

SSM_API size_t ssm_scan_fwd_workspace_size(const ssm_scan_fwd_params* p);
SSM_API ssm_status ssm_scan_fwd(const ssm_scan_fwd_params* p, void* workspace,
                        size_t workspace_bytes, ssm_stream_t stream);

/* Schedule override of ssm_scan_fwd, for tests and tuning: the same
 * computation with a forced schedule (results agree with ssm_scan_fwd up to
 * the order of floating-point sums).  This is not part of the method; it makes
 * every schedule reachable at any problem size.
 *   lanes_per_channel : 1, 2 or 4 lanes share a channel's states; 0 = automatic
 *   generic_path      : 1 = the register-prefetch path even where the cp.async
 *                       pipeline applies; 0 = automatic
 *   segments          : cut the sequence into this many segments (at least 256
 *                       steps each; fewer are used when the sequence is short),
 *                       scanned in parallel and joined by the carry pass; 0 =
 *                       automatic, 1 = one sequential pass
 *   warp_scan         : 1 = one warp per channel, the sequence in chunks of
 *                       32 x 16 steps whose lanes are joined by a warp-shuffle
 *                       associative scan (bf16 inputs, d_state <= 16, no
 *                       checkpoints, and under ZOH every A[d,n] != 0: a zero
 *                       there is not detected and gives undefined outputs);
 *                       the other fields are then ignored
 * Any other value returns SSM_ERR_INVALID_ARG.  The workspace size depends on
 * the schedule: query it with ssm_scan_fwd_scheduled_workspace_size. */
typedef struct {
    int lanes_per_channel;
    int generic_path;
    int64_t segments;
    int warp_scan;
} ssm_fwd_schedule;

SSM_API size_t ssm_scan_fwd_scheduled_workspace_size(const ssm_scan_fwd_params* p, const ssm_fwd_schedule* s);
SSM_API ssm_status ssm_scan_fwd_scheduled(const ssm_scan_fwd_params* p, const ssm_fwd_schedule* s,
                                          void* workspace, size_t workspace_bytes, ssm_stream_t stream);

/* ssm_scan_fwd for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point: it exists for callers that are
 * not allowed to call cudaMalloc, such as a plugin inside an inference
 * runtime that receives only its input and output buffers and must keep to
 * a memory plan fixed at load time (an allocation can also synchronise the
 * device), and that therefore cannot supply the workspace ssm_scan_fwd's
 * long-sequence schedule needs.
 * Same parameters, results and asynchrony as ssm_scan_fwd, but no workspace:
 * the scratch is a 4 MiB array built into the library, reserved on every GPU
 * that loads the library until the process exits.  The call allocates and
 * frees nothing.
 *  - A problem that needs more scratch than 4 MiB (ssm_scan_fwd_workspace_size
 *    tells) returns SSM_ERR_UNSUPPORTED and launches nothing.
 *  - All calls on a device share that array: calls that may overlap on the GPU
 *    (other streams, other host threads) race on it and must be ordered by
 *    the caller.  No part of the array needs clearing between calls.
 *  - The first call in each CUDA context looks up the array's device address
 *    (cudaGetSymbolAddress, with that context's device current) and keeps it
 *    under the context's unique id, so a context created later on the same
 *    device (for example after cudaDeviceReset) gets its own lookup.  Make the
 *    first call in a context before any stream capture there. */
SSM_API ssm_status ssm_scan_fwd_static_ws(const ssm_scan_fwd_params* p, ssm_stream_t stream);

/* ------------------------------------------------------------------------
 * Selective scan, backward, with recompute of h (the states are not stored by
 * the forward; they are recomputed on chip from checkpoints).
 * world.lapla.si section 07 ("训练时反向传播要用的中间状态不存，到时候重新算
 * 一遍"); deepseek.csdn.net section 3.2.3 C.  The pages give no gradient
 * formulas: these are the chain rule of the forward above for the loss
 * sum(dout * out) + sum(dfinal_state * final_state).
 *
 *   forward inputs   : as ssm_scan_fwd (same shapes, strides and flags)
 *   dout             : (batch, dim, seqlen) in_dtype
 *   dfinal_state     : (batch, dim, dstate) float32 or NULL (= 0)
 *   checkpoints      : the forward's checkpoints (16-byte aligned) with
 *                      checkpoint_every == 4, or NULL / another interval: the
 *                      backward then recomputes them into the workspace first
 *   du, ddelta, dz   : (batch, dim, seqlen) grad_dtype, strides as above;
 *                      ddelta is the gradient with respect to the delta INPUT
 *                      (before bias and softplus); dz required iff z != NULL
 *   dB, dC           : (batch, dstate, seqlen) float32 contiguous (summed over
 *                      the channels d)
 *   dA               : (dim, dstate) float32; dD, ddelta_bias: (dim) float32 or
 *                      NULL; dh0: (batch, dim, dstate) float32 or NULL
 * Workspace: ssm_scan_bwd_workspace_size() bytes, 256-byte aligned (per-CTA
 * partial sums, and recomputed checkpoints when none are passed).
 * Results are deterministic (fixed-order reductions, no atomics). */
typedef struct {
    int64_t batch, dim, seqlen, dstate;
    ssm_dtype in_dtype;
    ssm_dtype grad_dtype;
    int bbar_mode;
    int delta_softplus;
    const void* u;     ssm_strides u_strides;
    const void* delta; ssm_strides delta_strides;
    const void* z;     ssm_strides z_strides;
    const void* B;     ssm_strides B_strides;
    const void* C;     ssm_strides C_strides;
    const void* dout;  ssm_strides dout_strides;
    const float* A;
    const float* D;
    const float* delta_bias;
    const float* h0;
    const float* dfinal_state;
    const float* checkpoints;
    int64_t checkpoint_every;
    void* du;          ssm_strides du_strides;
    void* ddelta;      ssm_strides ddelta_strides;
    void* dz;          ssm_strides dz_strides;
    float* dB;
    float* dC;
    float* dA;
    float* dD;
    float* ddelta_bias;
    float* dh0;
    /* B/C groups: channel d reads B, C of group d / (dim / ngroups); B is then
     * (batch, ngroups, dstate, L) with group stride B_group_stride elements
     * (C likewise); dB, dC are then
     * (batch, ngroups, dstate, L), each group summed over its own channels.  0 or 1 = one group shared by all channels.  With more than
     * one group, dim / ngroups must be a multiple of 128. */
    int64_t ngroups;
    int64_t B_group_stride, C_group_stride;
} ssm_scan_bwd_params;

SSM_API size_t ssm_scan_bwd_workspace_size(const ssm_scan_bwd_params* p);
SSM_API ssm_status ssm_scan_bwd(const ssm_scan_bwd_params* p, void* workspace,
                        size_t workspace_bytes, ssm_stream_t stream);

/* ------------------------------------------------------------------------
 * Single-token decode step: state <- update(state, x_t), then readout and
 * gate for that token.  "Mamba 模型", section "为什么 Mamba 推理更省".
 *
 *   x, delta, z, out : (batch, dim), rows of length dim, batch stride in
 *                      elements (x_stride etc.), unit dim stride.  x is the
 *                      scan input u_t (the conv output).  z may be NULL.
 *   B, C             : (batch, dstate), batch stride in elements
 *   state            : (batch, dim, dstate) float32 contiguous, updated IN
 *                      PLACE
 *   A, D, delta_bias : as for ssm_scan_fwd
 * Memory-bound: reads and writes the state once. */
typedef struct {
    int64_t batch, dim, dstate;
    ssm_dtype in_dtype;
    ssm_dtype out_dtype;
    int bbar_mode;
    int delta_softplus;
    const void* x;     int64_t x_stride;
    const void* delta; int64_t delta_stride;
    const void* z;     int64_t z_stride;
    const void* B;     int64_t B_stride;
    const void* C;     int64_t C_stride;
    void* out;         int64_t out_stride;
    const float* A;
    const float* D;
    const float* delta_bias;
    float* state;
    /* B/C groups: channel d reads row d / (dim / ngroups) of group rows
     * B + b * B_stride + group * B_group_stride (C likewise); 0 or 1 = shared.
     * ngroups must divide dim. */
    int64_t ngroups;
    int64_t B_group_stride, C_group_stride;
} ssm_state_update_params;

SSM_API ssm_status ssm_state_update(const ssm_state_update_params* p, ssm_stream_t stream);

/* ------------------------------------------------------------------------
 * Causal depthwise conv1d + SiLU over a sequence.
 * "Mamba 模型" conv node Uc_t = sum_i W_i U_{t-i} (tap i = 0 is the current
 * token) and SiLU node; world.lapla.si section 03 (the short conv keeps the
 * last 4 inputs).
 *
 *   x, out     : (batch, dim, seqlen) dtype, strides as above
 *   weight     : (dim, width) float32 contiguous; weight[d,i] multiplies
 *                x[t-i].  (PyTorch's Conv1d stores the taps in the reverse
 *                order.)
 *   bias       : (dim) float32 or NULL
 *   state_in   : (batch, dim, width) dtype contiguous or NULL: the `width`
 *                inputs before t = 0, oldest first; NULL = zeros
 *   state_out  : (batch, dim, width) dtype contiguous or NULL: the last
 *                `width` inputs, oldest first (for a following decode)
 * width: 1..4.  Memory-bound: reads x once, writes out once. */
typedef struct {
    int64_t batch, dim, seqlen, width;
    ssm_dtype dtype;
    const void* x;  ssm_strides x_strides;
    void* out;      ssm_strides out_strides;
    const float* weight;
    const float* bias;
    const void* state_in;
    void* state_out;
} ssm_conv_params;

SSM_API ssm_status causal_conv1d_silu(const ssm_conv_params* p, ssm_stream_t stream);

/* Backward of causal_conv1d_silu for the loss sum(dout * out): the chain rule
 * of the conv and SiLU nodes of the "Mamba 模型" flowchart.
 *   x, weight, bias, state_in : as for causal_conv1d_silu (dtype of x)
 *   dout       : (batch, dim, seqlen) dtype, strides as x
 *   dx         : (batch, dim, seqlen) grad_dtype, strides dx_strides
 *   dweight    : (dim, width) float32, summed over batch and t
 *   dbias      : (dim) float32 or NULL
 *   dstate_in  : (batch, dim, width) float32 or NULL: gradient of state_in
 *                (zero where state_in is NULL)
 * Memory-bound: reads x and dout once, writes dx once.  dweight and dbias
 * are summed in a fixed order through per-block partials in the workspace
 * (causal_conv1d_silu_bwd_workspace_size bytes, 256-byte aligned), so the
 * result is bitwise reproducible. */
typedef struct {
    int64_t batch, dim, seqlen, width;
    ssm_dtype dtype;
    ssm_dtype grad_dtype;
    const void* x;     ssm_strides x_strides;
    const void* dout;  ssm_strides dout_strides;
    void* dx;          ssm_strides dx_strides;
    const float* weight;
    const float* bias;
    const void* state_in;
    float* dweight;
    float* dbias;
    float* dstate_in;
} ssm_conv_bwd_params;

SSM_API size_t causal_conv1d_silu_bwd_workspace_size(const ssm_conv_bwd_params* p);
SSM_API ssm_status causal_conv1d_silu_bwd(const ssm_conv_bwd_params* p, void* workspace, size_t workspace_bytes,
                                          ssm_stream_t stream);

/* One-token conv update: shift x_t into the window, then conv + SiLU.
 *   state : (batch, dim, width) dtype contiguous, oldest first, IN PLACE
 *   x,out : (batch, dim), batch stride in elements, unit dim stride */
typedef struct {
    int64_t batch, dim, width;
    ssm_dtype dtype;
    const void* x;  int64_t x_stride;
    void* out;      int64_t out_stride;
    const float* weight;
    const float* bias;
    void* state;
} ssm_conv_update_params;

SSM_API ssm_status causal_conv1d_silu_update(const ssm_conv_update_params* p, ssm_stream_t stream);

/* ------------------------------------------------------------------------
 * Fused single-token decode step: the conv update followed by the state
 * update, in one kernel.  "Mamba 模型" flowchart for one token (conv node,
 * SiLU, scan node, readout and gate) and its decode section "为什么 Mamba
 * 推理更省" (per token only the fixed-size conv window and state change).
 * The conv output xc_t = silu(sum_i weight[d,i] x_{t-i} + conv_bias[d]) is
 * the scan input u_t; it stays in registers (fp32), so the result equals
 * causal_conv1d_silu_update followed by ssm_state_update on an fp32 xc, and
 * it is valid when delta, B, C and z of the token do not depend on xc_t
 * (they are inputs here).
 *
 *   x                : (batch, dim) raw token input (before the conv), in_dtype
 *   conv_state       : (batch, dim, width) in_dtype contiguous, oldest first,
 *                      shifted IN PLACE; width 1..4
 *   conv_weight      : (dim, width) float32 contiguous, weight[d,i] multiplies
 *                      x_{t-i}; conv_bias: (dim) float32 or NULL
 *   delta, z, B, C, A, D, delta_bias, state, out : as for ssm_state_update
 *   xc_out           : (batch, dim) in_dtype or NULL: the conv output, if the
 *                      caller wants it
 * Memory-bound: reads and writes the state and the conv window once. */
typedef struct {
    int64_t batch, dim, dstate, width;
    ssm_dtype in_dtype;
    ssm_dtype out_dtype;
    int bbar_mode;
    int delta_softplus;
    const void* x;     int64_t x_stride;
    const void* delta; int64_t delta_stride;
    const void* z;     int64_t z_stride;
    const void* B;     int64_t B_stride;
    const void* C;     int64_t C_stride;
    void* out;         int64_t out_stride;
    void* xc_out;      int64_t xc_stride;
    void* conv_state;
    const float* conv_weight;
    const float* conv_bias;
    const float* A;
    const float* D;
    const float* delta_bias;
    float* state;
    /* B/C groups: channel d reads row d / (dim / ngroups) of group rows
     * B + b * B_stride + group * B_group_stride (C likewise); 0 or 1 = shared.
     * ngroups must divide dim. */
    int64_t ngroups;
    int64_t B_group_stride, C_group_stride;
} ssm_decode_step_params;

SSM_API ssm_status ssm_decode_step(const ssm_decode_step_params* p, ssm_stream_t stream);

/* ------------------------------------------------------------------------
 * Mamba-2 state-space-duality (SSD) layer, forward, by the chunked algorithm.
 * world.lapla.si section 09 ("Mamba-2：两种算法"): A is one number per head times
 * the identity; the layer is the product with a lower-triangular matrix whose
 * (i, j) entry is C_i . B_j times the decay between steps j and i, evaluated in
 * chunks -- matrix products inside a chunk, only the state passed between
 * chunks (pnsm.cn overview, section "Mamba-2：状态空间对偶性").  The input enters
 * scaled by the step size (Bbar = Delta B).  Per (b, head h), state H (N x P):
 *
 *   Delta_t = softplus(dt[b,t,h] + dt_bias[h])   (delta_softplus = 0: dt + dt_bias)
 *   H       = exp(Delta_t A[h]) H + Delta_t B_t x_t^T
 *   y_t     = C_t^T H + D[h] x_t
 *
 *   x      : (batch, seqlen, nheads, headdim) bf16, contiguous; headdim = 64
 *   dt     : (batch, seqlen, nheads) bf16, contiguous
 *   A      : (nheads) fp32, expected <= 0 (a decay); D, dt_bias: (nheads) fp32 or NULL
 *   B, C   : (batch, seqlen, ngroups, dstate) bf16, contiguous; head h reads
 *            group h / (nheads / ngroups); dstate in {16, 32, 64, 128}
 *   h0     : (batch, nheads, dstate, headdim) fp32 or NULL (zero state)
 *   final_state : same layout, written when not NULL
 *   out    : (batch, seqlen, nheads, headdim), out_dtype (bf16 or fp32), contiguous
 * x, B, C, out and final_state must be 16-byte aligned (SSM_ERR_MISALIGNED
 * otherwise).  Contractions run on the tensor cores (tcgen05) in bf16 with
 * fp32 accumulation, in chunks of 128 steps; the operands that are not inputs
 * (the decay-weighted C B^T, the decay-weighted x of the state update, the
 * copy of the fp32 state that multiplies C) are rounded to bf16 once, so an
 * output is within 2^-7 times the same layer evaluated on absolute values
 * (|x|, |B|, |C|, |D|, |h0|) and the final state within 2^-8 of it.  No
 * workspace; asynchronous on `stream`.  The kernel's waits are bounded: if one
 * gives up, the outputs are undefined and ssm_device_status reports
 * SSM_ERR_TIMEOUT. */
typedef struct {
    int64_t batch, seqlen, nheads, headdim, dstate, ngroups;
    const void* x;
    const void* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const float* dt_bias;
    int delta_softplus;
    ssm_dtype out_dtype;
    const float* h0;
    float* final_state;
    void* out;
} ssm_ssd_fwd_params;

SSM_API ssm_status ssm_ssd_fwd(const ssm_ssd_fwd_params* p, ssm_stream_t stream);

/* ------------------------------------------------------------------------
 * Mamba-2 SSD layer, backward: the gradients of
 *   loss = sum(dout * out) + sum(dfinal_state * final_state)
 * for the layer of ssm_ssd_fwd (same sections), through its chunked form.
 * Per chunk of 64 steps, with s the in-chunk prefix sums of Delta A, K = C B^T
 * masked by the decays exp(s_i - s_j) (j <= i), H the state entering the chunk
 * and G the adjoint of the state leaving it:
 *   dx_j = Delta_j (sum_i K[i][j] dy_i + exp(s_last - s_j) G^T B_j) + D dy_j,
 *   dC_i, dB_j from (dy_i . x_j) times the masked decays and Delta_j, plus
 *   exp(s_i) H dy_i and exp(s_last - s_j) Delta_j G x_j; the step sizes'
 *   gradient through the prefix sums s; and G of the previous chunk =
 *   exp(s_last) G + sum_i exp(s_i) C_i dy_i^T.
 *
 *   inputs : as ssm_ssd_fwd (x, dt, A, B, C, D, dt_bias, delta_softplus, h0),
 *            plus dout (batch, seqlen, nheads, headdim) bf16 contiguous and
 *            dfinal_state (batch, nheads, dstate, headdim) fp32 or NULL (zero)
 *   dx     : (batch, seqlen, nheads, headdim), grad_dtype (bf16 or fp32)
 *   ddt    : (batch, seqlen, nheads), grad_dtype (the gradient of dt itself,
 *            i.e. through the softplus when delta_softplus is set)
 *   dA     : (nheads) fp32
 *   dB, dC : (batch, seqlen, ngroups, dstate) fp32, summed over the heads of a group
 *   dD, ddt_bias : (nheads) fp32 or NULL (not computed); the gradients of D
 *            and dt_bias at the given values (a NULL D or dt_bias reads as zero)
 *   dh0    : (batch, nheads, dstate, headdim) fp32 or NULL
 * headdim = 64; dstate in {16, 32, 64, 128}; x, B, C, dout, dx, dB and dC
 * must be 16-byte aligned, h0, dfinal_state and dh0 too when given
 * (SSM_ERR_MISALIGNED otherwise).  Every contraction is a bf16 tensor-core MMA with fp32
 * accumulation; operands that are not inputs are split into a bf16 value and
 * a bf16 residual, so results keep about 16 significant bits.  Sums over
 * heads, batch and chunks are taken in a fixed order (bitwise reproducible).
 * The workspace (ssm_ssd_bwd_workspace_size bytes, 256-byte aligned, owned by
 * the caller) holds the states entering and the adjoints leaving every chunk
 * (each as a bf16 value and residual: 2 x batch nheads ceil(seqlen/64) dstate
 * 64 x 4 bytes), per-head dB
 * and dC (2 x batch seqlen nheads dstate x 4 bytes) and per-chunk partial sums.
 * Asynchronous on `stream`; no device-side waits. */
typedef struct {
    int64_t batch, seqlen, nheads, headdim, dstate, ngroups;
    const void* x;
    const void* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const float* dt_bias;
    int delta_softplus;
    const float* h0;
    const void* dout;
    const float* dfinal_state;
    ssm_dtype grad_dtype;
    void* dx;
    void* ddt;
    float* dA;
    float* dB;
    float* dC;
    float* dD;
    float* ddt_bias;
    float* dh0;
} ssm_ssd_bwd_params;

SSM_API size_t ssm_ssd_bwd_workspace_size(const ssm_ssd_bwd_params* p);
SSM_API ssm_status ssm_ssd_bwd(const ssm_ssd_bwd_params* p, void* workspace, size_t workspace_bytes,
                               ssm_stream_t stream);

/* ------------------------------------------------------------------------
 * Measured unit rates for the roofline (not part of the method): FP32 lanes
 * per SM per clock through scalar FMA and through packed f32x2 FMA, and SFU
 * 2^x results per SM per clock, each from a probe kernel of independent
 * dependency chains timed with the SM's cycle counter (so independent of the
 * clock).  Runs on the calling thread's current device, synchronously; each
 * output pointer (host memory) may be NULL to skip that probe.  Allocates
 * nothing (cycle counts return through a device array built into the
 * library).  SSM_ERR_CUDA if a launch fails. */
SSM_API ssm_status ssm_probe_unit_rates(double* fp32_lanes_per_sm_clock, double* f32x2_lanes_per_sm_clock,
                                        double* ex2_per_sm_clock);

/* ------------------------------------------------------------------------ */
/* Human-readable name of a status code (static string). */
/* ------------------------------------------------------------------------
 * Projections beside the scan, on the tensor cores: x_proj and dt_proj.
 * "Mamba 模型" (gaos6e.github.io) block flowchart: the conv output Xc_t feeds
 * the x_proj node, which produces dt_raw_t, B_t and C_t; dt_raw_t feeds the
 * dt_proj + softplus node, which produces delta_t.  Both are the same batched
 * product with a weight shared by every token:
 *
 *   out[b] (m x n) = W (m x k) X[b] (k x n)        (+ bias, optional softplus)
 *
 * with X[b] channel-major and its n tokens contiguous -- the layout of the
 * scan's inputs -- so x_proj (W = W_x, (R + 2N) x D; X = the conv output
 * (batch, D, L)) writes dt_raw, B and C as rows [0, R), [R, R+N), [R+N, R+2N)
 * of one (batch, R + 2N, L) tensor whose B and C rows the scan reads as
 * (batch, N, L) views, and dt_proj (W = W_dt, D x R; X = those dt_raw rows)
 * writes delta as (batch, D, L).
 *
 *   W    : bf16, row-major, row stride ldw elements (>= k)
 *   X    : bf16, (batch, k, n) with n contiguous; row stride ldx (>= n) and
 *          batch stride x_batch_stride, in elements
 *   out  : bf16, (batch, m, n) with n contiguous; row stride ldo (>= n),
 *          batch stride out_batch_stride
 *   bias : (m) float32 or NULL, added to every row of the product
 *   epilogue : 0 = the product (+ bias); 1 = softplus(product + bias)
 * W, X and out must be 16-byte aligned and every stride a multiple of 8
 * elements (SSM_ERR_MISALIGNED otherwise); batch <= 65535.  Products are bf16
 * x bf16 with fp32 accumulation (tcgen05), rounded to bf16 once.  No
 * workspace.  The kernel's waits are bounded: if one gives up, the call's
 * outputs are undefined and ssm_device_status reports SSM_ERR_TIMEOUT. */
typedef struct {
    int64_t batch, m, n, k;
    const void* W;
    int64_t ldw;
    const void* X;
    int64_t ldx, x_batch_stride;
    void* out;
    int64_t ldo, out_batch_stride;
    const float* bias;
    int epilogue;
} ssm_proj_params;

SSM_API ssm_status ssm_proj(const ssm_proj_params* p, ssm_stream_t stream);

/* Device-side status of the library's asynchronous kernels on the current
 * device: *status receives SSM_OK or the first error a kernel recorded (so far
 * only SSM_ERR_TIMEOUT, from a bounded wait that gave up); clear != 0 resets
 * it.  Synchronises with the device (it reads a device word). */
SSM_API ssm_status ssm_device_status(int* status, int clear);

SSM_API const char* ssm_status_string(ssm_status s);
/* Message describing the calling thread's last failure ("" if none). */
SSM_API const char* ssm_last_error(void);
/* Library ABI version, incremented on any incompatible change. */
SSM_API int ssm_abi_version(void);
/* Number of CUDA kernels this library has launched in the process so far
 * (all devices, all threads; a diagnostic for counting launches inside a
 * timed region). */
SSM_API uint64_t ssm_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* SSM_H */
