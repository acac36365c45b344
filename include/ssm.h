/*
 * ssm.h -- C ABI of libssm, the selective state space scan (Mamba S6) for
 * NVIDIA B300 (sm_103a).
 *
 * What the library computes. For every batch row b and channel d (d < dim),
 * with an N-wide diagonal state h (N = dstate) that starts at zero:
 *
 *     dt_t   = delta[b,t,d] (+ delta_bias[d])  (then softplus, if asked)
 *     Abar_t = exp(dt_t * A[d,:])                 -- N values
 *     h_t    = Abar_t * h_{t-1} + dt_t * B[b,t,:] * x[b,t,d]
 *     y_t    = sum_n C[b,t,n] * h_t[n]  + D[d] * x[b,t,d]
 *     out    = y_t * silu(z[b,t,d])                (when z is given)
 *
 * Sources (page title, section):
 *  - "State Space Models -- Mamba, S4, and Beyond", "Mamba (S6 -- Selective
 *    State Space)", method _selective_scan: the per-token discretization
 *    exp(delta * A) and delta * B, the recurrence, C . h and the D skip.
 *  - "Mamba: State Space Models Challenge Transformers", "Selective Scan
 *    Algorithm": the call selective_scan(x, delta, A, B, C, D), x [B, L, D],
 *    A [D, N], D [D]; "Mamba's Innovation: Selection": softplus on delta and
 *    the output gate y * silu(z).
 *  - "State-space models (Mamba, S4)", "The Convolution View" (h_0 = 0; y
 *    reads the updated state) and "Training vs Inference Modes" (the O(1)
 *    recurrent step of generation, ssm_state_update below).
 *  - "State Space Models and Mamba", "Mamba: Selective State Spaces"
 *    (Delta_t = softplus(Linear(x_t))).
 *
 * Entry points:
 *  - the scan: ssm_selective_scan_fwd (from h = 0), _from_state (from a given
 *    state), _static (library-owned scratch), _conv (the Mamba block's causal
 *    conv1d + SiLU fused in front), and the input stage alone,
 *    ssm_causal_conv1d_silu, with its gradients ssm_causal_conv1d_silu_bwd;
 *  - training: ssm_selective_scan_fwd_ckpt (saves states for the backward)
 *    and ssm_selective_scan_bwd (every gradient);
 *  - generation: ssm_state_update (one token on a cached state);
 *  - variants through dims->flags: SSM_FLAG_ZOH (exact zero-order-hold Bbar)
 *    and SSM_FLAG_BC_PER_CHANNEL (B, C [batch, seqlen, dim, dstate]);
 *  - sizes, plans and errors: ssm_scan_workspace_bytes, ssm_scan_plan,
 *    ssm_scan_checkpoint_bytes, ssm_scan_bwd_workspace_bytes,
 *    ssm_get_device_status, ssm_strerror, ssm_last_cuda_error, ssm_version;
 *  - Mamba-2's SSD layer: ssm_ssd_fwd (tensor cores), ssm_ssd_workspace_bytes,
 *    ssm_ssd_get_device_status;
 *  - tests of the failure path: ssm_debug_timeout_probe, _static.
 *
 * Conventions for every entry point:
 *  - All tensors are contiguous, row-major, in DEVICE memory, caller-owned.
 *    The library never allocates, frees or keeps pointers past a call.
 *  - I/O tensors (x, delta, z, B, C, out) are fp32 or bf16 (dims->io_dtype);
 *    A, D, delta_bias, final_state and state are always fp32. All arithmetic
 *    is fp32; bf16 outputs are rounded to nearest even.
 *  - Every device pointer must be 16-byte aligned, and dim must be a multiple
 *    of 8 for bf16 I/O and of 4 for fp32 I/O (128-bit accesses along d).
 *  - Calls only enqueue work on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and return; they never synchronize. Arguments are fully
 *    validated on the host before anything is enqueued; on error nothing is
 *    enqueued and a negative SSM_ERR_* code is returned.
 *  - `out` and `final_state` must not overlap any input (SSM_ERR_ALIAS).
 *  - Calls that share a workspace must not run concurrently.
 */
#ifndef LIBSSM_SSM_H
#define LIBSSM_SSM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so that the header needs no CUDA
 * include. */
struct CUstream_st;
typedef struct CUstream_st* ssm_stream_t;

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

/* Return codes. 0 is success; every error is negative. */
enum {
    SSM_OK = 0,
    SSM_ERR_NULL = -1,      /* a required pointer is NULL                         */
    SSM_ERR_DIMS = -2,      /* a size is negative, too large, or dstate unsupported */
    SSM_ERR_DTYPE = -3,     /* io_dtype is not SSM_F32 / SSM_BF16                 */
    SSM_ERR_ALIGN = -4,     /* pointer not 16-byte aligned, or dim not a multiple
                               of 8 (bf16) / 4 (fp32)                             */
    SSM_ERR_WORKSPACE = -5, /* workspace NULL or smaller than ssm_scan_workspace_bytes */
    SSM_ERR_CUDA = -6,      /* a CUDA launch or query failed (see ssm_last_cuda_error) */
    SSM_ERR_TIMEOUT = -7,   /* device side: a scan kernel's bounded wait for its
                               own TMA copy gave up (ssm_get_device_status)   */
    SSM_ERR_ALIAS = -8      /* an output overlaps an input                         */
};

/* Problem sizes and the caller-owned workspace.
 *   batch   : b >= 0
 *   seqlen  : L >= 0 (ignored by ssm_state_update)
 *   dim     : d_inner >= 0 (channels)
 *   dstate  : N, one of 1, 2, 4, 8, 16 (16 is the production size)
 *   io_dtype: ssm_dtype of x, delta, z, B, C, out
 *   workspace, workspace_bytes: device scratch for ssm_selective_scan_fwd (see
 *     ssm_scan_workspace_bytes: a 256-byte header with the status word, plus
 *     the chunk carries when the sequence is split); may be NULL only for
 *     empty problems. Must be zero-filled once before its first use; the
 *     library leaves it in a state that the next call accepts. Ignored by
 *     ssm_state_update. */
typedef struct {
    int64_t batch, seqlen, dim, dstate;
    int32_t io_dtype;
    int32_t chunk_len_hint; /* 0: library's choice; else tokens per L-chunk of the
                               scan (rounded up to a multiple of 32; the
                               workspace size follows it)                 */
    void* workspace;
    size_t workspace_bytes;
    int32_t tile_config_hint; /* 0: library's choice; 1..4: force tile configuration
                                 0..3 of the scan: 4, 2, 1 or 3 warps per CTA
                                 (32 channels per warp); dstate 16 only,
                                 other dstate always use configuration 0      */
    int32_t flags;            /* SSM_FLAG_* bits; 0 for the defaults          */
} ssm_dims;

/*
 * SSM_FLAG_ZOH -- the exact zero-order-hold input matrix instead of the first-
 * order dt * B: Bbar = A^-1 (e^{A dt} - 1) B = dt * phi(dt A) * B with phi(z) =
 * (e^z - 1) / z ("State-space models (Mamba, S4)", "From Continuous to
 * Discrete: The Key Step": the exact solution for an input held constant over
 * the step, and its flashcard Bbar = (A^-1 (e^{A Delta} - I)) B). Abar is the
 * same exp(dt A) either way. Taken by ssm_selective_scan_fwd,
 * ssm_selective_scan_fwd_from_state, ssm_selective_scan_fwd_static, the
 * training pair ssm_selective_scan_fwd_ckpt / ssm_selective_scan_bwd (dstate
 * 16, tile_config_hint 0 or 1; the backward then differentiates the exact hold:
 * e^{dt A} in dt and dt^2 phi'(dt A) in A) and ssm_state_update (any dstate);
 * the other entry points return SSM_ERR_DIMS when it is set. An unknown bit is
 * SSM_ERR_DIMS.
 */
#define SSM_FLAG_ZOH 1

/*
 * SSM_FLAG_BC_PER_CHANNEL -- B and C hold one row per channel: [batch, seqlen,
 * dim, dstate] instead of [batch, seqlen, dstate] shared by all channels (the
 * shape "Mamba: State Space Models Challenge Transformers", "Selective Scan
 * Algorithm" gives them in its docstring). Each channel then reads its own 2 *
 * dstate values per token and the scan is bound by HBM. Taken by
 * ssm_selective_scan_fwd, ssm_selective_scan_fwd_from_state,
 * ssm_selective_scan_fwd_static and the training pair
 * ssm_selective_scan_fwd_ckpt / ssm_selective_scan_bwd (whose dB and dC then
 * have B's shape) with dstate 16, tile_config_hint 0 or 1, and not together
 * with SSM_FLAG_ZOH; by ssm_state_update (any dstate, also with SSM_FLAG_ZOH),
 * whose B and C are then [batch, dim, dstate]; other entry points return
 * SSM_ERR_DIMS.
 */
#define SSM_FLAG_BC_PER_CHANNEL 2

/*
 * ssm_selective_scan_fwd -- the selective scan over a whole sequence.
 *
 *   x, delta, z, out : [batch, seqlen, dim]  io dtype (z may be NULL: no gate)
 *   A                : [dim, dstate] fp32 (any sign; < 0 for a stable scan)
 *   B, C             : [batch, seqlen, dstate] io dtype, shared by all channels
 *   D                : [dim] fp32, or NULL (no skip term)
 *   delta_bias       : [dim] fp32, or NULL; added to delta before softplus
 *   delta_softplus   : nonzero -> dt = softplus(delta + bias)
 *   final_state      : [batch, dim, dstate] fp32 state after the last token,
 *                      or NULL
 * The scan starts from h = 0. seqlen == 0 writes zeros to final_state.
 */
int ssm_selective_scan_fwd(const void* x, const void* delta, const float* A,
                           const void* B, const void* C, const float* D,
                           const void* z, const float* delta_bias, int delta_softplus,
                           void* out, float* final_state, const ssm_dims* dims,
                           ssm_stream_t stream);

/*
 * ssm_selective_scan_fwd_from_state -- the same scan started from a given
 * state instead of zero, so that a sequence can be continued: prefill a prompt
 * in several pieces, or hand a generation state back to the scan. The pages
 * write the recurrence from an arbitrary h_{t-1} ("State-space models (Mamba,
 * S4)", "Worked Example: 2D SSM Step" starts from h_0 != 0; "Training vs
 * Inference Modes" keeps h between tokens); the scan above is this call with
 * h0 = 0.
 *
 *   h0 : [batch, dim, dstate] fp32, the state before the first token; read
 *        only, must not overlap out or final_state (SSM_ERR_ALIAS)
 * Every other argument is as for ssm_selective_scan_fwd. seqlen == 0 copies
 * h0 to final_state. h0 == NULL with a non-empty problem is SSM_ERR_NULL.
 */
int ssm_selective_scan_fwd_from_state(const void* x, const void* delta, const float* A,
                                      const void* B, const void* C, const float* D,
                                      const void* z, const float* delta_bias,
                                      int delta_softplus, const float* h0, void* out,
                                      float* final_state, const ssm_dims* dims,
                                      ssm_stream_t stream);

/*
 * The Mamba block's input stage: a causal depthwise conv1d of width conv_k
 * followed by SiLU ("State Space Models -- Mamba, S4, and Beyond", "Mamba (S6
 * -- Selective State Space)", MambaBlock: Conv1d with kernel_size = d_conv,
 * groups = d_inner, padding = d_conv - 1, the output cut to seq_len, then
 * F.silu; "State-space models (Mamba, S4)", "The Mamba Architecture Block"
 * draws a Conv1D + SiLU step too). Conv1d is a cross-correlation, so with x = 0 before
 * the first token:
 *
 *     u[b,t,d] = silu(conv_b[d] + sum_{k < conv_k} conv_w[d,k] * x[b, t-conv_k+1+k, d])
 *
 *   x, u    : [batch, seqlen, dim] io dtype
 *   conv_w  : [dim, conv_k] fp32 (the depthwise weight [dim, 1, conv_k]
 *             without its middle axis); conv_k in 1 .. 4 (d_conv = 4 on the
 *             pages), else SSM_ERR_DIMS
 *   conv_b  : [dim] fp32 or NULL (no bias; the pages' block has bias=False)
 */

/*
 * ssm_causal_conv1d_silu -- the input stage alone: writes u. In the pages'
 * block x_proj forms delta, B and C from u, so u is needed in memory before
 * the scan; this is the call that makes it. u must not overlap x, conv_w or
 * conv_b (SSM_ERR_ALIAS; the op is not in-place). Only batch, seqlen, dim and
 * io_dtype of dims are read; dstate, the hints and the workspace are ignored.
 */
int ssm_causal_conv1d_silu(const void* x, const float* conv_w, const float* conv_b, int conv_k,
                           void* u, const ssm_dims* dims, ssm_stream_t stream);

/*
 * ssm_selective_scan_fwd_conv -- the scan of ssm_selective_scan_fwd with the
 * input stage fused in front: every x of the scan (the B * x input and the
 * D * x skip) is replaced by u computed on the fly from x, and u is never
 * written. Results equal ssm_causal_conv1d_silu followed by
 * ssm_selective_scan_fwd on u (up to the rounding of u to the io dtype, which
 * the fused call skips). For callers that form delta, B and C without u, or
 * that recompute u rather than keep it resident. Arguments are those of
 * ssm_selective_scan_fwd plus conv_w, conv_b and conv_k as above; with
 * dstate 16, tile_config_hint must be 0 or 1 (SSM_ERR_DIMS otherwise), and the
 * workspace is sized by ssm_scan_workspace_bytes as usual.
 */
int ssm_selective_scan_fwd_conv(const void* x, const float* conv_w, const float* conv_b,
                                int conv_k, const void* delta, const float* A, const void* B,
                                const void* C, const float* D, const void* z,
                                const float* delta_bias, int delta_softplus, void* out,
                                float* final_state, const ssm_dims* dims, ssm_stream_t stream);

/*
 * Training through the scan ("State-space models (Mamba, S4)", "Training vs
 * Inference Modes": training runs the scan over whole sequences and
 * backpropagates through it; "State Space Models -- Mamba, S4, and Beyond",
 * "Verification Checklist": gradients flow through the discretization).
 * dstate must be 16 and tile_config_hint 0 or 1 (SSM_ERR_DIMS otherwise).
 * dims->flags may hold SSM_FLAG_ZOH or SSM_FLAG_BC_PER_CHANNEL (not both); the
 * checkpointing forward and the backward of one step take the same flags.
 *
 * ssm_selective_scan_fwd_ckpt -- ssm_selective_scan_fwd_from_state (h0 may be
 * NULL for zero) that also saves the fp32 state before every 8th token:
 *   ckpt : [batch, ceil(seqlen / 8), dim, 16] fp32, ckpt[b, m, d, :] = the
 *          state before token 8m; ssm_scan_checkpoint_bytes(dims) bytes;
 *          an output (must not overlap anything else)
 * The backward recomputes the states in between from these.
 */
size_t ssm_scan_checkpoint_bytes(const ssm_dims* dims);
int ssm_selective_scan_fwd_ckpt(const void* x, const void* delta, const float* A, const void* B,
                                const void* C, const float* D, const void* z,
                                const float* delta_bias, int delta_softplus, const float* h0,
                                void* out, float* final_state, float* ckpt, const ssm_dims* dims,
                                ssm_stream_t stream);

/*
 * ssm_selective_scan_bwd -- gradients of the scan for a loss L(out,
 * final_state), given dout = dL/dout and optionally dfinal_state =
 * dL/dfinal_state. The forward's inputs are passed again, with the ckpt its
 * checkpointing call wrote (same sizes, dtypes, flags and h0):
 *   dout                : [batch, seqlen, dim] io dtype (read only)
 *   dfinal_state        : [batch, dim, 16] fp32 or NULL (zero)
 *   dx, ddelta          : [batch, seqlen, dim] io dtype; ddelta is the gradient
 *                         of the delta input (through softplus and the bias)
 *   dz                  : [batch, seqlen, dim] io dtype, given exactly when z is
 *                         (SSM_ERR_NULL otherwise)
 *   dB, dC              : [batch, seqlen, 16] io dtype (summed over channels);
 *                         [batch, seqlen, dim, 16] with SSM_FLAG_BC_PER_CHANNEL
 *                         (B and C of that shape too; nothing summed)
 *   dA                  : [dim, 16] fp32 (summed over batch rows and tokens)
 *   dD, ddelta_bias     : [dim] fp32 or NULL (not computed); defined whether or
 *                         not D / delta_bias were given (their gradient at zero)
 *   dh0                 : [batch, dim, 16] fp32 or NULL: dL/dh0
 * Every gradient is written, not accumulated. Outputs must not overlap inputs,
 * each other or the workspace (SSM_ERR_ALIAS). dims->workspace must hold
 * ssm_scan_bwd_workspace_bytes(dims) bytes (no initial contents needed). The
 * backward splits the sequence into L-chunks of its own (enough to fill the
 * device in one wave; dims->chunk_len_hint, when given, sets them as for the
 * forward); the checkpoints do not depend on the forward's chunks. The sums
 * over channels, rows and chunks are added in a fixed order: results do not
 * depend on scheduling (for a given chunk plan). seqlen == 0 zeroes dA, dD,
 * ddelta_bias and copies dfinal_state (or zero) to dh0.
 */
size_t ssm_scan_bwd_workspace_bytes(const ssm_dims* dims);
int ssm_selective_scan_bwd(const void* x, const void* delta, const float* A, const void* B,
                           const void* C, const float* D, const void* z, const float* delta_bias,
                           int delta_softplus, const float* ckpt, const void* dout,
                           const float* dfinal_state, void* dx, void* ddelta, float* dA, void* dB,
                           void* dC, float* dD, void* dz, float* ddelta_bias, float* dh0,
                           const ssm_dims* dims, ssm_stream_t stream);

/*
 * ssm_causal_conv1d_silu_bwd -- the gradients of the input stage
 * (ssm_causal_conv1d_silu) for a loss whose gradient with respect to its output
 * u is du; the chain rule on the stage's definition ("State Space Models --
 * Mamba, S4, and Beyond", "Mamba (S6 -- Selective State Space)", MambaBlock:
 * Conv1d of width d_conv, left padding d_conv - 1, then SiLU):
 *   dpre_t = du_t silu'(pre_t),  dx_s = sum_k w[k] dpre_{s+K-1-k},
 *   dconv_w[d,k] = sum_{b,t} dpre_t x_{t-K+1+k},  dconv_b[d] = sum_{b,t} dpre_t.
 *   x, du, dx : [batch, seqlen, dim] io dtype
 *   conv_w    : [dim, conv_k] fp32 (1 <= conv_k <= 4); conv_b [dim] fp32 or NULL
 *   dconv_w   : [dim, conv_k] fp32; dconv_b [dim] fp32 or NULL (not computed)
 * dims->workspace must hold ssm_causal_conv1d_silu_bwd_workspace_bytes(dims,
 * conv_k) bytes (no initial contents needed). The sums over rows and tokens
 * are added in a fixed order. Chained after ssm_selective_scan_bwd (du = the
 * scan's dx), it gives the gradients of the input stage followed by the scan.
 * Two launches on `stream`.
 */
size_t ssm_causal_conv1d_silu_bwd_workspace_bytes(const ssm_dims* dims, int conv_k);
int ssm_causal_conv1d_silu_bwd(const void* x, const float* conv_w, const float* conv_b,
                               int conv_k, const void* du, void* dx, float* dconv_w,
                               float* dconv_b, const ssm_dims* dims, ssm_stream_t stream);

/*
 * ssm_state_update -- one token of recurrent generation on a cached state
 * ("State-space models (Mamba, S4)", "Training vs Inference Modes"). Exactly
 * one step of the scan above, with the state updated in place:
 *
 *   state            : [batch, dim, dstate] fp32, read and overwritten
 *   x, delta, z, out : [batch, dim] io dtype (z may be NULL)
 *   B, C             : [batch, dstate] io dtype ([batch, dim, dstate] with
 *                      SSM_FLAG_BC_PER_CHANNEL in dims->flags)
 *   A, D, delta_bias, delta_softplus : as for the scan
 * dims->seqlen and the workspace fields are ignored.
 */
int ssm_state_update(float* state, const void* x, const void* delta, const float* A,
                     const void* B, const void* C, const float* D, const void* z,
                     const float* delta_bias, int delta_softplus, void* out,
                     const ssm_dims* dims, ssm_stream_t stream);

/*
 * ssm_ssd_fwd -- Mamba-2's SSD layer ("Mamba: State Space Models Challenge
 * Transformers", "Mamba-2: Improved Architecture": a multi-head structure, the
 * pages' sizes n_heads 8, d_head 64, d_state 128; "State Space Models and
 * Mamba", "Mamba 2 and Hybrid Architectures": the SSM as a structured matrix
 * multiplication). Per batch row b and head hd, with one scalar decay per head
 * and one step per token shared by the head's d_head channels:
 *
 *     dt_t = dt[b,t,hd] (+ dt_bias[hd])  (then softplus, if asked)
 *     h_t  = exp(dt_t A[hd]) h_{t-1} + dt_t x[b,t,hd,:] B[b,t,g,:]^T   (h: [P, N])
 *     y[b,t,hd,:] = h_t C[b,t,g,:] + D[hd] x[b,t,hd,:]
 *
 * where head hd reads group g = hd / (nheads / ngroups). Layouts (row-major):
 *   x, y            : [batch, seqlen, nheads, headdim] bf16
 *   dt              : [batch, seqlen, nheads] bf16
 *   A, D, dt_bias   : [nheads] fp32 (D, dt_bias may be NULL)
 *   B, C            : [batch, seqlen, ngroups, dstate] bf16
 *   h0, final_state : [batch, nheads, headdim, dstate] fp32 (h0 NULL = zero;
 *                     final_state may be NULL)
 * Supported: io_dtype SSM_BF16, headdim 64, dstate 128, ngroups dividing
 * nheads (SSM_ERR_DIMS / SSM_ERR_DTYPE otherwise). The products run on the
 * tensor cores with fp32 accumulation; operands the kernel forms itself are
 * carried as a bf16 pair (high part + remainder). dims->workspace must hold
 * ssm_ssd_workspace_bytes(dims) (256) bytes, zero-filled once: its first word
 * is the status word that ssm_ssd_get_device_status reads (SSM_ERR_TIMEOUT
 * when a bounded wait gave up). Pointers 16-byte aligned; y and final_state
 * must not overlap an input. Enqueues one kernel on `stream`.
 */
typedef struct {
    int64_t batch, seqlen, nheads, headdim, ngroups, dstate;
    int32_t io_dtype;
    int32_t flags;          /* 0 */
    void* workspace;
    size_t workspace_bytes;
} ssm_ssd_dims;

size_t ssm_ssd_workspace_bytes(const ssm_ssd_dims* dims);
int ssm_ssd_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                const float* D, const float* dt_bias, int dt_softplus, const float* h0,
                void* y, float* final_state, const ssm_ssd_dims* dims, ssm_stream_t stream);
/* Synchronizes `stream`, then reads and clears the status word of the SSD
 * workspace (as ssm_get_device_status does for the scan). */
int ssm_ssd_get_device_status(const ssm_ssd_dims* dims, ssm_stream_t stream);

/* Size of the library-owned scratch used by ssm_selective_scan_fwd_static. */
#define SSM_STATIC_SCRATCH_BYTES (16u << 20)

/*
 * ssm_selective_scan_fwd_static -- ssm_selective_scan_fwd for callers that
 * cannot allocate device memory. The pages have no counterpart: this entry
 * point is a library convenience, not part of the method.
 *
 * Who needs it: plain C hosts and plugins inside another runtime that are
 * handed only their inputs and outputs and have no allocator, and callers that
 * must not call cudaMalloc on the hot path (it can synchronize the device and
 * can fail under memory pressure at an arbitrary point).
 *
 * Arguments, layouts, validation and results are those of
 * ssm_selective_scan_fwd; dims->workspace and dims->workspace_bytes are
 * ignored. The scan's scratch is a fixed array of SSM_STATIC_SCRATCH_BYTES
 * (16 MiB) inside the library, which every GPU that loads the library holds
 * until the process exits. When ssm_scan_workspace_bytes(dims) exceeds that
 * size the call returns SSM_ERR_WORKSPACE and enqueues nothing (use
 * ssm_selective_scan_fwd with a workspace, or a larger chunk_len_hint, which
 * needs fewer carries). The call allocates nothing.
 *
 * Every call looks up the array's device address in the current context
 * (cudaGetSymbolAddress; nothing is cached, so a context torn down and
 * recreated is handled). The first call on a device may load the library's
 * device code into that context: make it before any stream capture. Every call
 * on a device shares the one array, which keeps the last call's contents
 * (nothing in it has to start at zero): calls that can overlap on the GPU --
 * on different streams, or from different host threads -- race on it and must
 * be serialized by the caller.
 *
 * Device-side failures: the array starts with the same status word a caller
 * workspace holds. A bounded wait inside a scan kernel that gives up sets it
 * (the call's outputs are then undefined); ssm_get_static_status reads and
 * clears it. ssm_get_device_status does not apply to this entry point.
 */
int ssm_selective_scan_fwd_static(const void* x, const void* delta, const float* A,
                                  const void* B, const void* C, const float* D,
                                  const void* z, const float* delta_bias, int delta_softplus,
                                  void* out, float* final_state, const ssm_dims* dims,
                                  ssm_stream_t stream);

/* Synchronizes `stream`, then reads the status word of the scratch of
 * ssm_selective_scan_fwd_static on the current device: SSM_OK, or
 * SSM_ERR_TIMEOUT when a bounded wait inside a scan kernel running on that
 * scratch gave up since the word was last read. Reading a nonzero word clears
 * it. Allocates nothing. */
int ssm_get_static_status(ssm_stream_t stream);

/* Bytes of workspace ssm_selective_scan_fwd needs for these sizes (256 when
 * the scan runs in one pass, 0 for empty problems). Depends only on batch,
 * seqlen, dim, dstate, io_dtype, chunk_len_hint, tile_config_hint and flags
 * (per-channel B, C are planned with more L-chunks) and, when chunk_len_hint
 * is 0, on the current device's multiprocessor count (148 when no device is
 * present); returns 0 for invalid sizes. */
size_t ssm_scan_workspace_bytes(const ssm_dims* dims);

/* Launch plan the scan will use for these sizes (for benchmarks and tests). */
typedef struct {
    int64_t chunk_len;      /* tokens per L-chunk                       */
    int64_t nchunks;        /* L-chunks per channel                     */
    int64_t channels_per_cta;
    int64_t ctas;           /* CTAs of the main (output) kernel         */
    int32_t kernels;        /* kernel launches per call                 */
    int32_t tile_config;    /* tile configuration id (0..3)             */
} ssm_plan;
int ssm_scan_plan(const ssm_dims* dims, ssm_plan* plan);

/*
 * ssm_debug_timeout_probe -- for tests of the failure path. Enqueues a one-CTA
 * kernel that waits, with the scan kernels' bounded mbarrier wait, on a barrier
 * nothing arrives on, gives up after max_polls probes (1 .. 2^24; each probe may
 * suspend the thread for a short, hardware-chosen time) and sets the status
 * word of `workspace` (at least 256 bytes, 16-byte aligned) as a scan kernel
 * whose copy never landed would. The next ssm_get_device_status on that
 * workspace returns SSM_ERR_TIMEOUT. Nothing faults or hangs; the context
 * stays usable.
 */
int ssm_debug_timeout_probe(void* workspace, size_t workspace_bytes, uint32_t max_polls,
                            ssm_stream_t stream);

/* The same probe aimed at the status word of the scratch of
 * ssm_selective_scan_fwd_static on the current device; the next
 * ssm_get_static_status returns SSM_ERR_TIMEOUT. */
int ssm_debug_timeout_probe_static(uint32_t max_polls, ssm_stream_t stream);

/* Synchronizes `stream`, then reads the device-side status word of the
 * workspace: SSM_OK, or SSM_ERR_TIMEOUT when a bounded wait inside a scan
 * kernel gave up since the word was last read (the affected outputs are then
 * undefined). The word is sticky across calls; reading a nonzero word clears
 * it. Returns SSM_OK for empty problems. */
int ssm_get_device_status(const ssm_dims* dims, ssm_stream_t stream);

/* Human-readable text for a return code (static storage). */
const char* ssm_strerror(int code);

/* The last CUDA error code (cudaError_t as int) seen by this thread, 0 if none. */
int ssm_last_cuda_error(void);

/* Library ABI version: (major << 16) | minor. */
int ssm_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LIBSSM_SSM_H */
