/*
 * ssfwd.h - C ABI of libssfwd.so, the GB300 (sm_103a) Mamba-1 selective-scan
 * forward.
 *
 * The operation is the forward pass of `selective_scan_fn(u, delta, A, B, C,
 * D=None, z=None, delta_bias=None, delta_softplus=False,
 * return_last_state=False)`, whose operands and shapes are those of the page
 * "PaddleNLP Kernel 算子库：CUDA 与 Triton 双实现的高性能 NLP GPU 算子实战指南",
 * section 4.1 "CUDA 算子 selective_scan". That page names the operator but
 * prints no formula; the recurrence computed is the Mamba-1 selective scan
 * with an Euler input term, per (batch b, channel d, state n, step t):
 *
 *     dt    = softplus(delta[b,d,t] + delta_bias[d])   (plain sum if !delta_softplus)
 *     x[n]  = exp(dt * A[d,n]) * x[n] + dt * B[n,t] * u[b,d,t]
 *             (x = initial_state[b,d,n] before t = 0 when given, else 0)
 *     y     = sum_n C[n,t] * x[n] + D[d] * u[b,d,t]
 *     out   = y * silu(z[b,d,t])  if z is given, else y;  silu(v) = v / (1 + e^-v)
 *     last_state[b,d,n] = x[n] after the last step
 *
 * B[n,t]/C[n,t] is B[d,n] for fixed B/C, or B[b, d / (dim/ngroups), n, t] for
 * variable (grouped) B/C; the page's 3-D (batch, dstate, seqlen) form is
 * ngroups = 1. The state is carried in fp32.
 *
 * Conventions for every entry point:
 *   - All tensor pointers in ss_fwd_params are DEVICE pointers owned by the
 *     caller. The library allocates no memory, keeps no per-call global state,
 *     never synchronises, and is safe to call from several host threads.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Work is enqueued on it; results are ready when it is.
 *   - Validation happens before anything is enqueued: on any error status
 *     nothing was launched and no memory was touched.
 *   - Asynchronous device faults surface on the caller's next synchronisation
 *     with the stream, as for any CUDA launch.
 */
#ifndef SSFWD_H_
#define SSFWD_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SS_ABI_VERSION 5

/* Element types. u, delta, z and out share `in_dtype`. */
typedef enum ss_dtype { SS_F32 = 0, SS_F16 = 1, SS_BF16 = 2 } ss_dtype;

/* B/C forms (section 4.1: fixed (dim, dstate), or varying over the sequence as
 * (batch, groups, dstate, seqlen); (batch, dstate, seqlen) is groups = 1). */
typedef enum ss_bc_mode { SS_BC_FIXED = 0, SS_BC_VARIABLE = 1 } ss_bc_mode;

typedef enum ss_status {
  SS_OK = 0,
  SS_ERR_NULL = 1,         /* a required pointer is NULL                      */
  SS_ERR_SHAPE = 2,        /* negative size, dim % ngroups != 0, ...          */
  SS_ERR_DTYPE = 3,        /* unknown dtype or unsupported dtype combination  */
  SS_ERR_STRIDE = 4,       /* seqlen (or state, for fixed B/C / A) stride != 1, or a negative stride */
  SS_ERR_ALIGN = 5,        /* a pointer is not aligned to its element size    */
  SS_ERR_ALIAS = 6,        /* out or last_state overlaps an input or each other */
  SS_ERR_UNSUPPORTED = 7,  /* dstate > 64, or a feature this build lacks      */
  SS_ERR_CUDA = 8,         /* a CUDA runtime/driver call failed               */
  SS_ERR_INTERNAL = 9,     /* a device-side self-check tripped                */
  SS_ERR_VERSION = 10,     /* params->abi_version != SS_ABI_VERSION           */
  SS_ERR_SCRATCH = 11      /* ss_fwd_noalloc: needs more than SS_NOALLOC_MAX_SCRATCH; ss_bwd: workspace missing or too small */
} ss_status;

/*
 * Parameters of one forward call. Strides are in ELEMENTS of the tensor's own
 * type and may be any non-negative value (views are fine) except where a unit
 * stride is required.
 *
 *   u, delta, z, out   (batch, dim, seqlen), stride[2] (seqlen) must be 1.
 *                      dtype in_dtype. z may be NULL (no gating).
 *   A                  (dim, dstate) fp32, A_stride = {dim, state}; state stride 1.
 *   B, C  variable     (batch, ngroups, dstate, seqlen), dtype bc_dtype
 *                      (in_dtype or SS_F32); stride = {batch, group, state, seqlen},
 *                      seqlen stride 1.
 *         fixed        (dim, dstate) fp32; stride[0] = dim stride, stride[1]
 *                      must be 1, stride[2..3] ignored. ngroups is ignored.
 *   D, delta_bias      (dim,) fp32, contiguous; NULL = absent (treated as 0).
 *   out                written, in_dtype, rounded once to nearest-even.
 *   last_state         (batch, dim, dstate) fp32 with last_state_stride =
 *                      {batch, dim, state}, state stride 1; NULL = not returned.
 *                      For seqlen == 0 it is filled with zeros.
 *
 * Sizes: batch, dim, seqlen >= 0; 1 <= dstate <= 64. batch*dim*seqlen == 0 is
 * a no-op (except the zero fill of last_state when seqlen == 0).
 *
 * Memory touched: the call may read any byte between the first and the last
 * element of u, delta, z, B and C (the gaps of a strided layout included:
 * rows whose start is not 16-byte aligned are read as the aligned 16-byte
 * blocks that cover them); it writes only the elements of out and last_state.
 */
typedef struct ss_fwd_params {
  int32_t abi_version;      /* must be SS_ABI_VERSION */
  int32_t in_dtype;         /* ss_dtype */
  int32_t bc_dtype;         /* ss_dtype */
  int32_t bc_mode;          /* ss_bc_mode */
  int32_t delta_softplus;   /* nonzero: dt = softplus(delta + delta_bias) */
  int32_t reserved0;
  int64_t batch, dim, seqlen, dstate, ngroups;
  const void *u, *delta, *z, *B, *C;
  const float *A, *D, *delta_bias;
  void *out;
  float *last_state;
  int64_t u_stride[3], delta_stride[3], z_stride[3], out_stride[3];
  int64_t B_stride[4], C_stride[4];
  int64_t A_stride[2];
  int64_t last_state_stride[3];
  /* Optional device workspace (caller-owned, 16-byte aligned, not
   * overlapping any tensor). When the (batch, group, channel-tile) work units
   * cannot fill the GPU (few channels, long sequences), the forward splits the
   * sequence into segments and keeps per-segment state summaries here; size it
   * with ss_fwd_workspace_size. NULL / too small: the single-pass path runs
   * instead (same results up to fp32 rounding, fewer CTAs). */
  void *workspace;
  int64_t workspace_bytes;
  /* Optional start state (batch, dim, dstate) fp32 with stride {batch, dim,
   * state}, state stride 1; NULL = zero. It lets a call continue a sequence
   * from a previous call's last_state (the page's signature has none; it is
   * the chaining input of the decode step below). It may be the very buffer
   * passed as last_state with the same strides (each row is read before it is
   * written); any other overlap with an output is SS_ERR_ALIAS. */
  const float *initial_state;
  int64_t initial_state_stride[3];
  /* Optional caller-owned device int32 (4-byte aligned, not overlapping any
   * tensor or the workspace) that receives this call's device-side error
   * code; NULL = the library's per-device word read by ss_device_error. The
   * kernels only ever write a nonzero code into it, and only if it still
   * holds 0 (the first error wins), so the caller zeroes it before the call
   * and reads it after the stream completes. With a word of its own, each
   * caller (stream, thread) can tell whether its own launch gave up on a
   * bounded wait, which the shared word cannot show. */
  int32_t *error_word;
} ss_fwd_params;

/* SS_ABI_VERSION of the loaded library. */
int ss_abi_version(void);

/* Static, never-NULL description of a status code. */
const char *ss_status_string(int status);

/* Validate `p` without launching anything (no CUDA call is made). Returns the
 * status ss_fwd would return before launching. */
int ss_fwd_validate(const ss_fwd_params *p);

/* Bytes of `workspace` the fastest schedule of `p` uses on the current device
 * (0 if it uses none). Validates `p` like ss_fwd; makes a device-attribute
 * query (no allocation, no launch). */
int ss_fwd_workspace_size(const ss_fwd_params *p, int64_t *bytes);

/* The selective-scan forward on device buffers, enqueued on `stream`.
 * Returns SS_OK once enqueued, or an error status with nothing enqueued
 * (SS_ERR_CUDA if the launch itself failed). */
int ss_fwd(const ss_fwd_params *p, void *stream);

/*
 * The same forward for HOST data, with the host<->device copies enqueued on
 * the same stream: each non-NULL host input (`h_u`, `h_delta`, `h_z`, `h_B`,
 * `h_C`, `h_A`, `h_D`, `h_delta_bias`) is copied into the matching device
 * buffer of `p` (which must already exist and be laid out contiguously, as
 * the strides in `p` must then describe), the kernel runs, and `out` (and
 * `last_state` when `h_last_state` is non-NULL) are copied back into the host
 * buffers. Host buffers should be pinned for the copies to be asynchronous.
 * Nothing is synchronised: host outputs are valid once `stream` completes.
 * Copy sizes are the contiguous sizes of each tensor. Returns as ss_fwd.
 *
 * The copies overlap the work: the problem is cut into row blocks (whole
 * batch rows, or channel ranges of one batch row that keep groups whole), and
 * block i's inputs travel host-to-device while block i-1 runs and block i-2's
 * outputs travel back. The copies run on two streams internal to the library
 * (created with a few events on the first call on each device and kept until
 * the process exits), forked from `stream` by an event and joined back into
 * it, so the results still complete in `stream`'s order. All blocks share
 * p->workspace. On an error after the copies began, `stream` still waits for
 * the copies already issued.
 */
int ss_fwd_host(const ss_fwd_params *p,
                const void *h_u, const void *h_delta, const void *h_z,
                const void *h_B, const void *h_C,
                const float *h_A, const float *h_D, const float *h_delta_bias,
                void *h_out, float *h_last_state, void *stream);

/*
 * Allocation-free variant of ss_fwd, for callers that cannot allocate device
 * memory: for instance code running where device allocation is forbidden or
 * unavailable (an inference runtime that owns all device memory and hands
 * out only input/output buffers, or a plugin inside another framework's
 * allocator). It has no counterpart in the pages describing the operator; it
 * is the same forward, including the split-sequence schedule, with that
 * schedule's segment summaries kept in a static device buffer of
 * SS_NOALLOC_MAX_SCRATCH bytes that the library carries on every device
 * (held until the process exits) instead of a caller workspace.
 *
 *  - p->workspace / p->workspace_bytes are ignored: they are neither used
 *    nor validated (a stale pointer left there is harmless). Inputs and
 *    outputs are the caller's device buffers as for ss_fwd. Nothing is
 *    allocated: no cudaMalloc, cudaFree or allocating library call.
 *  - A problem whose schedule needs more scratch than the buffer holds is
 *    rejected with SS_ERR_SCRATCH before anything is enqueued (ss_fwd with a
 *    workspace handles it).
 *  - The first call on a device that passes validation, whatever its size
 *    (an empty problem will do), looks up the buffer's device address
 *    (cudaGetSymbolAddress) with that device current and caches it; later
 *    calls on that device make no such query. Make that first call before
 *    any stream capture on the device.
 *  - All calls share the one buffer and it keeps the previous call's
 *    contents. Each call writes every summary it later reads, so nothing needs
 *    clearing, but calls whose work overlaps on the GPU (e.g. concurrent
 *    streams) race on it: serialise them.
 */
#define SS_NOALLOC_MAX_SCRATCH (2 * 1024 * 1024)
int ss_fwd_noalloc(const ss_fwd_params *p, void *stream);

/*
 * One decode step of the same recurrence: section 4.4 of the page lists a
 * "selective_state_update" operator for the Mamba models but prints no
 * signature, so the operands are the scan's at a single time step. For every
 * (batch b, channel d, state n):
 *
 *     dt    = softplus(delta[b,d] + delta_bias[d])   (plain sum if !delta_softplus)
 *     state[b,d,n] = exp(dt * A[d,n]) * state[b,d,n] + dt * B[n] * u[b,d]
 *     out[b,d]     = (sum_n C[n] * state[b,d,n] + D[d] * u[b,d]) * silu(z[b,d])
 *
 * with B[n] = B[b, d / (dim/ngroups), n] (variable) or B[d, n] (fixed), and
 * no gate when z is NULL. The state is updated in place.
 *
 *   state              (batch, dim, dstate) fp32, stride {batch, dim, state},
 *                      state stride 1; read and written.
 *   u, delta, z, out   (batch, dim), in_dtype, stride {batch, dim}. z may be NULL.
 *   B, C  variable     (batch, ngroups, dstate), dtype bc_dtype (in_dtype or
 *                      SS_F32), stride {batch, group, state}, state stride 1.
 *         fixed        (dim, dstate) fp32, stride {dim, 1}; ngroups ignored.
 *   A                  (dim, dstate) fp32, state stride 1.
 *   D, delta_bias      (dim,) fp32 contiguous, or NULL (absent = 0).
 *
 * Sizes: batch, dim >= 0, 1 <= dstate <= 64; batch * dim == 0 is a no-op.
 * out must not overlap any input or the state, and the state must not
 * overlap any input (SS_ERR_ALIAS). Same conventions as ss_fwd otherwise
 * (device pointers, asynchronous on `stream`, nothing enqueued on error).
 */
typedef struct ss_state_update_params {
  int32_t abi_version;      /* must be SS_ABI_VERSION */
  int32_t in_dtype;         /* ss_dtype of u, delta, z, out */
  int32_t bc_dtype;         /* ss_dtype of B, C */
  int32_t bc_mode;          /* ss_bc_mode */
  int32_t delta_softplus;
  int32_t reserved0;
  int64_t batch, dim, dstate, ngroups;
  float *state;
  const void *u, *delta, *z, *B, *C;
  const float *A, *D, *delta_bias;
  void *out;
  int64_t state_stride[3];
  int64_t u_stride[2], delta_stride[2], z_stride[2], out_stride[2];
  int64_t B_stride[3], C_stride[3];
  int64_t A_stride[2];
} ss_state_update_params;

/* Validate without launching (no CUDA call). */
int ss_state_update_validate(const ss_state_update_params *p);

/* The decode step on device buffers, enqueued on `stream`. */
int ss_state_update(const ss_state_update_params *p, void *stream);

/*
 * Causal depthwise 1-D convolution, the `causal_conv1d_fn(x, weight, bias,
 * seq_idx, initial_states, return_final_states, final_states_out,
 * activation)` operator of the same page, section 4.2, which runs in front of
 * the scan in a Mamba block. The page gives the operands; the computation
 * taken is, per (batch b, channel d, step t) with kernel width W:
 *
 *     out[b,d,t] = act(bias[d] + sum_{k<W} weight[d,k] * x[b,d,t-(W-1)+k])
 *
 * where x at a position before 0 is initial_states[b,d,W-1+pos] (else 0), a
 * position whose seq_idx differs from step t's counts as 0 (packed
 * variable-length sequences), and act is the identity or silu (= swish,
 * v / (1 + e^-v)). final_states[b,d,k] = the last W-1 inputs of the row,
 * oldest first (initial states / zeros to the left of a short row).
 *
 *   x, out             (batch, dim, seqlen), dtype, seqlen stride 1.
 *   weight             (dim, width) fp32, width stride 1; 2 <= width <= 4.
 *   bias               (dim,) fp32 contiguous, or NULL.
 *   seq_idx            (batch, seqlen) int32, seqlen stride 1, or NULL; not
 *                      together with initial_states or final_states
 *                      (SS_ERR_UNSUPPORTED), as on the page.
 *   initial_states, final_states   (batch, dim, width-1) in dtype, or NULL.
 *   activation         SS_ACT_NONE or SS_ACT_SILU.
 * out and final_states must not overlap any input or each other.
 */
typedef enum ss_activation { SS_ACT_NONE = 0, SS_ACT_SILU = 1 } ss_activation;

typedef struct ss_conv1d_params {
  int32_t abi_version;      /* must be SS_ABI_VERSION */
  int32_t dtype;            /* ss_dtype of x, out and the states */
  int32_t activation;       /* ss_activation */
  int32_t reserved0;
  int64_t batch, dim, seqlen, width;
  const void *x;
  const float *weight, *bias;
  const int32_t *seq_idx;
  const void *initial_states;
  void *final_states;
  void *out;
  int64_t x_stride[3], out_stride[3], weight_stride[2], seq_idx_stride[2];
  int64_t initial_states_stride[3], final_states_stride[3];
} ss_conv1d_params;

int ss_causal_conv1d_validate(const ss_conv1d_params *p);
int ss_causal_conv1d(const ss_conv1d_params *p, void *stream);

/*
 * One decode step of the convolution (the page's causal_conv1d_update):
 * conv_state (batch, dim, width-1) holds the previous width-1 inputs, oldest
 * first; with x (batch, dim) the new input,
 *     out[b,d] = act(bias[d] + sum_{k<W-1} weight[d,k] conv_state[b,d,k] + weight[d,W-1] x[b,d])
 * and conv_state shifts left by one with x appended (in place). The page's
 * optional circular buffer (cache_seqlens) is not provided.
 */
typedef struct ss_conv1d_update_params {
  int32_t abi_version;
  int32_t dtype;            /* x, out, conv_state */
  int32_t activation;
  int32_t reserved0;
  int64_t batch, dim, width;
  const void *x;
  void *conv_state;
  const float *weight, *bias;
  void *out;
  int64_t x_stride[2], conv_state_stride[3], weight_stride[2], out_stride[2];
} ss_conv1d_update_params;

int ss_causal_conv1d_update_validate(const ss_conv1d_update_params *p);
int ss_causal_conv1d_update(const ss_conv1d_update_params *p, void *stream);

/*
 * Backward of ss_fwd. Section 4.1 of the page routes the backward of
 * selective_scan_fn to a CUDA kernel that returns the gradient of every input;
 * it prints no formula. Given dout, the gradient of a scalar loss with respect
 * to out, this computes the exact derivatives of sum(dout * out) for the
 * forward above (reverse-mode through the recurrence; lam = dL/dx):
 *
 *     dy_t   = dout_t silu(z_t)                 dz_t  = dout_t y_t silu'(z_t)
 *     lam_t  = dy_t C_t + exp(dt_{t+1} A) lam_{t+1}
 *     du_t   = dy_t D + sum_n lam_t dt_t B_t    dD   += dy_t u_t
 *     ddt_t  = sum_n lam_t (A exp(dt_t A) x_{t-1} + B_t u_t)
 *     ddelta_t = ddt_t sigmoid(delta_t + delta_bias)   (ddt_t without softplus)
 *     dA    += lam_t exp(dt_t A) x_{t-1} dt_t   dB_t += lam_t dt_t u_t
 *     dC_t  += dy_t x_t                         ddelta_bias += ddelta_t
 *     dinitial_state = exp(dt_0 A) lam_0
 *
 * with dA, dD, ddelta_bias and fixed dB/dC summed over batch and steps, and
 * variable dB/dC summed over the channels of each group. The states x_t are
 * recomputed from checkpoints kept in `workspace`; nothing from the forward
 * call is needed.
 *
 * Inputs (the forward's operands, same shapes, dtypes and stride rules as in
 * ss_fwd_params): u, delta, z, B, C, A, D, delta_bias, initial_state, and
 *   dout               (batch, dim, seqlen) in_dtype, seqlen stride 1.
 * Outputs (all written, never accumulated into; none may overlap an input,
 * the workspace or another output):
 *   du, ddelta         (batch, dim, seqlen) in_dtype, seqlen stride 1.
 *   dz                 same, required when z is given (ignored otherwise).
 *   dA                 (dim, dstate) fp32, contiguous.
 *   dB, dC             fp32, contiguous, in B/C's shape: (dim, dstate) for
 *                      fixed B/C, (batch, ngroups, dstate, seqlen) for variable.
 *   dD, ddelta_bias    (dim,) fp32 contiguous, or NULL = not wanted. An absent
 *                      D / delta_bias counts as 0, so its gradient is still
 *                      defined.
 *   dinitial_state     (batch, dim, dstate) fp32 contiguous, or NULL = not
 *                      wanted: the gradient of the start state (initial_state,
 *                      or the zero state when that is NULL).
 *   workspace          device memory of at least ss_bwd_workspace_size bytes,
 *                      16-byte aligned, caller-owned; contents need no
 *                      initialisation (SS_ERR_SCRATCH if too small or NULL).
 * dA, dB, dC, dD, ddelta_bias are reduced with fp32 atomic additions, so
 * their last bits may differ between runs. seqlen == 0 gives zero gradients.
 */
typedef struct ss_bwd_params {
  int32_t abi_version;      /* must be SS_ABI_VERSION */
  int32_t in_dtype;         /* ss_dtype of u, delta, z, dout, du, ddelta, dz */
  int32_t bc_dtype;         /* ss_dtype of B, C (outputs dB, dC are fp32) */
  int32_t bc_mode;          /* ss_bc_mode */
  int32_t delta_softplus;
  int32_t reserved0;
  int64_t batch, dim, seqlen, dstate, ngroups;
  const void *u, *delta, *z, *B, *C, *dout;
  const float *A, *D, *delta_bias, *initial_state;
  void *du, *ddelta, *dz;
  float *dA, *dB, *dC, *dD, *ddelta_bias, *dinitial_state;
  int64_t u_stride[3], delta_stride[3], z_stride[3], dout_stride[3];
  int64_t du_stride[3], ddelta_stride[3], dz_stride[3];
  int64_t B_stride[4], C_stride[4];
  int64_t A_stride[2];
  int64_t initial_state_stride[3];
  void *workspace;
  int64_t workspace_bytes;
} ss_bwd_params;

/* Validate without launching (no CUDA call; the workspace size is checked). */
int ss_bwd_validate(const ss_bwd_params *p);

/* Bytes of workspace ss_bwd needs for `p` (validated as by ss_bwd, except
 * for the workspace itself). */
int ss_bwd_workspace_size(const ss_bwd_params *p, int64_t *bytes);

/* The backward on device buffers, enqueued on `stream`. */
int ss_bwd(const ss_bwd_params *p, void *stream);

/*
 * Complex-A variant of ss_fwd. Section 4.1 of the page says that A (dim,
 * dstate) may be real or complex and gives B and C only their real shapes.
 * With complex A the state is complex and the real output takes the real part
 * of the contraction, per (batch b, channel d, state n, step t):
 *
 *     x[n] = exp(dt * A[d,n]) * x[n] + dt * B[n,t] * u[b,d,t]     (complex A, x)
 *     y    = Re(sum_n C[n,t] * x[n]) + D[d] * u[b,d,t]
 *     out  = y * silu(z[b,d,t])  if z is given, else y
 *
 * with dt, B, C, D, z and delta_bias as for ss_fwd (real).
 *
 * Layout as in ss_fwd_params, except:
 *   A                  (dim, dstate) complex64: interleaved (re, im) fp32
 *                      pairs, 8-byte aligned; A_stride in complex elements,
 *                      state stride 1.
 *   last_state         (batch, dim, dstate) complex64 interleaved, strides in
 *                      complex elements, state stride 1, 8-byte aligned; NULL =
 *                      not returned (zeros for seqlen == 0).
 *   initial_state      same layout, NULL = zero start; may be last_state itself
 *                      with the same strides.
 * Sizes: 1 <= dstate <= 64. Validation, errors and streams as for ss_fwd; no
 * workspace is used.
 */
typedef struct ss_fwd_complex_params {
  int32_t abi_version;      /* must be SS_ABI_VERSION */
  int32_t in_dtype;         /* ss_dtype of u, delta, z, out */
  int32_t bc_dtype;         /* ss_dtype of B, C */
  int32_t bc_mode;          /* ss_bc_mode */
  int32_t delta_softplus;
  int32_t reserved0;
  int64_t batch, dim, seqlen, dstate, ngroups;
  const void *u, *delta, *z, *B, *C;
  const float *A;           /* complex64, interleaved */
  const float *D, *delta_bias;
  void *out;
  float *last_state;        /* complex64, interleaved */
  const float *initial_state;
  int64_t u_stride[3], delta_stride[3], z_stride[3], out_stride[3];
  int64_t B_stride[4], C_stride[4];
  int64_t A_stride[2];
  int64_t last_state_stride[3], initial_state_stride[3];
} ss_fwd_complex_params;

int ss_fwd_complex_validate(const ss_fwd_complex_params *p);
int ss_fwd_complex(const ss_fwd_complex_params *p, void *stream);

/*
 * Device-side error word of the library on the current device (nonzero after
 * a kernel gave up on a bounded wait or tripped a self-check; 0 otherwise).
 * Reading it synchronises with the device. `clear` nonzero resets it to 0.
 * Returns SS_OK and writes the word into *out_word, or SS_ERR_CUDA.
 *
 * The word is shared by every call on the device that passes no error_word of
 * its own (ss_fwd_params.error_word), across streams and host threads, and is
 * sticky: it keeps the first code written until it is cleared here. A
 * nonzero value therefore says that SOME such call failed since the last
 * clear, not which one; give each call its own error_word to tell them apart.
 * An ss_fwd call that gave up on a wait still returned SS_OK when it was
 * enqueued (the failure happens later, on the device), so the word is the
 * only report of it.
 */
int ss_device_error(int32_t *out_word, int clear);

#ifdef __cplusplus
}
#endif

#endif /* SSFWD_H_ */
