/*
 * ssm_scan.h -- C ABI of the B300 (sm_103a) Mamba-1 selective scan library
 * (libssmscan.so).
 *
 * Operation (Mamba SSM complete guide (youngju.dev), section 5, "complete Mamba
 * implementation": MambaBlock.ssm / selective_scan / forward). For every batch
 * row b, channel d and state n:
 *     dt_t  = softplus(delta[b,d,t] + delta_bias[d])     (or the raw sum when softplus == 0)
 *     h_t,n = exp(dt_t * A[d,n]) * h_{t-1,n} + dt_t * B[b,n,t] * u[b,d,t]
 *     y_t   = sum_n C[b,n,t] * h_t,n + D[d] * u[b,d,t]
 *     y_t  *= silu(z[b,d,t]) = z / (1 + exp(-z))          (only when z != NULL)
 * starting from h_{-1} = h0 (zero when h0 == NULL). The input matrix is the
 * simplified dt*B of the page's selective_scan (not the exact zero-order-hold
 * form of its section 2 "Discretization"). The d_state == 1 case is the
 * Scalar Mamba1 (SM1) page's closed form (aitrends.kr, section details);
 * one-token decode is the same recurrence applied once to a resident state.
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller. The library
 *     allocates no memory, never synchronises the device, and launches only on
 *     the caller's `stream` (a cudaStream_t passed as void*; NULL = legacy
 *     default stream).
 *   - Layouts are dense row-major, last index fastest:
 *       u, delta, z, y : (batch, dim, seqlen)    seqlen innermost
 *       B, C           : (batch, dstate, seqlen) seqlen innermost
 *       A              : (dim, dstate) fp32
 *       D, delta_bias  : (dim) fp32
 *       h0, h_last     : (batch, dim, dstate) fp32
 *   - in_dtype gives the dtype of u, delta, z, B, C; out_dtype the dtype of y.
 *     A, D, delta_bias and the state are always fp32; all arithmetic is fp32.
 *   - Optional pointers (D, z, delta_bias, h0, h_last) may be NULL. A required
 *     pointer may be NULL only when its tensor has no elements.
 *   - Argument errors are returned synchronously as a negative ssm_status and
 *     nothing is launched. Errors raised on the device (a look-back wait that ran
 *     out of its iteration budget) are written to the workspace status word and
 *     read back with ssm_query_status().
 *   - Sizes are int64. Any batch, dim and seqlen >= 0 are accepted (ragged
 *     seqlen included); supported dstate: 1, 2, 4, 8, 16.
 *   - Pointers must be aligned to their element size (SSM_ERR_ALIGN otherwise);
 *     16-byte aligned rows take the vectorised paths.
 */
#ifndef SSM_SCAN_H_
#define SSM_SCAN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSM_SCAN_ABI_VERSION 1

/* Exported entry points (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype_t;

typedef enum {
    SSM_OK = 0,
    SSM_ERR_NULL = -1,              /* a required pointer is NULL */
    SSM_ERR_DIM = -2,               /* a negative size, or sizes overflow int64 */
    SSM_ERR_DTYPE = -3,             /* in_dtype / out_dtype not an ssm_dtype_t */
    SSM_ERR_ALIGN = -4,             /* a pointer not aligned to its element size */
    SSM_ERR_WORKSPACE = -5,         /* workspace NULL or smaller than required */
    SSM_ERR_LAUNCH = -6,            /* the CUDA launch itself failed */
    SSM_ERR_LOOKBACK_TIMEOUT = -7,  /* device: a look-back wait exhausted its budget */
    SSM_ERR_UNSUPPORTED_N = -8,     /* dstate not in {1, 2, 4, 8, 16} */
    SSM_ERR_ALIAS = -9,             /* an output overlaps an input it must not */
    SSM_ERR_ALGO = -10,             /* unknown algorithm selector */
    SSM_ERR_SCRATCH_LIMIT = -11,    /* problem needs more than SSM_STATIC_SCRATCH_BYTES of scratch */
    SSM_ERR_WIDTH = -12,            /* conv width not in 1..4 */
    SSM_ERR_SHAPE = -13,            /* SSD: headdim not 64, dstate not 64/128 or
                                       nheads not a multiple of ngroups */
    SSM_ERR_WAIT_TIMEOUT = -14,     /* device: an SSD tensor-core wait exhausted its budget */
    SSM_ERR_ORDER = -15             /* traversal order not in 0..3, or rows * cols != seqlen */
} ssm_status_t;

/* Algorithm selectors for ssm_scan_fwd_algo. All compute the same result.
 *   SSM_ALGO_AUTO         : choose from the shape (what ssm_scan_fwd does).
 *   SSM_ALGO_THREAD       : one channel's state vector split over 1-4 lanes, each
 *                           lane walking time sequentially (large batch*dim).
 *   SSM_ALGO_WARPSCAN     : lanes own consecutive time steps; (a, b) affine pairs
 *                           composed by a warp-shuffle scan inside each chunk,
 *                           serial carry across chunks.
 *   SSM_ALGO_LOOKBACK     : WARPSCAN split along seqlen over many blocks, carries
 *                           joined by single-pass decoupled look-back (long
 *                           seqlen at small batch*dim). Needs a workspace. */
typedef enum {
    SSM_ALGO_AUTO = 0,
    SSM_ALGO_THREAD = 1,
    SSM_ALGO_WARPSCAN = 2,
    SSM_ALGO_LOOKBACK = 3
} ssm_algo_t;

/* ABI version of the loaded library (SSM_SCAN_ABI_VERSION at build time). */
SSM_API int ssm_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
SSM_API const char* ssm_status_string(int status);

/* Bytes of device workspace ssm_scan_fwd / ssm_scan_fwd_algo need for these
 * sizes under any algorithm (always >= 16 so that the status word fits). The
 * caller allocates it; the library zeroes what it uses, on `stream`, inside
 * each look-back or time-serial call. */
SSM_API size_t ssm_scan_workspace_size(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate);

/* Selective scan, forward (prefill). See the operation above.
 *   u, delta   : (batch, dim, seqlen), in_dtype           [required]
 *   A          : (dim, dstate) fp32                       [required]
 *   B, C       : (batch, dstate, seqlen), in_dtype        [required]
 *   D          : (dim) fp32 skip weight                   [optional]
 *   z          : (batch, dim, seqlen), in_dtype gate      [optional]
 *   delta_bias : (dim) fp32, added to delta               [optional]
 *   softplus   : nonzero applies softplus to delta + bias
 *   h0         : (batch, dim, dstate) fp32 initial state  [optional, zero]
 *   y          : (batch, dim, seqlen), out_dtype output   [required]
 *   h_last     : (batch, dim, dstate) fp32 final state    [optional]
 *   workspace  : device scratch of ssm_scan_workspace_size() bytes, 16-byte
 *                aligned; the look-back needs it (SSM_ERR_WORKSPACE without). The
 *                time-serial algorithm uses it when given (NULL is allowed): its
 *                CTAs then split the (channel group, time chunk) work evenly over
 *                the SMs and pass the state across each split through it; without
 *                it every CTA walks one channel group over the whole sequence.
 * y must not overlap any input; h_last may equal h0 (in-place resume). */
SSM_API int ssm_scan_fwd(const void* u, const void* delta, const float* A, const void* B,
                         const void* C, const float* D, const void* z, const float* delta_bias,
                         int softplus, const float* h0, void* y, float* h_last, int64_t batch,
                         int64_t dim, int64_t seqlen, int64_t dstate, int in_dtype, int out_dtype,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Same as ssm_scan_fwd with an explicit algorithm (ssm_algo_t). */
SSM_API int ssm_scan_fwd_algo(const void* u, const void* delta, const float* A, const void* B,
                              const void* C, const float* D, const void* z,
                              const float* delta_bias, int softplus, const float* h0, void* y,
                              float* h_last, int64_t batch, int64_t dim, int64_t seqlen,
                              int64_t dstate, int in_dtype, int out_dtype, void* workspace,
                              size_t workspace_bytes, int algo, void* stream);

/* d_state == 1 scalar scan (Scalar Mamba1 page, section details: with
 * L = cumprod(exp(dt*A)), h = L * (h0 + cumsum(dt*B*u / L)), y = h * C).
 * Shapes: A (dim), B and C (batch, seqlen), h0 and h_last (batch, dim); the
 * rest as ssm_scan_fwd. Computed by the recurrence, which equals the closed
 * form exactly in exact arithmetic and never divides by the cumulative product. */
SSM_API int ssm_scalar_scan_fwd(const void* u, const void* delta, const float* A, const void* B,
                                const void* C, const float* D, const void* z,
                                const float* delta_bias, int softplus, const float* h0, void* y,
                                float* h_last, int64_t batch, int64_t dim, int64_t seqlen,
                                int in_dtype, int out_dtype, void* workspace,
                                size_t workspace_bytes, void* stream);

/* One decode token, updating `state` in place (the per-step body of the same
 * recurrence; O(1) work and memory per token).
 *   state : (batch, dim, dstate) fp32, read and written   [required; 16-byte
 *           aligned when dstate >= 4]
 *   x, delta, z : (batch, dim), in_dtype                  [x, delta required]
 *   B, C  : (batch, dstate), in_dtype                     [required]
 *   A (dim, dstate), D (dim), delta_bias (dim) fp32       [A required]
 *   y     : (batch, dim), out_dtype                       [required]
 * y must not overlap state or any input. */
SSM_API int ssm_state_update(float* state, const void* x, const void* delta, const float* A,
                             const void* B, const void* C, const float* D, const void* z,
                             const float* delta_bias, int softplus, void* y, int64_t batch,
                             int64_t dim, int64_t dstate, int in_dtype, int out_dtype,
                             void* stream);

/* Bytes of device workspace ssm_scan_bwd needs: the state at every 8-step chunk
 * start, (batch, dim, ceil(seqlen/8), dstate) fp32. 0 for invalid sizes. */
SSM_API size_t ssm_scan_bwd_workspace_size(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate);

/* Backward of ssm_scan_fwd: the gradients of a loss l given dout = dl/d(y)
 * (the gated output) and dh_last = dl/d(h_last), by the chain rule through the
 * forward's steps in reverse time (the pages print no backward). With g =
 * dl/dh_t carried from the end:
 *   dy = dout silu(z),  dz = dout y silu'(z),  g += C_t dy,  dC_t += dy h_t,
 *   dD += dy u_t,  du_t = D dy + sum_n g dt B_t,
 *   d(dt) = sum_n g (h_{t-1} a A + B_t u_t),  dA += g h_{t-1} a dt,
 *   dB_t += g dt u_t,  ddelta_t = d(dt) softplus'(delta_t + bias),  dbias += ddelta_t,
 *   g *= a;  dh0 = g at t = 0.
 * Inputs as ssm_scan_fwd (same u, delta, A, B, C, D, z, delta_bias, softplus,
 * h0), plus
 *   dout    : (batch, dim, seqlen), dout_dtype                       [required]
 *   dh_last : (batch, dim, dstate) fp32                    [optional, zero]
 * Outputs (all overwritten):
 *   du, ddelta : (batch, dim, seqlen), in_dtype                     [required]
 *   dz         : (batch, dim, seqlen), in_dtype                     [required iff z]
 *   dA         : (dim, dstate) fp32 (summed over batch rows)        [required]
 *   dB, dC     : (batch, dstate, seqlen) fp32 (summed over channels) [required]
 *   dD, ddelta_bias : (dim) fp32                [dD required iff D; optional]
 *   dh0        : (batch, dim, dstate) fp32                          [optional]
 *   workspace  : ssm_scan_bwd_workspace_size() bytes, 16-byte aligned
 * The summed gradients are zeroed on `stream` and accumulated with atomic adds,
 * so their low bits vary between runs. Outputs overlap no input, the workspace
 * or each other. */
SSM_API int ssm_scan_bwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
                         const float* D, const void* z, const float* delta_bias, int softplus,
                         const float* h0, const void* dout, const float* dh_last, void* du, void* ddelta,
                         float* dA, float* dB, float* dC, float* dD, void* dz, float* ddelta_bias,
                         float* dh0, int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                         int in_dtype, int dout_dtype, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Causal depthwise conv1d (+ silu), the step that produces the scan's input u
 * in the Mamba block (Mamba SSM complete guide (youngju.dev), section 5,
 * "complete Mamba implementation": MambaBlock.__init__'s depthwise nn.Conv1d
 * with kernel d_conv = width and padding width - 1, and forward's trim to the
 * first seqlen outputs followed by silu). PyTorch's Conv1d is a cross-correlation
 * over the left-padded input, so with xp the input preceded by width-1 earlier
 * values:
 *     out[b,d,t] = silu( bias[d] + sum_{k<width} weight[d,k] * xp[b,d,t+k] )
 * (weight[d,width-1] multiplies x[b,d,t]; no silu when silu == 0).
 *   x              : (batch, dim, seqlen), in_dtype                [required]
 *   weight         : (dim, width) fp32, width in 1..4              [required]
 *   bias           : (dim) fp32                                    [optional]
 *   conv_state_in  : (batch, dim, width-1) fp32, the width-1 inputs before x,
 *                    oldest first                         [optional, zeros]
 *   conv_state_out : (batch, dim, width-1) fp32, receives the last width-1
 *                    entries of xp (what a following call or the decode update
 *                    continues from); may be conv_state_in itself  [optional]
 *   out            : (batch, dim, seqlen), out_dtype               [required]
 * out overlaps no input. Errors as ssm_scan_fwd, plus SSM_ERR_WIDTH. */
SSM_API int ssm_causal_conv1d_fwd(const void* x, const float* weight, const float* bias,
                                  const float* conv_state_in, float* conv_state_out, void* out,
                                  int64_t batch, int64_t dim, int64_t seqlen, int64_t width,
                                  int silu, int in_dtype, int out_dtype, void* stream);

/* One decode token of the same convolution, in place on the state:
 *     out[b,d] = silu( bias[d] + sum_{k<width-1} weight[d,k] * conv_state[b,d,k]
 *                      + weight[d,width-1] * x[b,d] )
 * then conv_state[b,d] drops its oldest entry and appends x[b,d].
 *   conv_state : (batch, dim, width-1) fp32, read and written  [required if width > 1]
 *   x          : (batch, dim), in_dtype                        [required]
 *   weight     : (dim, width) fp32; bias (dim) fp32 optional
 *   out        : (batch, dim), out_dtype                       [required]
 * out overlaps no input and not the state. */
SSM_API int ssm_causal_conv1d_update(float* conv_state, const void* x, const float* weight,
                                     const float* bias, void* out, int64_t batch, int64_t dim,
                                     int64_t width, int silu, int in_dtype, int out_dtype,
                                     void* stream);

/* The selective scan along another traversal of the sequence, and with the
 * exact zero-order-hold input matrix as an option.
 *
 * Traversal (Mamba SSM complete guide (youngju.dev), section 9, VMamba: an image
 * of rows x cols patches stored in raster order is scanned in four directions).
 * Step k = 0 .. seqlen-1 of the recurrence visits sequence position pos(k):
 *   SSM_ORDER_RASTER          (0)  pos(k) = k
 *   SSM_ORDER_REVERSE         (1)  pos(k) = seqlen - 1 - k
 *   SSM_ORDER_COLUMNS         (2)  pos(k) = (k % rows) * cols + k / rows
 *   SSM_ORDER_COLUMNS_REVERSE (3)  the column order of step seqlen - 1 - k
 * Every input is read at pos(k) and the step's output is written to y at pos(k),
 * so each direction's y is in raster order (rows and cols are used by orders 2
 * and 3 only, where rows * cols must equal seqlen). h0 is the state before the
 * first visited step, h_last the state after the last.
 * zoh != 0: the input matrix is the zero-order hold of the same guide's section
 * 2 ("Discretization"), (dt A)^-1 (exp(dt A) - 1) dt B = (exp(dt A) - 1) / A * B
 * per (d, n), and dt * B where A = 0; zoh == 0 gives ssm_scan_fwd's dt * B.
 * Tensors, layouts and the remaining arguments are those of ssm_scan_fwd (no
 * workspace: the warp-scan algorithm; ssm_scan_fwd_dir_ws below takes one).
 * Errors as ssm_scan_fwd, plus SSM_ERR_ORDER. */
typedef enum {
    SSM_ORDER_RASTER = 0,
    SSM_ORDER_REVERSE = 1,
    SSM_ORDER_COLUMNS = 2,
    SSM_ORDER_COLUMNS_REVERSE = 3
} ssm_order_t;

SSM_API int ssm_scan_fwd_dir(const void* u, const void* delta, const float* A, const void* B, const void* C,
                             const float* D, const void* z, const float* delta_bias, int softplus,
                             const float* h0, void* y, float* h_last, int64_t batch, int64_t dim,
                             int64_t seqlen, int64_t dstate, int order, int64_t rows, int64_t cols, int zoh,
                             int in_dtype, int out_dtype, void* stream);

/* Bytes of device workspace ssm_scan_fwd_dir_ws can use for these sizes and
 * dtypes, in any order (>= 16): the prefill's own workspace plus, for the column
 * orders, transposed copies of u, delta, z, B, C and y. */
SSM_API size_t ssm_scan_dir_workspace_size(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                           int in_dtype, int out_dtype);

/* ssm_scan_fwd_dir with a device workspace (16-byte aligned, workspace_bytes of
 * it; ssm_scan_dir_workspace_size() bytes enable everything; NULL allowed).
 * Without the exact-ZOH input matrix, when the prefill's plan for these sizes is
 * the time-serial scan, or the look-back and the workspace holds it:
 *   raster                the prefill's scan itself;
 *   reversed              the same kernels walking from the end (bf16 inputs with
 *                         16-byte aligned rows, dstate > 1: each bulk copy is
 *                         mirrored and each 8-step vector reversed);
 *   columns / reversed    the raster / reversed walk of the transposed image: u,
 *   columns               delta, z, B, C are transposed into the workspace, the
 *                         scan writes a transposed y there, which is transposed
 *                         back into y (the transposed rows keep length seqlen).
 * Every other case is ssm_scan_fwd_dir. Results agree with ssm_scan_fwd_dir to the
 * prefill's tolerance, not bit for bit. */
SSM_API int ssm_scan_fwd_dir_ws(const void* u, const void* delta, const float* A, const void* B,
                                const void* C, const float* D, const void* z, const float* delta_bias,
                                int softplus, const float* h0, void* y, float* h_last, int64_t batch,
                                int64_t dim, int64_t seqlen, int64_t dstate, int order, int64_t rows,
                                int64_t cols, int zoh, int in_dtype, int out_dtype, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Mamba-2 state-space-duality (SSD) scan on the tensor cores (Mamba SSM
 * complete guide (youngju.dev), section 6 "Mamba 2": a multi-head SSM with one
 * scalar A per head, computed by chunks -- matrix products inside a chunk, the
 * recurrence between chunks). For batch row b, head h of group g = h / (nheads /
 * ngroups), step t, head channel p < headdim and state n < dstate:
 *     dt_t     = softplus(dt[b,t,h] + dt_bias[h])           (raw sum when softplus == 0)
 *     H_t[p,n] = exp(dt_t * A[h]) * H_{t-1}[p,n] + dt_t * x[b,t,h,p] * B[b,t,g,n]
 *     y[b,t,h,p] = sum_n C[b,t,g,n] * H_t[p,n] + D[h] * x[b,t,h,p]
 *     y       *= silu(z[b,t,h,p])                            (only when z != NULL)
 * starting from H_{-1} = h0[b,h] (zero when h0 == NULL); h_last receives H at the
 * last step. Chunks of 128 steps; inside a chunk the four products (C B^T, the
 * decay-masked matrix times x, C times the incoming state, the state update)
 * run as tcgen05 bf16 MMAs with fp32 accumulators in tensor memory, the computed
 * operands split into bf16 high and low parts.
 *   x, z    : (batch, seqlen, nheads, headdim) bf16, headdim == 64  [z optional]
 *   dt      : (batch, seqlen, nheads) bf16                          [required]
 *   A       : (nheads) fp32 (negative for a decaying state)         [required]
 *   B, C    : (batch, seqlen, ngroups, dstate) bf16, dstate 64 or 128 [required]
 *   D, dt_bias : (nheads) fp32                                      [optional]
 *   h0, h_last : (batch, nheads, headdim, dstate) fp32; h_last may be h0 itself [optional]
 *   y       : (batch, seqlen, nheads, headdim), out_dtype (bf16 or fp32) [required]
 * in_dtype must be SSM_BF16 (SSM_ERR_DTYPE otherwise). x, z, y, B and C must be
 * 16-byte aligned (SSM_ERR_ALIGN); other shapes give SSM_ERR_SHAPE. y and h_last
 * overlap no input (except h_last == h0). A tensor-core wait that runs out of
 * its budget is recorded on the device and read with ssm_device_status(). */
SSM_API int ssm_ssd_scan_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                             const float* D, const void* z, const float* dt_bias, int softplus,
                             const float* h0, void* y, float* h_last, int64_t batch, int64_t seqlen,
                             int64_t nheads, int64_t headdim, int64_t ngroups, int64_t dstate,
                             int in_dtype, int out_dtype, void* stream);

/* ssm_ssd_scan_fwd with a device workspace (16-byte aligned, `workspace_bytes`
 * of it; ssm_ssd_workspace_size() bytes enable everything). When the batch *
 * nheads sequences do not fill whole rounds of the resident CTAs, the CTAs then
 * split the (sequence, 128-step chunk) work into equal runs, a multiple of the SM
 * count of them, each walking the head of one sequence, any whole sequences and
 * the tail of another, and pass the 64 x dstate state across each split through
 * the workspace (the library zeroes what it uses, on `stream`). Otherwise, or with
 * a NULL or smaller workspace, it is ssm_ssd_scan_fwd. A state hand-over wait
 * that runs out is recorded like the other waits (ssm_device_status). */
SSM_API int ssm_ssd_scan_fwd_ws(const void* x, const void* dt, const float* A, const void* B, const void* C,
                                const float* D, const void* z, const float* dt_bias, int softplus,
                                const float* h0, void* y, float* h_last, int64_t batch, int64_t seqlen,
                                int64_t nheads, int64_t headdim, int64_t ngroups, int64_t dstate,
                                int in_dtype, int out_dtype, void* workspace, size_t workspace_bytes,
                                void* stream);

/* Bytes of device workspace ssm_ssd_scan_fwd_ws uses for these sizes (>= 16). */
SSM_API size_t ssm_ssd_workspace_size(int64_t batch, int64_t nheads, int64_t dstate);

/* Chunk length (time steps) of ssm_ssd_scan_fwd. */
SSM_API int64_t ssm_ssd_chunk_len(void);

/* Synchronises `stream`, then returns SSM_ERR_WAIT_TIMEOUT if, since the last
 * clear, a launch recorded a wait that ran out of its budget -- an SSD
 * tensor-core or copy wait, a bulk-copy wait of the prefill kernels (the
 * d_state = 1 kernel's included), or the state hand-over wait of the
 * work-balanced time-serial kernel -- else SSM_OK
 * (SSM_ERR_LAUNCH if the read itself failed). clear != 0 resets the record. */
SSM_API int ssm_device_status(int clear, void* stream);

/* Test hook for the SSD kernel's failure paths (Mamba SSM complete guide, section 6:
 * the same chunked SSD computation as ssm_ssd_scan_fwd_ws, softplus on, no D, z,
 * dt_bias, h0 or h_last; bf16 x, dt, B, C and y). Every pipeline wait of the
 * launch polls its mbarrier at most `wait_limit` times, and a state hand-over wait
 * of the work-balanced launch polls its flag at most that many times (1 .. 2^31 - 1,
 * else SSM_ERR_DIM). withhold_arrive != 0: compute warp 0 skips its first "w o x
 * ready" arrival, so the control warp's wait for it runs out. drop_ticket >= 0 (with
 * a workspace, as ssm_ssd_scan_fwd_ws): that ticket of the work-balanced launch
 * withholds its state publication, so the next ticket's hand-over wait runs out.
 * Either way the kernel records the wait's source line, raises its abort flag, lets
 * the tensor core and the copies in flight finish, frees tensor memory and returns
 * (y is then unspecified). Returns the launch status; read the record with
 * ssm_device_status(). Nothing faults or hangs. */
SSM_API int ssm_test_ssd_wait_fault(const void* x, const void* dt, const float* A, const void* B,
                                    const void* C, void* y, int64_t batch, int64_t seqlen, int64_t nheads,
                                    int64_t ngroups, int64_t dstate, int64_t wait_limit,
                                    int withhold_arrive, void* workspace, size_t workspace_bytes,
                                    int64_t drop_ticket, void* stream);

/* Test hook for the state hand-over of the work-balanced time-serial scan (the
 * time-serial algorithm of ssm_scan_fwd_algo with a workspace; softplus on, no D,
 * z, bias, h0 or h_last; y in in_dtype): ticket `drop_ticket` withholds its state
 * publication, so the next ticket's wait runs out after `spin_limit` polls; the
 * kernel records it (ssm_device_status reports SSM_ERR_WAIT_TIMEOUT), continues
 * from a zero state and finishes (y is then unspecified). Returns the launch
 * status. */
SSM_API int ssm_test_serial_handover_timeout(const void* u, const void* delta, const float* A,
                                             const void* B, const void* C, void* y, int64_t batch,
                                             int64_t dim, int64_t seqlen, int64_t dstate, int in_dtype,
                                             void* workspace, size_t workspace_bytes,
                                             int64_t drop_ticket, uint32_t spin_limit, void* stream);

/* Test hook for the look-back error path. Runs the look-back scan (softplus on,
 * no D, z, bias or h0; y in in_dtype) with segment `drop_segment` withholding
 * its publication, so the waits of the next segment run out after `spin_limit`
 * polls: the kernel then records SSM_ERR_LOOKBACK_TIMEOUT in the workspace
 * status word and finishes (y is then unspecified). Returns the launch status;
 * read the device status with ssm_query_status(). */
SSM_API int ssm_test_lookback_timeout(const void* u, const void* delta, const float* A,
                                      const void* B, const void* C, void* y, int64_t batch,
                                      int64_t dim, int64_t seqlen, int64_t dstate, int in_dtype,
                                      void* workspace, size_t workspace_bytes,
                                      int64_t drop_segment, uint32_t spin_limit, void* stream);

/* Test hook for the device math behind the scan's softplus, decays and gate
 * (Mamba SSM complete guide, section 5: dt = softplus(dt_proj), dA = exp(dt A),
 * the silu(z) gate of the block's forward). Evaluates helper `fn` on n fp32
 * device values x, writing n fp32 device values y, on `stream`:
 *   SSM_MATH_EXP          exp(x), the accurate form (x <= 88)
 *   SSM_MATH_LOG1P01      log1p(x) for x in [0, 1] (the fitted polynomial)
 *   SSM_MATH_EXPM1        expm1(x), the accurate form (the fp32-input decays)
 *   SSM_MATH_SOFTPLUS     softplus(x), the accurate form (fp32 inputs)
 *   SSM_MATH_SILU         silu(x), the accurate form (fp32 inputs)
 *   SSM_MATH_SOFTPLUS_SFU softplus(x) through the SFU (bf16 inputs)
 *   SSM_MATH_SILU_SFU     silu(x) through the SFU (bf16 inputs)
 * Returns SSM_OK, SSM_ERR_ALGO for an unknown fn, SSM_ERR_NULL, SSM_ERR_DIM or
 * SSM_ERR_LAUNCH. */
enum {
    SSM_MATH_EXP = 0,
    SSM_MATH_LOG1P01 = 1,
    SSM_MATH_EXPM1 = 2,
    SSM_MATH_SOFTPLUS = 3,
    SSM_MATH_SILU = 4,
    SSM_MATH_SOFTPLUS_SFU = 5,
    SSM_MATH_SILU_SFU = 6
};
SSM_API int ssm_test_math(int fn, const float* x, float* y, int64_t n, void* stream);

/* Size of the library's own device scratch area used by
 * ssm_scan_fwd_lookback_static (4 MiB). */
#define SSM_STATIC_SCRATCH_BYTES ((size_t)4 << 20)

/* The look-back scan (SSM_ALGO_LOOKBACK of ssm_scan_fwd_algo) without a caller
 * workspace: the pages have no counterpart to this entry point; it exists for
 * callers that cannot allocate device memory or hand the library a workspace --
 * for instance a plugin or callback running inside a host application that owns
 * all device memory and exposes no allocator to it, or a latency-critical path
 * that must not call cudaMalloc, which can synchronise the device and stall
 * every other stream.
 *   Arguments and results are those of ssm_scan_fwd (the caller still passes the
 *   inputs and outputs as device pointers); the scratch is a 4 MiB device array
 *   owned by the library. The library allocates nothing: no cudaMalloc or
 *   cudaFree, no allocating library routine.
 *   Limit: sizes whose look-back scratch, ssm_scan_workspace_size(batch, dim,
 *   seqlen, dstate), exceeds SSM_STATIC_SCRATCH_BYTES return SSM_ERR_SCRATCH_LIMIT
 *   with nothing launched (at dstate 16 that is about 16,000 channel-segments:
 *   batch*dim = 1536 fits up to seqlen of about 20K; longer sequences need a
 *   caller workspace).
 *   Memory: every GPU that loads the library holds the 4 MiB array until the
 *   process exits.
 *   First call on a device: it looks up the array's device address on the
 *   current device (cudaGetSymbolAddress) and caches it, so make that first
 *   call before any stream capture.
 *   Sharing: all calls on a device use the same array, which keeps what the last
 *   call left there; each call zeroes the part it needs, on `stream`, before its
 *   kernel. Calls whose executions overlap on the GPU (issued on different
 *   streams with no ordering between them) race on the array and give undefined
 *   results: serialise them, e.g. on one stream.
 *   Device-side errors: the look-back waits stay bounded, but the status word
 *   lives in the library's array, so a wait that runs out of budget is not
 *   reported to the caller (the output is then unspecified); use ssm_scan_fwd_algo
 *   with a workspace when that report is needed. */
SSM_API int ssm_scan_fwd_lookback_static(const void* u, const void* delta, const float* A,
                                         const void* B, const void* C, const float* D,
                                         const void* z, const float* delta_bias, int softplus,
                                         const float* h0, void* y, float* h_last, int64_t batch,
                                         int64_t dim, int64_t seqlen, int64_t dstate,
                                         int in_dtype, int out_dtype, void* stream);

/* Reads the device status word of `workspace` (reset and written by a previous
 * look-back scan on the same stream; other algorithms leave it untouched),
 * synchronising `stream` to do so. Returns SSM_OK or the device-side error
 * (e.g. SSM_ERR_LOOKBACK_TIMEOUT); SSM_ERR_WORKSPACE when the workspace is
 * NULL or under 16 bytes. */
SSM_API int ssm_query_status(const void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H_ */
