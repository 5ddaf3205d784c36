/*
 * instant.h -- C ABI of the GB300 (sm_103a) low-rank linear-backward library.
 *
 * The library computes the per-step path and the calibration of INSTANT
 * low-rank backpropagation for one linear layer y = x w^T, as described on the
 * page "INSTANT: Compressing Gradients and Activations for Resource-Efficient
 * Training" (ICLR 2026 paper notes): sections 整体框架 (overall framework) and
 * 关键设计 1-3 (key designs 1-3).
 *
 * Notation (one sample b of a batch of B):
 *   x_b   [L, Cx]  layer input          g_y,b [L, Cy]  output gradient
 *   w     [Cy, Cx] weight                P [Rx, L], Q [Ry, L] projectors
 *   PQ    [Rx+Ry, L]  = [P; Q] stacked row-wise (P rows first)
 *
 * Conventions shared by every entry point
 *   - Every tensor argument is a DEVICE pointer to caller-owned memory,
 *     row-major and contiguous, unless the argument says "host".  The library
 *     never allocates or frees device memory; scratch comes from `ws`.
 *   - Device pointers must be 16-byte aligned, and for INSTANT_BF16 the
 *     innermost extent of every 2-D/3-D operand read by TMA (L for PQ/P/Q is
 *     exempt) must be a multiple of 8 elements; otherwise INSTANT_ERR_ALIGN.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on that stream except instant_calib_solve,
 *     instant_calib_solve_batch, instant_reconstruction_error and
 *     instant_device_status, which synchronise it.
 *   - Argument, shape and dtype errors are reported before anything is
 *     launched; nothing is written in that case.  A launch error returns
 *     INSTANT_ERR_CUDA.  Kernels never trap: a device-side wait that runs out
 *     of time sets a sticky device status that instant_device_status reads.
 *   - dtype INSTANT_BF16: bf16 inputs and outputs, fp32 accumulation
 *     (tcgen05 tensor cores).  INSTANT_F32: fp32 everywhere, plain FFMA (no
 *     TF32), intended for small problems.
 */
#ifndef INSTANT_H_
#define INSTANT_H_

#include <stddef.h>

#if defined(__GNUC__)
#pragma GCC visibility push(default) /* the library exports exactly these names */
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  INSTANT_OK = 0,
  INSTANT_ERR_ARG = 1,           /* null pointer or bad scalar argument          */
  INSTANT_ERR_SHAPE = 2,         /* unsupported or inconsistent extent           */
  INSTANT_ERR_DTYPE = 3,         /* unknown dtype                                */
  INSTANT_ERR_ALIGN = 4,         /* pointer or row pitch not 16-byte aligned     */
  INSTANT_ERR_WORKSPACE = 5,     /* workspace missing or too small               */
  INSTANT_ERR_CUDA = 6,          /* CUDA runtime / launch error                  */
  INSTANT_ERR_NOT_CONVERGED = 7, /* eigensolver hit its iteration cap            */
  INSTANT_ERR_NONFINITE = 8,     /* autocorrelation has no finite positive energy*/
  INSTANT_ERR_DEVICE = 9         /* a device-side wait ran out of time           */
} instant_status;

typedef enum { INSTANT_F32 = 0, INSTANT_BF16 = 1 } instant_dtype;

/* Calibration parameters (关键设计 2). */
typedef struct {
  double eps;       /* energy threshold epsilon (the page fixes 0.95)            */
  int p;            /* oversampling p: R = min(k + p, L)                         */
  int r_override;   /* > 0: output exactly this many rows (k is still reported)  */
  int scale_on;     /* 1: rows scaled by (sum_{i<=R} sigma_i^2)^(-1/2); 0: off   */
  int max_iter;     /* subspace-iteration cap; 0 selects 300                     */
  double tol;       /* Ritz residual tolerance relative to sigma_1; 0 selects 2e-5 */
  int warm_start;   /* 1: rows_out already holds a projector of this statistic   */
                    /* (e.g. the previous calibration); its rows seed the solve  */
} instant_calib_params;

/*
 * Activation compression x_hat_b = P x_b (整体框架: the forward stores
 * x_hat = P x instead of x).
 *   x     [B, L, Cx]  dtype dt (read)
 *   P     [Rx, L]     dtype dt (read)
 *   xhat  [B, Rx, Cx] dtype dt (written)
 * Limits: 1 <= Rx <= 64.
 */
instant_status instant_compress_act(const void* x, const void* P, void* xhat,
                                    int B, int L, int Cx, int Rx,
                                    instant_dtype dt, void* stream);

/*
 * The layer's forward with the stored activation computed on the way
 * (整体框架: the forward product y = x w^T is unchanged, and the layer keeps
 * x_hat = P x for its backward instead of x):
 *   y_b = x_b w^T,   x_hat_b = P x_b   (P may be NULL with Rx = 0: y only)
 *   x     [B, L, Cx]  dtype dt (read)      w  [Cy, Cx] dtype dt (read)
 *   P     [Rx, L]     dtype dt (read)      y  [B, L, Cy] dtype dt (written)
 *   xhat  [B, Rx, Cx] dtype dt (written)
 *   ws    device scratch of instant_forward_workspace_bytes(B, L, Cx, Rx, dt)
 *         bytes, ZEROED by the caller before its first use; every call leaves
 *         it zero again (fp32 partial sums of x_hat and per-sample counters),
 *         so one workspace serves every later call.  Calls that share a
 *         workspace must not overlap in time.
 * bf16: a persistent tcgen05 GEMM (128 x 192 tiles, fp32 accumulation, bf16
 * y); where L % 128 == 0, Cx % 128 == 0 and Rx <= 32, the tiles of the first column strip
 * also contract the x tiles they have staged with P, so x is read from HBM
 * once for both products; otherwise x_hat comes from instant_compress_act's
 * kernel after the GEMM (two launches).  x_hat is formed in fp32 and rounded
 * once to bf16, as by instant_compress_act.  f32: plain FFMA kernels.
 * Limits: 0 <= Rx <= 64; bf16 rows 16-byte aligned (Cx, Cy multiples of 8).
 */
instant_status instant_forward(const void* x, const void* w, const void* P, void* y, void* xhat,
                               void* ws, size_t ws_bytes, int B, int L, int Cx, int Cy, int Rx,
                               instant_dtype dt, void* stream);
size_t instant_forward_workspace_bytes(int B, int L, int Cx, int Rx, instant_dtype dt);

/*
 * Gradient projection with one read of g_y (关键设计 3):
 *   Sx_b = P g_y,b  (so g_hat_y1,b = Sx_b^T)    Sq_b = Q g_y,b  (g_hat_y2,b)
 *   gy  [B, L, Cy]      dtype dt (read)
 *   PQ  [Rx+Ry, L]      dtype dt (read), P rows then Q rows
 *   Sx  [B*Rx, Cy]      dtype dt (written), row b*Rx + r
 *   Sq  [B*Ry, Cy]      dtype dt (written), row b*Ry + r
 * Limits: 1 <= Rx, Ry and Rx + Ry <= 128.
 */
instant_status instant_project_grad(const void* gy, const void* PQ, void* Sx, void* Sq,
                                    int B, int L, int Cy, int Rx, int Ry,
                                    instant_dtype dt, void* stream);

/*
 * Weight gradient g_w = sum_b Sx_b^T x_hat_b = Sx^T x_hat (关键设计 3:
 * g_w ~ g_hat_y1 x_hat), contraction over K = B*Rx.
 *   Sx    [B*Rx, Cy]  dtype dt (read)
 *   xhat  [B*Rx, Cx]  dtype dt (read; the [B, Rx, Cx] output of compress_act)
 *   gw    [Cy, Cx]    fp32 (written, or accumulated into when accumulate != 0)
 */
instant_status instant_grad_w(const void* Sx, const void* xhat, float* gw, int accumulate,
                              int B, int Rx, int Cx, int Cy,
                              instant_dtype dt, void* stream);

/*
 * Input gradient g_tilde_x,b = Q^T (Sq_b w) (关键设计 3: g_hat_x = g_hat_y2 w,
 * g_tilde_x = Q^T g_hat_x).
 *   Sq  [B*Ry, Cy]  dtype dt (read)
 *   w   [Cy, Cx]    dtype dt (read)
 *   Q   [Ry, L]     dtype dt (read)
 *   gx  [B, L, Cx]  dtype dt (written)
 *   ws  device scratch of at least instant_grad_x_workspace_bytes(...) bytes
 *       (may be NULL when that size is 0).  Contents are overwritten.
 * Limits: 1 <= Ry <= 64.
 */
instant_status instant_grad_x(const void* Sq, const void* w, const void* Q, void* gx,
                              void* ws, size_t ws_bytes,
                              int B, int L, int Cx, int Cy, int Ry,
                              instant_dtype dt, void* stream);

size_t instant_grad_x_workspace_bytes(int B, int L, int Cx, int Cy, int Ry, instant_dtype dt);

/*
 * Both products of the low-rank backward (关键设计 3: g_w ~ g_hat_y1 x_hat and
 * g_tilde_x = Q^T g_hat_y2 w) in one call: the same products as
 * instant_grad_w(Sx, xhat, gw, accumulate, ...) followed by
 * instant_grad_x(Sq, w, Q, gx, ws, ...) (g_w may differ in the order of its
 * fp32 additions), with the same arguments, layouts and limits.  Where the
 * single-kernel input gradient applies (bf16, short Cy, and at most 64 MiB of
 * g_tilde_x when L >= 128) the weight-gradient tiles run inside the same
 * launch, on the SMs the input gradient leaves free; otherwise the two calls
 * are made in turn.
 */
instant_status instant_grad_w_x(const void* Sx, const void* xhat, float* gw, int accumulate,
                                const void* Sq, const void* w, const void* Q, void* gx,
                                void* ws, size_t ws_bytes,
                                int B, int L, int Cx, int Cy, int Rx, int Ry,
                                instant_dtype dt, void* stream);

/*
 * The layer's whole low-rank backward in one call (关键设计 3): the same
 * results, bit for bit, as instant_project_grad(gy, PQ, Sx, Sq, ...) followed
 * by instant_grad_w_x(Sx, xhat, gw, accumulate, Sq, w, Q = rows Rx.. of PQ,
 * gx, ...), which is what it runs.  With the environment variable
 * INSTANT_ONE_LAUNCH_BACKWARD set, and where the single-kernel input gradient
 * applies (bf16, short Cy, and at most 64 MiB of g_tilde_x when L >= 128), it
 * is ONE launch instead: clusters take tickets as they start; the first
 * tickets project (sample, 128-column) tiles of g_y and signal each finished
 * tile through counters in `ws`, the input-gradient
 * items of a sample group wait for their group's tiles and the
 * weight-gradient tiles for all of them (a consumer only waits for smaller
 * tickets, so the waits end whatever the scheduling).  That launch measured
 * slower than the two on a BERT-base block, hence opt-in.
 *   gy    [B, L, Cy]     dtype dt (read)
 *   PQ    [Rx+Ry, L]     dtype dt (read)
 *   xhat  [B, Rx, Cx]    dtype dt (read)
 *   w     [Cy, Cx]       dtype dt (read)
 *   Sx    [B*Rx, Cy], Sq [B*Ry, Cy]  dtype dt (written: the projections)
 *   gw    [Cy, Cx]       fp32 (written, or added to when accumulate = 1)
 *   gx    [B, L, Cx]     dtype dt (written)
 *   ws    device scratch of instant_backward_workspace_bytes(...) bytes,
 *         16-byte aligned.  ZERO IT ONCE after allocating it: its first bytes
 *         are the counters, which every call leaves zero again; zero it again
 *         after instant_device_status has reported INSTANT_ERR_DEVICE.  Calls
 *         that may run at the same time need separate workspaces.
 * Limits: 1 <= Ry <= 64, Rx + Ry <= 128.
 */
instant_status instant_backward(const void* gy, const void* PQ, const void* xhat, const void* w,
                                void* Sx, void* Sq, float* gw, int accumulate, void* gx,
                                void* ws, size_t ws_bytes, int B, int L, int Cx, int Cy,
                                int Rx, int Ry, instant_dtype dt, void* stream);

size_t instant_backward_workspace_bytes(int B, int L, int Cx, int Cy, int Ry, instant_dtype dt);

/*
 * The two halves of instant_grad_x, for callers that schedule or time them
 * separately.  instant_grad_x_core computes g_hat_x = Sq w (关键设计 3,
 * g_hat_x = g_hat_y2 w) into `ws` as [B*Ry, Cx] in dtype dt (its split-K
 * partial sums are reduced on chip); instant_expand reads it back and writes
 * g_tilde_x,b = Q^T g_hat_x,b.  Call them with the same sizes and the same
 * workspace (of instant_grad_x_workspace_bytes bytes), in that order on one
 * stream.
 */
instant_status instant_grad_x_core(const void* Sq, const void* w, void* ws, size_t ws_bytes,
                                   int B, int Cx, int Cy, int Ry,
                                   instant_dtype dt, void* stream);
instant_status instant_expand(const void* Q, void* gx, const void* ws, size_t ws_bytes,
                              int B, int L, int Cx, int Cy, int Ry,
                              instant_dtype dt, void* stream);

/*
 * instant_grad_x without a workspace argument.  The page has no counterpart:
 * this is a convenience of the library for callers that cannot allocate
 * device memory -- a C host linking only this library, with no device
 * allocator of its own, or a training loop whose device memory is planned at
 * start-up and must not grow (or synchronise on a cudaMalloc) afterwards.
 *
 * Same arguments, result and limits as instant_grad_x, minus ws/ws_bytes.  It
 * always runs the two-kernel form (instant_grad_x_core, then instant_expand)
 * with g_hat_x in a fixed device array of INSTANT_GRAD_X_STATIC_SCRATCH_BYTES
 * bytes that belongs to the library's CUDA module; no device memory is
 * allocated or freed by the call.
 *   - Returns INSTANT_ERR_WORKSPACE when the intermediate,
 *     instant_grad_x_workspace_bytes(B, L, Cx, Cy, Ry, dt) bytes, is larger
 *     than INSTANT_GRAD_X_STATIC_SCRATCH_BYTES; nothing is launched then.
 *   - The first call on each device looks up the array's device address with
 *     that device current (this may load the module there); make that first
 *     call before any stream capture begins.
 *   - There is one array per device, shared by every call on it: two calls
 *     whose executions overlap on one device (other streams, other host
 *     threads) race on it and both results are undefined.  Serialise them,
 *     e.g. by issuing them on one stream.
 */
#define INSTANT_GRAD_X_STATIC_SCRATCH_BYTES ((size_t)8 << 20)
instant_status instant_grad_x_static(const void* Sq, const void* w, const void* Q, void* gx,
                                     int B, int L, int Cx, int Cy, int Ry,
                                     instant_dtype dt, void* stream);

/*
 * Autocorrelation statistic (关键设计 1: C = E[t t^T], only statistics are
 * accumulated during calibration, not the batch):
 *   C += sum_b t_b t_b^T
 *   t  [B, L, Cdim]  dtype dt (read)
 *   C  [L, L]        fp32, accumulated in place (caller zeroes it and keeps
 *                    the sample count; E[t t^T] = C / count)
 * Limits: L <= 8192.
 */
instant_status instant_calib_accumulate(const void* t, float* C, int B, int L, int Cdim,
                                        instant_dtype dt, void* stream);

/*
 * Several statistics of one token length L accumulated in one call (关键设计
 * 1: a layer accumulates C_X from its activations and C_G from its output
 * gradients at the same step): for each item, C += sum_b t_b t_b^T exactly
 * as instant_calib_accumulate does (the fp32 sums may add in another order).
 * Up to four statistics share one launch.
 *   items  HOST array of `count` items: t [B, L, Cdim] (device, dtype dt),
 *          C [L, L] fp32 (device, accumulated in place), B, Cdim
 * Limits: L <= 8192; the items' C must not overlap.
 */
typedef struct {
  const void* t;
  float* C;
  int B;
  int Cdim;
} instant_accumulate_item;

instant_status instant_calib_accumulate_batch(const instant_accumulate_item* items, int count,
                                              int L, instant_dtype dt, void* stream);

/*
 * Projector from an accumulated statistic (关键设计 1 and 2):
 *   C/n = U Sigma U^T (symmetric PSD, so the SVD is the eigendecomposition);
 *   E = ||C/n||_F^2 (fp64, from C directly);
 *   k = smallest index with sum_{i<=k} sigma_i^2 >= eps * E  (fp64);
 *   R = r_override if > 0, else min(k + p, L);
 *   s = (sum_{i<=R} sigma_i^2)^(-1/2) if scale_on, else 1;
 *   rows_out[i, :] = s * u_i^T for i < R, each u_i signed so that its
 *   largest-magnitude entry is positive.
 * Arguments
 *   C          [L, L] fp32 device (read): the accumulated sum
 *   n_samples  number of samples summed into C (> 0)
 *   rows_out   [r_cap, L] device, dtype dt: rows 0..R-1 written, rows R..r_cap-1 zeroed
 *   k_out, r_out, scale_out, energy_out: HOST pointers (energy_out may be NULL)
 *   eig_out    HOST, r_cap doubles (may be NULL): sigma_1..sigma_{r_cap}, 0 past
 *              the solved block
 *   ws         device scratch of instant_calib_workspace_bytes(L, r_cap) bytes
 * Method: L <= 128 -> one-CTA cyclic Jacobi on the full matrix; larger L ->
 * block subspace iteration with Rayleigh-Ritz (block <= 128 columns), as a
 * single launch of one cluster (8 CTAs; 16 above 1024 tokens) up to L = 2048
 * with blocks of 16 or 32 columns, as a host loop of launches otherwise.  A Ritz pair counts as
 * converged when its residual is below 1e-3 of its own Ritz value (so that
 * the trailing rows of a decaying spectrum are accurate too), or when it is
 * below prm->tol (default 2e-5) times the largest Ritz value and no longer
 * shrinking (the fp32 rounding floor).
 * Returns INSTANT_ERR_NOT_CONVERGED when the cap is hit or when k + p does not
 * fit the block, INSTANT_ERR_NONFINITE when E is not finite and positive.
 * Synchronises `stream`.
 */
instant_status instant_calib_solve(const float* C, long long n_samples, int L,
                                   const instant_calib_params* prm,
                                   void* rows_out, int r_cap, instant_dtype dt,
                                   int* k_out, int* r_out, float* scale_out,
                                   double* energy_out, double* eig_out,
                                   void* ws, size_t ws_bytes, void* stream);

size_t instant_calib_workspace_bytes(int L, int r_cap);

/*
 * Several statistics of one token length L solved in one call (关键设计 1
 * and 2: a layer calibrates P from its activations and Q from its output
 * gradients at the same step, and a model calibrates all its layers at the
 * same step).  Each problem gets what instant_calib_solve would give it
 * alone (same kernels, same arithmetic: bit for bit on the one-launch solver;
 * the multi-launch path adds some partial sums with atomics, so any two of its
 * runs agree only up to that rounding order); the problems that the
 * one-launch solver takes (128 < L <= 2048, block of 16 or 32 columns) run
 * together, one cluster each (8 CTAs; 16 above 1024 tokens), up to 16 per
 * launch, with one synchronisation for all of them.
 *
 * instant_calib_problem: one statistic.
 *   C, n_samples, prm, rows_out, r_cap, eig_out   as for instant_calib_solve
 *                 (C, rows_out: device; eig_out: HOST or NULL)
 *   k, R, scale, energy   outputs (host struct, written by the call)
 *   status        this problem's own result
 * Arguments
 *   problems   HOST array of `count` problems (count >= 1)
 *   dt         dtype of every rows_out
 *   ws         device scratch of instant_calib_batch_workspace_bytes(L, count)
 *              bytes: the one-launch results of all problems side by side (one
 *              copy to the host), then one slice per problem
 * Returns INSTANT_OK when every problem succeeded, else the first failing
 * problem's status.  Argument, shape, dtype, alignment or workspace errors of
 * any problem are reported before anything is launched, with that error in
 * every problem's `status`.  Synchronises `stream`.
 */
typedef struct {
  const float* C;
  long long n_samples;
  instant_calib_params prm;
  void* rows_out;
  int r_cap;
  double* eig_out;
  int k;
  int R;
  float scale;
  double energy;
  instant_status status;
} instant_calib_problem;

instant_status instant_calib_solve_batch(instant_calib_problem* problems, int count, int L,
                                         instant_dtype dt, void* ws, size_t ws_bytes,
                                         void* stream);

size_t instant_calib_batch_workspace_bytes(int L, int count);

/*
 * How much of a tensor a projector keeps (关键设计 2: the oversampling p guards
 * the compression against the subspace drifting between recalibrations):
 *   err2   = sum_b ||t_b - Q^T S_b||_F^2        energy = sum_b ||t_b||_F^2
 * with S_b = Q t_b already computed, e.g. by instant_compress_act(t, Q, S, ...).
 * For orthonormal rows of Q (a projector solved with scale_on = 0),
 * sqrt(err2 / energy) = ||t - Q^T Q t|| / ||t||.
 *   t   [B, L, C]   dtype dt (read)
 *   Q   [R, L]      dtype dt (read)
 *   S   [B*R, C]    dtype dt (read), row b*R + r
 *   err2_out, energy_out: HOST doubles
 *   ws  device scratch of at least 16 bytes, 8-byte aligned (two fp64 totals)
 * Limits: 1 <= R <= 64, R * L <= 12288.  Synchronises `stream`.
 */
instant_status instant_reconstruction_error(const void* t, const void* Q, const void* S,
                                           int B, int L, int C, int R, instant_dtype dt,
                                           double* err2_out, double* energy_out,
                                           void* ws, size_t ws_bytes, void* stream);

/* Reads (and clears when clear != 0) the sticky device status word after
 * synchronising `stream`; INSTANT_OK when no device-side wait ran out. */
instant_status instant_device_status(int clear, void* stream);

const char* instant_status_string(instant_status s);

/* Library version: major * 10000 + minor * 100 + patch. */
int instant_version(void);

/* Number of kernels the library has launched in this process (host-side
 * counter, incremented at every launch; monotonic). */
unsigned long long instant_launch_count(void);

#ifdef __cplusplus
}
#endif

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif
#endif /* INSTANT_H_ */
