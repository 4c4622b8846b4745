/*
 * muon.h -- C ABI of the one-GPU Muon optimiser step for GB300 (sm_103a).
 *
 * The step is the local part of the distributed Muon update described in
 * "Frontier Pre-training at Microsoft AI" (papercache deepnotes summary),
 * Method details §5 "Scaling Muon to 16K GPUs", resharding steps 1, 3 and 5,
 * and in "Microsoft Reveals MAI-Base-2 Training Recipe" (xiaohu-jiedu),
 * section "How to Make Parameter Updates Faster and More Stable?":
 *   1. update the FP32 momentum in place and cast it to BF16;
 *   2. batch parameters of identical shape;
 *   3. orthogonalise every whole momentum matrix with a symmetry-aware
 *      Newton-Schulz operator;
 *   4. cast the result back to FP32 and apply it to the FP32 weights.
 * The two all-to-all exchanges between the steps move data between GPUs
 * and are not part of this one-GPU library.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named *_dev are CUDA device pointers owned by the caller; the
 *    library never frees them.  Pointers named *_host are host pointers.
 *  - Matrices are dense, row-major and contiguous.  A group of `count`
 *    matrices of rows x cols is one buffer of count*rows*cols elements.
 *  - "Wide" layout: a matrix with rows > cols is orthogonalised as its
 *    transpose, so the BF16 working copy of every matrix is m x n with
 *    m = min(rows, cols) <= n = max(rows, cols).
 *  - BF16 values travel as uint16_t bit patterns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued asynchronously; no entry point synchronises
 *    the stream unless it says so.  Kernels are launched with programmatic
 *    stream serialisation: a kernel may be scheduled while the previous
 *    kernel in the stream still runs, but reads and writes global memory
 *    only after that kernel has completed, so stream order is kept.  The
 *    environment variable MUON_PDL=0 turns this off (plain launches).
 *  - Arguments are validated on the host before anything is enqueued: an
 *    invalid argument returns MUON_ERR_INVALID_ARG and launches nothing.
 *  - A handle is bound to the device that was current when it was created
 *    and is not thread-safe.
 *  - Kernels report device-side failures (a bounded wait that expired, a
 *    non-finite norm) through a flag read by muon_last_device_error().
 */
#ifndef MUON_GB300_H_
#define MUON_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MUON_OK = 0,
  MUON_ERR_INVALID_ARG = 1,       /* bad pointer, size, count or value */
  MUON_ERR_NOMEM = 2,             /* workspace allocation failed */
  MUON_ERR_CUDA = 3,              /* a CUDA runtime/driver call failed */
  MUON_ERR_UNSUPPORTED_ARCH = 4,  /* device is not compute capability 10.3 */
  MUON_ERR_TIMEOUT = 5,           /* a bounded device-side wait expired */
  MUON_ERR_NONFINITE = 6,         /* a momentum norm was NaN or Inf */
  MUON_ERR_NO_DEVICE = 7          /* no CUDA device is visible */
} muon_status_t;

typedef struct muon_handle_s* muon_handle_t;

/* One group of same-shape parameters ("Scaling Muon to 16K GPUs",
 * resharding step 2: parameters of identical shape are batched).
 * `update_scale` multiplies the orthogonalised update (1.0 = plain step). */
typedef struct {
  int32_t rows;
  int32_t cols;
  int32_t count;
  float update_scale;
} muon_group_t;

/* Kernel classes, for timing and launch accounting. */
typedef enum {
  MUON_KERNEL_MOMENTUM_CAST = 0,  /* momentum update + BF16 cast + transpose */
  MUON_KERNEL_NORM = 1,           /* per-matrix Frobenius norm finalisation */
  MUON_KERNEL_NS_GRAM = 2,        /* A = alpha X X^T (symmetric storage, see below) */
  MUON_KERNEL_NS_POLY = 3,        /* B' = a I + b A + c A A (same storage as A) */
  MUON_KERNEL_NS_UPDATE = 4,      /* X' = alpha B' X  (= alpha (a X + b A X + c A^2 X)) */
  MUON_KERNEL_APPLY = 5,          /* W = W (1 - lr wd) - lr s O */
  MUON_KERNEL_SCALE = 6,          /* ns_steps == 0: O = X / s */
  MUON_KERNEL_ADAMW = 7,          /* AdamW companion */
  MUON_KERNEL_TRANSPOSE = 8,      /* BF16 transpose (resharded step) */
  MUON_KERNEL_COUNT = 9
} muon_kernel_t;

typedef struct {
  double total_ms[MUON_KERNEL_COUNT];   /* summed device time per class */
  int64_t launches[MUON_KERNEL_COUNT];  /* launches per class */
  int64_t total_launches;               /* all kernel launches of the handle */
} muon_kernel_stats_t;

/* Plan summary of a group list (pure host computation, no GPU needed). */
typedef struct {
  int32_t n_batches;          /* distinct wide shapes (Newton-Schulz batches) */
  int32_t n_chunks;           /* batch chunks that fit the workspace */
  int32_t max_chunk_matrices; /* largest chunk */
  int64_t matrices;           /* total matrices */
  size_t workspace_bytes;     /* device workspace the plan needs */
  double ns_algorithmic_flops;/* sum over matrices of ns_steps*(3 m^2 n + m^3) */
  int64_t launches_per_step;  /* kernel launches one muon_step makes */
} muon_plan_info_t;

/* Default Newton-Schulz configuration: quintic coefficients (a, b, c),
 * 5 iterations and the epsilon added to the Frobenius norm. */
#define MUON_NS_A 3.4445f
#define MUON_NS_B (-4.7750f)
#define MUON_NS_C 2.0315f
#define MUON_NS_STEPS 5
#define MUON_NORM_EPS 1e-7f

/* Human-readable name of a status code (static string, never NULL). */
const char* muon_status_string(muon_status_t status);

/* Text of the last error raised on the calling thread ("" if none). */
const char* muon_last_error_message(void);

/* Library version string. */
const char* muon_version(void);

/* Create a handle on `device` (-1 = the calling thread's current device).
 * `workspace_bytes_max` caps the device workspace the handle may allocate
 * (0 = default of 8 GiB); groups whose whole batch does not fit are
 * processed in chunks.  No device memory is allocated until first use.
 * Errors: INVALID_ARG (out == NULL), NO_DEVICE, UNSUPPORTED_ARCH (not
 * sm_103), CUDA. */
muon_status_t muon_create(muon_handle_t* out, int32_t device, size_t workspace_bytes_max);

/* Destroy a handle and free its workspace (synchronises the device). */
muon_status_t muon_destroy(muon_handle_t handle);

/* Plan of a group list under a workspace cap, without a GPU.
 * Same group rules as muon_step.  Errors: INVALID_ARG. */
muon_status_t muon_plan_describe(const muon_group_t* groups, int32_t n_groups,
                                 int32_t ns_steps, size_t workspace_bytes_max,
                                 muon_plan_info_t* out);

/* Partition of a group list's whole matrices over `world` data-parallel
 * ranks ("Scaling Muon to 16K GPUs", resharding step 2: after the
 * exchange every GPU holds a subset of complete matrices and orthogonalises
 * them independently, step 3).  Matrices are independent, so each rank
 * steps its own subset with no exchange between ranks.
 * The split is longest-processing-time-first over single matrices: in
 * order of decreasing estimated device time (ns_steps*(3 m^2 n + m^3)
 * algorithmic flops at 1.9 PFLOP/s plus 24 bytes per element at 6.8 TB/s),
 * each matrix goes to the rank with the least estimated time so far.  A
 * rank's matrices of one group are then laid out as one contiguous slice,
 * ranks in order (same loads, since a group's matrices are identical).
 * first_out, count_out: [n_groups * world] host arrays; entry g*world + r
 *   receives the first matrix index and the matrix count of rank r's slice
 *   of group g (count 0: none).  The slices of a group cover it exactly.
 * rank_seconds_out: NULL or [world] host array: each rank's estimated time.
 * Pure host computation, no GPU needed.  Errors: INVALID_ARG (bad groups,
 * ns_steps outside 0..64, world outside 1..65536, NULL outputs). */
muon_status_t muon_partition(const muon_group_t* groups, int32_t n_groups, int32_t ns_steps,
                             int32_t world, int64_t* first_out, int32_t* count_out,
                             double* rank_seconds_out);

/* The whole Muon step on device buffers ("Scaling Muon to 16K GPUs",
 * resharding steps 1, 3, 5; "How to Make Parameter Updates Faster and More
 * Stable?").  For every matrix of every group:
 *   M  <- mu * M + G                          (FP32, in place)
 *   X  <- bf16_rne(M), transposed if rows > cols
 *   s  <- ||M||_F + 1e-7
 *   X  <- X / s; then ns_steps times: A = X X^T; B = b A + c A^2;
 *         X = a X + B X                       (BF16 operands, FP32 accumulate)
 *   W  <- W (1 - lr*wd) - lr * update_scale * fp32(X), transposed back
 * groups:          [n_groups] host array; rows, cols >= 1; count >= 0.
 * momentum_dev:    [n_groups] host array of device pointers, FP32 in/out.
 * grad_dev:        [n_groups] host array of device pointers, FP32 read-only.
 * weights_dev:     [n_groups] host array of device pointers, FP32 in/out.
 * ns_steps:        0..64 (0 applies the normalised BF16 momentum).
 * The three buffers of a group must not overlap each other.
 * Same-wide-shape groups share one Newton-Schulz batch.
 * Errors: INVALID_ARG (NULL pointer with count > 0, bad sizes, non-finite
 * lr/wd/mu, unaligned pointer: 16-byte alignment is required), NOMEM, CUDA. */
muon_status_t muon_step(muon_handle_t handle, const muon_group_t* groups, int32_t n_groups,
                        float* const* momentum_dev, const float* const* grad_dev,
                        float* const* weights_dev, float lr, float wd, float mu,
                        int32_t ns_steps, void* stream);

/* The same step on HOST buffers: copies momentum, gradient and weights to
 * device staging owned by the handle, runs muon_step, copies momentum and
 * weights back, and synchronises `stream` before returning.  Pinned host
 * memory gives asynchronous copies.  Staging is grown on demand. */
muon_status_t muon_step_host(muon_handle_t handle, const muon_group_t* groups, int32_t n_groups,
                             float* const* momentum_host, const float* const* grad_host,
                             float* const* weights_host, float lr, float wd, float mu,
                             int32_t ns_steps, void* stream);

/* ------------------------------------------------------------------
 * Resharded step (ZeRO data parallelism over several GPUs).
 * "Frontier Pre-training at Microsoft AI", Method details §5, resharding
 * pipeline steps 1-5, and "How to Make Parameter Updates Faster and More
 * Stable?" ("batched momentum resharding"): each rank holds a flat shard
 * of every group's FP32 momentum, gradient and weights; it updates and
 * casts its momentum shard (step 1), an all-to-all per group gives every
 * rank the complete matrices muon_partition assigns it (step 2), the owner
 * orthogonalises them (step 3), a second all-to-all returns each shard's
 * update (step 4), and each rank applies it to its weight shard (step 5).
 * The exchanges themselves are collectives of the caller's communication
 * library; these entry points are the local compute between them.  A
 * shard is the element range [shard_begin, shard_end) of a group's flat
 * buffer; matrix k occupies [k E, (k + 1) E) with E = rows * cols.
 * ------------------------------------------------------------------ */

/* Step 1 on a shard: M <- mu M + G in place (FP32, fused multiply-add, the
 * same arithmetic as muon_step), x_shard <- bf16_rne(M) in the shard's
 * flat layout, and sumsq_out[y] <- the sum of M^2 over the shard's piece
 * of matrix shard_begin / E + y, for every matrix the shard touches
 * ((shard_end - 1) / E - shard_begin / E + 1 entries; FP32 per block,
 * FP64 across blocks, rounded to FP32).  momentum_shard, grad_shard:
 * shard_end - shard_begin FP32 (device); x_shard: as many BF16 (device);
 * sumsq_out: device FP32.  Uses the handle's workspace for the block
 * partials.  Errors: INVALID_ARG, NOMEM, CUDA. */
muon_status_t muon_shard_momentum_cast(muon_handle_t handle, int64_t shard_begin,
                                       int64_t shard_end, int64_t matrix_elems,
                                       float* momentum_shard, const float* grad_shard, float mu,
                                       uint16_t* x_shard, float* sumsq_out, void* stream);

/* On the owner of `count` whole wide matrices m x n (x_wide, BF16,
 * contiguous): inv_norm[k] <- 1 / (sqrt(sum of sumsq[k * parts + j] over j)
 * + 1e-7), the partial sums being the pieces' sums of squares gathered
 * from the shards (parts per matrix, zero where a rank held no piece).
 * As in muon_momentum_cast, a norm above 2^60 rescales x_wide by an exact
 * power of two and inv_norm by its inverse; a non-finite norm sets the
 * device error flag (MUON_ERR_NONFINITE).  Errors: INVALID_ARG, CUDA. */
muon_status_t muon_norm_from_sumsq(muon_handle_t handle, int32_t m, int32_t n, int32_t count,
                                   int32_t parts, const float* sumsq, uint16_t* x_wide,
                                   float* inv_norm, void* stream);

/* dst[k] <- src[k]^T for `count` BF16 matrices of rows x cols (both
 * contiguous, device, not overlapping): the owner turns tall matrices wide
 * for the Newton-Schulz products and the updates back.  Errors:
 * INVALID_ARG (sizes as muon_step's groups, NULL, overlap), CUDA. */
muon_status_t muon_transpose_bf16(muon_handle_t handle, int32_t rows, int32_t cols, int32_t count,
                                  const uint16_t* src, uint16_t* dst, void* stream);

/* Step 5 on a shard: W <- W (1 - lr wd) - lr scale fp32(O) over n_elems
 * flat elements (the same arithmetic as muon_step's apply).
 * weights_shard: FP32 in/out; o_shard: BF16 (device).  Errors:
 * INVALID_ARG (n_elems < 0, NULL, non-finite scalars), CUDA. */
muon_status_t muon_shard_apply(muon_handle_t handle, int64_t n_elems, float* weights_shard,
                               const uint16_t* o_shard, float lr, float wd, float scale,
                               void* stream);

/* Page-locked host memory for the buffers of muon_step_host
 * (cudaHostAlloc, portable across devices).  Copies from it run at the
 * host link's rate; on GB300 hosts measured here, memory locked after the
 * fact with cudaHostRegister copied at a fraction of that rate once more
 * than about 8 GiB of it was locked, while memory from this call kept the
 * full rate.  *out receives the pointer (NULL on failure); free it with
 * muon_host_free.  Errors: INVALID_ARG (out == NULL, bytes == 0), NOMEM. */
muon_status_t muon_host_alloc(size_t bytes, void** out);

/* Free memory from muon_host_alloc (NULL is accepted).  Synchronises with
 * copies still reading or writing it.  Errors: CUDA. */
muon_status_t muon_host_free(void* ptr);

/* Shape rules for the update scale (common Muon variants; the pages give
 * no formula).  The factor multiplies each group's own update_scale. */
typedef enum {
  MUON_SCALE_NONE = 0,         /* 1 */
  MUON_SCALE_SQRT_ASPECT = 1,  /* sqrt(max(1, rows / cols)), rows = output dim */
  MUON_SCALE_RMS_MATCH = 2     /* rms_target * sqrt(max(rows, cols)) */
} muon_scale_rule_t;

/* Options of muon_step_ex. */
typedef struct {
  float lr, wd, mu;
  int32_t ns_steps;       /* 0..64 */
  int32_t nesterov;       /* 0: orthogonalise M' ; 1: orthogonalise G + mu*M' */
  const float* coeffs;    /* host, NULL or 3*ns_steps floats: (a, b, c) per iteration */
  int32_t scale_rule;     /* muon_scale_rule_t */
  float rms_target;       /* MUON_SCALE_RMS_MATCH target (<= 0: 0.2) */
} muon_options_t;

/* muon_step with method variants: Nesterov momentum (the matrix
 * orthogonalised, and normed, is U = G + mu*M' with M' the updated
 * momentum), a per-iteration coefficient schedule, and a shape rule for
 * the update scale.  With nesterov = 0, coeffs = NULL and
 * MUON_SCALE_NONE it equals muon_step.  Same buffers and errors as
 * muon_step; INVALID_ARG also for a NULL opts, an unknown rule or
 * non-finite coefficients. */
muon_status_t muon_step_ex(muon_handle_t handle, const muon_group_t* groups, int32_t n_groups,
                           float* const* momentum_dev, const float* const* grad_dev,
                           float* const* weights_dev, const muon_options_t* opts, void* stream);

/* Step 1 alone: momentum update, BF16 cast into wide layout, and the
 * per-matrix inverse scale 1/(||M||_F + 1e-7).
 * momentum_dev:  count*rows*cols FP32, updated in place.
 * grad_dev:      count*rows*cols FP32.
 * x_wide_dev:    count*m*n BF16 output (m = min, n = max of rows, cols).
 * inv_norm_dev:  count FP32 output.
 * A matrix with ||M||_F > 2^60 (about 1.15e18) leaves its x_wide scaled by
 * an exact power of two 2^e (so that its norm is in [1, 2)) and inv_norm by
 * 2^-e: x * inv_norm, the Newton-Schulz input, is unchanged, and the
 * products' FP32 accumulators stay in range.  The same holds inside
 * muon_step and muon_step_ex. */
muon_status_t muon_momentum_cast(muon_handle_t handle, int32_t rows, int32_t cols, int32_t count,
                                 float* momentum_dev, const float* grad_dev, float mu,
                                 uint16_t* x_wide_dev, float* inv_norm_dev, void* stream);

/* Step 3 alone: batched symmetric Newton-Schulz on `count` wide BF16
 * matrices m x n (m <= n), each pre-scaled by inv_norm[i]:
 *   X0 = inv_norm[i] * x[i]; ns_steps times X = a X + (b A + c A^2) X,
 *   A = X X^T.
 * Each iteration is three products, every result rounded to BF16 where
 * it is stored:
 *   Gram    A  = alpha X X^T            (alpha = inv_norm^2 at iteration 0, else 1)
 *   square  B' = a I + b A + c A A      (the linear term folded into B')
 *   update  X' = alpha B' X             (alpha = inv_norm at iteration 0, else 1)
 * Storage of the symmetric A and B': for m > 128 only the 256 x 256 blocks
 * on and above the block diagonal are computed and stored, nothing is
 * mirrored, and a consumer reads a block left of the diagonal as the
 * transpose of the stored block above it; for m <= 128 the matrix is one
 * tile, computed once and stored in full (the part above the diagonal
 * also written mirrored below it).  MUON_NS_PAIR=0 in the environment
 * runs every size on the single-CTA kernels (128-row tiles, stored in
 * full), for comparisons.
 * x_dev, out_dev: count*m*n BF16, 16-byte aligned, must not overlap.
 * inv_norm_dev:   count FP32 (device).
 * coeffs_host:    3 floats (a, b, c) or NULL for the defaults.
 * m and n must be multiples of 8 (row pitch of 16 bytes for the tensor
 * memory accelerator).  Errors: INVALID_ARG, NOMEM, CUDA. */
muon_status_t muon_newton_schulz_bf16(muon_handle_t handle, int32_t m, int32_t n, int32_t count,
                                      const uint16_t* x_dev, uint16_t* out_dev,
                                      const float* inv_norm_dev, int32_t ns_steps,
                                      const float* coeffs_host, void* stream);

/* Step 5 alone: W <- W (1 - lr*wd) - lr*scale*fp32(O), O given in wide
 * layout (transposed back when rows > cols).
 * weights_dev: count*rows*cols FP32 in/out; o_wide_dev: count*m*n BF16. */
muon_status_t muon_apply_update(muon_handle_t handle, int32_t rows, int32_t cols, int32_t count,
                                float* weights_dev, const uint16_t* o_wide_dev,
                                float lr, float wd, float scale, void* stream);

/* Newton-Schulz without any memory allocation (no handle).
 *
 * The pages have no counterpart of this entry point: it exists for callers
 * that cannot allocate device memory at the time they orthogonalise --
 * code running inside CUDA graph construction, custom allocators or
 * runtimes that must not re-enter the CUDA allocator, and deployments
 * whose device memory is fixed at start-up.  It computes what
 * muon_newton_schulz_bf16 computes, with the same arguments and layout,
 * but its scratch (one more m x n iterate plus the m x m matrices A and B
 * per matrix) lives in a file-scope device array of
 * MUON_STATIC_SCRATCH_BYTES (64 MiB) that every GPU loading the library
 * holds until the process exits.  It calls no cudaMalloc, cudaFree or
 * allocating library routine.
 *  - Limit: one matrix must fit the array, i.e.
 *    2*m*n + 4*m*m bytes (each part rounded up to 256) <= 64 MiB - 256;
 *    larger matrices are rejected with MUON_ERR_INVALID_ARG and a message
 *    (muon_last_error_message).  Larger counts are processed in passes.
 *  - First call on a device: resolves the array's device address
 *    (cudaGetSymbolAddress) and sets kernel attributes, with that device
 *    current.  Make that first call before any stream capture.  If that
 *    set-up fails the call returns MUON_ERR_CUDA and the next call on the
 *    device tries the set-up again.
 *  - Sharing: every call uses the same array and leaves its last contents
 *    there; nothing in it needs to start at zero (every scratch element is
 *    written before it is read).  Calls that overlap on the GPU (different
 *    streams, or different host threads) race on the array: serialise them.
 *  - error_flag_dev: optional device int that receives the device error
 *    bits (1 = a bounded wait expired); the caller zeroes it.  With NULL,
 *    the bits go to a word inside the array (cleared at each call) and are
 *    not reported.
 * Errors: INVALID_ARG (shapes as for muon_newton_schulz_bf16, matrix too
 * large for the array, NULL or unaligned buffers, overlap), CUDA. */
#define MUON_STATIC_SCRATCH_BYTES (64u << 20)
muon_status_t muon_newton_schulz_bf16_static(int32_t m, int32_t n, int32_t count,
                                             const uint16_t* x_dev, uint16_t* out_dev,
                                             const float* inv_norm_dev, int32_t ns_steps,
                                             const float* coeffs_host, int32_t* error_flag_dev,
                                             void* stream);

/* Synchronise `stream`, then read and clear the handle's device error
 * flag: MUON_OK, MUON_ERR_TIMEOUT or MUON_ERR_NONFINITE. */
muon_status_t muon_last_device_error(muon_handle_t handle, void* stream);

/* AdamW options (decoupled weight decay, bias correction; step >= 1 is the
 * 1-based step count used for the bias corrections). */
typedef struct {
  float lr, beta1, beta2, eps, wd;
  int32_t step;
} muon_adamw_options_t;

/* AdamW companion for the parameters Muon does not handle -- embeddings,
 * norms, scalars ("Microsoft Reveals MAI-Base-2 Training Recipe", section
 * "How to Make Parameter Updates Faster and More Stable?": Muon for 2-D
 * non-embedding matrices, AdamW for the rest).  For every tensor i (FP32,
 * numel[i] elements, device pointers, updated in place except grads):
 *   p <- p (1 - lr wd);  m <- b1 m + (1 - b1) g;  v <- b2 v + (1 - b2) g^2
 *   p <- p - (lr / (1 - b1^step)) m / (sqrt(v) / sqrt(1 - b2^step) + eps)
 * numel: host array; the four pointer arrays are host arrays of device
 * pointers, 4-byte aligned (16-byte alignment enables vector access).
 * Up to 40 tensors per kernel launch; more are launched in batches.
 * Errors: INVALID_ARG (NULL, unaligned, beta outside [0,1), eps <= 0,
 * step < 1, non-finite), CUDA. */
muon_status_t muon_adamw_step(muon_handle_t handle, int32_t n_tensors, const int64_t* numel,
                              float* const* params_dev, const float* const* grads_dev,
                              float* const* exp_avg_dev, float* const* exp_avg_sq_dev,
                              const muon_adamw_options_t* opts, void* stream);

/* Failure-path self-test of the bounded device waits: launches one small
 * kernel that waits, through the same wait routine the Newton-Schulz
 * kernels use, on a barrier nothing will complete.  The wait gives up after
 * `limit_ms` (1..2000), sets the handle's device error flag and the kernel
 * returns normally, leaving the context usable; muon_last_device_error()
 * then reports MUON_ERR_TIMEOUT.  No fault, trap or hang is involved.
 * Errors: INVALID_ARG (limit out of range), CUDA. */
muon_status_t muon_selftest_bounded_wait(muon_handle_t handle, int32_t limit_ms, void* stream);

/* Per-kernel timing: when enabled, every launch is bracketed by CUDA
 * events on the launching stream.  muon_kernel_stats synchronises the
 * device, folds the recorded events into `out` and keeps accumulating;
 * muon_reset_kernel_stats clears the totals. */
muon_status_t muon_set_kernel_timing(muon_handle_t handle, int32_t enable);
muon_status_t muon_kernel_stats(muon_handle_t handle, muon_kernel_stats_t* out);
muon_status_t muon_reset_kernel_stats(muon_handle_t handle);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* MUON_GB300_H_ */
