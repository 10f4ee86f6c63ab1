/*
 * qk.h -- C ABI of the GB300 row-reduction library (libqk.so).
 *
 * Three forward operators over a row-major M x N matrix, each reading every
 * input element from HBM once and writing every output element once:
 *
 *   qk_softmax_fwd   y[i, :] = softmax(x[i, :])
 *   qk_rmsnorm_fwd   y[i, :] = x[i, :] * rstd[i] * w[:],
 *                    rstd[i] = 1 / sqrt(mean_j x[i, j]^2 + eps)
 *   qk_xent_fwd      lse[i]  = log sum_j exp(x[i, j]),  loss[i] = lse[i] - x[i, t[i]]
 *
 * The operators are the three reductions named in the QbitAI article on QuACK
 * ("无需CUDA代码，给H100加速33%-50%"), section "让内存密集型内核达到“光速”"
 * (RMSNorm, softmax and cross-entropy loss), benchmarked forward-only in its
 * section "内存吞吐量" (fp32 and bf16, batch 8k-32k rows, 256-262k columns).
 * The article gives no formulas; the textbook definitions above are used.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers are DEVICE pointers owned by the caller (for example the
 *    data_ptr() of CUDA tensors).  The library keeps no reference to them
 *    after the call is enqueued and allocates no device memory per call.
 *  - Matrices are dense and row-major with row stride N elements.  x, y and w
 *    have the element type `dtype`; rstd, loss and lse are float32; targets are
 *    int64.
 *  - Every call is asynchronous: it validates its arguments on the host, then
 *    enqueues kernels on `stream` (a cudaStream_t; NULL means the legacy
 *    default stream) on the calling thread's current device and returns.
 *  - Argument errors are returned synchronously and nothing is launched.  A
 *    launch failure returns QK_ERR_LAUNCH.  Device-side failures (a bounded
 *    wait inside a kernel that ran out) are recorded in a per-device status
 *    word that qk_get_device_status() reads and clears.
 *  - M == 0 is a no-op returning QK_OK.  N <= 0 or M < 0 is QK_ERR_INVALID_ARG.
 *  - Pointers must be aligned to their element size (QK_ERR_MISALIGNED
 *    otherwise).  The fast path additionally wants 16-byte aligned x, y, w and
 *    N * sizeof(dtype) a multiple of 16.  Other forward inputs take a shifted
 *    ring kernel when y has x's alignment modulo 16 (rows start anywhere inside
 *    a 16-byte vector) and a masked element kernel otherwise; both compute the
 *    same definitions within the same tolerances as the fast path (the order
 *    of their fp32 sums differs, so the last bits can).
 *  - Launches are stream-ordered with programmatic dependent launch: a kernel
 *    may start, and prefetch the first rows it will read into L2, while the
 *    previous kernel on the stream is still running, but it reads its inputs
 *    and writes its outputs only after that kernel has completed, so one call
 *    may consume another's output (or overwrite its input) with no extra
 *    synchronisation.
 *  - Accumulation is float32; bf16 outputs are rounded to nearest even once.
 *  - Per-device state (the device's properties, kernel attributes, occupancy
 *    answers, the device addresses of the status word and of the
 *    no-allocation scratch array) is set up by the first call made on each
 *    device and kept until the process exits.  A cudaDeviceReset() of a device
 *    after the library's first call on it is not supported: the cached
 *    addresses and kernel attributes no longer match the new context, so
 *    calls on that device may fail to launch or touch stale addresses.
 */
#ifndef QK_H_
#define QK_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QK_API __attribute__((visibility("default")))
#else
#define QK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { QK_F32 = 0, QK_BF16 = 1 } qk_dtype;

/* Operators, as named by qk_get_plan / qk_set_plan_override / qk_max_row_elements:
 * the three forward passes, their backward passes, and LayerNorm forward. */
typedef enum {
  QK_OP_SOFTMAX = 0,
  QK_OP_RMSNORM = 1,
  QK_OP_XENT = 2,
  QK_OP_SOFTMAX_BWD = 3,
  QK_OP_RMSNORM_BWD = 4,
  QK_OP_XENT_BWD = 5,
  QK_OP_LAYERNORM = 6
} qk_op;

typedef enum {
  QK_OK = 0,
  QK_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad dtype, overlapping buffers */
  QK_ERR_UNSUPPORTED = 2, /* row longer than the largest plan (see qk_max_row_elements) */
  QK_ERR_MISALIGNED = 3,  /* a pointer not aligned to its element size */
  QK_ERR_LAUNCH = 4,      /* the CUDA runtime refused a launch or a query */
  QK_ERR_TIMEOUT = 5,     /* a bounded wait inside a kernel ran out (device status) */
  QK_ERR_NO_DEVICE = 6    /* no usable CUDA device, or not an sm_103 device */
} qk_status;

/*
 * Softmax forward.  For each row i: m = max_j x[i,j];
 * y[i,j] = exp(x[i,j] - m) / sum_k exp(x[i,k] - m).
 * Cited: QbitAI article on QuACK, section "让内存密集型内核达到“光速”" (softmax as
 * a reduction over the row) and section "内存吞吐量" (three sweeps: maximum, sum
 * of exponentials, normalisation; here the first two are fused on chip).
 *
 *   x      [M, N] dtype, read once.
 *   y      [M, N] dtype, written once.  y == x (exact aliasing) is allowed;
 *          any other overlap with x is QK_ERR_INVALID_ARG.
 *   M, N   rows and columns (any N on the aligned path; see qk_max_row_elements).
 * Non-finite inputs (not part of the parity contract): a -inf entry gets
 * probability 0 and the rest of its row is the softmax of the finite entries
 * (masked logits); a row with no finite entry has no distribution (0/0) and
 * gets NaN in every entry, as the definition gives; NaN and +inf propagate.
 */
QK_API qk_status qk_softmax_fwd(const void* x, void* y, int64_t M, int64_t N, qk_dtype dtype,
                         void* stream);

/*
 * RMSNorm forward.  For each row i: rstd[i] = 1 / sqrt((1/N) sum_j x[i,j]^2 + eps);
 * y[i,j] = x[i,j] * rstd[i] * w[j]  (eps inside the root, plain weight, no bias).
 * Cited: QbitAI article on QuACK, section "让内存密集型内核达到“光速”" (RMSNorm as a
 * reduction over the row).
 *
 *   x      [M, N] dtype, read once.
 *   w      [N] dtype, read once per CTA (cached on chip).
 *   y      [M, N] dtype, written once; y == x allowed, other overlaps rejected.
 *   rstd   [M] float32, written once; may be NULL when not wanted.
 *   eps    added to the mean of squares; must be finite and >= 0.
 */
QK_API qk_status qk_rmsnorm_fwd(const void* x, const void* w, void* y, float* rstd, int64_t M,
                         int64_t N, float eps, qk_dtype dtype, void* stream);

/*
 * LayerNorm forward.  For each row i, with the population variance:
 *   mean[i] = (1/N) sum_j x[i,j],  var[i] = (1/N) sum_j (x[i,j] - mean[i])^2,
 *   rstd[i] = 1 / sqrt(var[i] + eps),  y[i,j] = (x[i,j] - mean[i]) * rstd[i] * w[j] + b[j].
 * The article names RMSNorm, softmax and cross-entropy only; its section "总结"
 * says the RMSNorm kernel's layout, copy strategy and reduction helpers carry
 * over to other row reductions, and LayerNorm is that carry-over with a
 * (mean, M2) pair reduced instead of a sum of squares.  The pair is merged
 * with the pairwise form of Welford's update (Chan et al.), so the variance
 * is not formed as a difference of two large sums.  Each element of x is read
 * from HBM once.
 *
 *   x      [M, N] dtype, read once.
 *   w      [N] dtype; b [N] dtype or NULL (no bias); both cached on chip.
 *   y      [M, N] dtype, written once; y == x allowed, other overlaps rejected.
 *   mean   [M] float32, may be NULL; rstd [M] float32, may be NULL.
 *   eps    added to the variance; must be finite and >= 0.
 *   Any N on the aligned path: rows longer than a cluster holds (1 MiB) are
 *   streamed through shared memory twice (three HBM passes).  Unaligned rows
 *   go up to 524,288 elements.
 */
QK_API qk_status qk_layernorm_fwd(const void* x, const void* w, const void* b, void* y,
                                  float* mean, float* rstd, int64_t M, int64_t N, float eps,
                                  qk_dtype dtype, void* stream);

/*
 * Cross-entropy loss forward, one value per row (no reduction over rows, no
 * ignore index, no label smoothing).  For each row i: lse[i] = log sum_j
 * exp(x[i,j]); loss[i] = lse[i] - x[i, targets[i]].  A target outside [0, N)
 * yields loss[i] = NaN (lse[i] is still written); nothing is read out of bounds.
 * Cited: QbitAI article on QuACK, section "让内存密集型内核达到“光速”" (cross-entropy
 * loss as the third reduction) and section "内存吞吐量" (an online softmax when
 * the row does not fit on chip: the row is streamed through shared memory).
 *
 *   logits  [M, N] dtype, read once.
 *   targets [M] int64.
 *   loss    [M] float32, written once.
 *   lse     [M] float32, written once; may be NULL when not wanted.
 *   Any N >= 1 is supported.
 * Non-finite logits: -inf entries drop out of the sum (masked logits); a
 * -inf target logit gives loss = +inf; a row with no finite entry gives
 * lse = -inf (the log of an empty sum) and loss = NaN.
 */
QK_API qk_status qk_xent_fwd(const void* logits, const int64_t* targets, float* loss, float* lse,
                      int64_t M, int64_t N, qk_dtype dtype, void* stream);

/*
 * Backward passes.  The article benchmarks the forward passes only; these are
 * the derivatives of the same definitions, built on the same read-once ring
 * kernels (each input element read from HBM once, each output written once).
 * The fast path wants x, y, dy, dx, w and the logits 16-byte aligned and
 * N * sizeof(dtype) a multiple of 16; rows may then hold up to half of
 * qk_max_row_elements' forward limit (softmax, RMSNorm; see
 * qk_max_row_elements(QK_OP_*_BWD, dtype)).  Other inputs (pointers aligned to
 * their element size) take a masked path with the same results: any N for
 * cross-entropy, rows of up to 131,072 elements for softmax and RMSNorm
 * (QK_ERR_UNSUPPORTED beyond).
 */

/*
 * Softmax backward: dx[i,j] = y[i,j] * (dy[i,j] - sum_k dy[i,k] * y[i,k]).
 *   y    [M, N] dtype, the forward output; dy [M, N] dtype, the upstream gradient.
 *   dx   [M, N] dtype, written once; may alias y or dy exactly.
 */
QK_API qk_status qk_softmax_bwd(const void* y, const void* dy, void* dx, int64_t M, int64_t N,
                                qk_dtype dtype, void* stream);

/*
 * Bytes of device workspace qk_rmsnorm_bwd needs for these sizes on the
 * current device (fp32 partial column sums of dw, one row per CTA): enough
 * for the fast and for the masked path, whichever the pointers select.
 */
QK_API qk_status qk_rmsnorm_bwd_workspace_size(int64_t M, int64_t N, qk_dtype dtype,
                                               size_t* bytes);

/*
 * RMSNorm backward, for y = x * rstd * w with rstd = 1/sqrt(mean(x^2) + eps):
 *   dx[i,j] = rstd_i dy[i,j] w_j - x[i,j] rstd_i^3 (1/N) sum_k dy[i,k] w_k x[i,k]
 *   dw[j]   = sum_i dy[i,j] x[i,j] rstd_i          (overwritten, not accumulated)
 *   x, dy  [M, N] dtype;  w [N] dtype;  rstd [M] float32 from qk_rmsnorm_fwd.
 *   dx     [M, N] dtype, written once; may alias x or dy exactly.
 *   dw     [N] float32.
 *   workspace  caller-owned device memory of at least
 *              qk_rmsnorm_bwd_workspace_size() bytes, 16-byte aligned; its
 *              contents are scratch (no need to clear it).  dw is summed from
 *              the per-CTA partials in a fixed order, so it is reproducible.
 */
QK_API qk_status qk_rmsnorm_bwd(const void* x, const void* w, const float* rstd, const void* dy,
                                void* dx, float* dw, void* workspace, size_t workspace_bytes,
                                int64_t M, int64_t N, qk_dtype dtype, void* stream);

/*
 * RMSNorm backward that allocates nothing.  (No counterpart in the article:
 * this is an interface variant of qk_rmsnorm_bwd for callers that cannot
 * allocate device memory -- code running under a device-memory budget that
 * was reserved up front, hooks that a host framework hands only tensors and a
 * stream, or code that must avoid the implicit device synchronisation that
 * cudaMalloc / cudaFree may cause.)
 *
 * Same arguments, results and aliasing rules as qk_rmsnorm_bwd, without the
 * workspace: the dw partial sums go to a fixed 16 MiB array in the library's
 * own device memory, which every GPU that loads the library's device code
 * holds until the process exits.  Calls whose workspace need
 * (qk_rmsnorm_bwd_workspace_size) exceeds 16 MiB return QK_ERR_UNSUPPORTED.
 *
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.  The
 * address is kept for the life of the process: after a cudaDeviceReset() of
 * that device it is stale, so do not call this entry point on a device that
 * was reset after its first call (see the per-device state note at the top).
 * Every call on a device shares the one array: calls whose kernels overlap on
 * the GPU (for example on two streams) race on it and must be serialised by
 * the caller.  Nothing in it needs clearing between calls: each call writes
 * every partial it later reads.  No cudaMalloc, cudaFree or other allocating
 * routine is called.
 */
QK_API qk_status qk_rmsnorm_bwd_noalloc(const void* x, const void* w, const float* rstd,
                                        const void* dy, void* dx, float* dw, int64_t M, int64_t N,
                                        qk_dtype dtype, void* stream);

/*
 * Cross-entropy backward: dlogits[i,j] = dloss_i * (exp(logits[i,j] - lse_i) - [j == t_i]).
 *   logits [M, N] dtype; targets [M] int64; lse [M] float32 from qk_xent_fwd;
 *   dloss  [M] float32 upstream gradient of each row's loss, or NULL for 1.
 *   dlogits [M, N] dtype, written once; may alias logits exactly.  A row whose
 *   target is outside [0, N) gets NaN gradients.
 */
QK_API qk_status qk_xent_bwd(const void* logits, const int64_t* targets, const float* lse,
                             const float* dloss, void* dlogits, int64_t M, int64_t N,
                             qk_dtype dtype, void* stream);

/*
 * Cross-entropy variants.  Options of qk_xent_fwd_ex / qk_xent_bwd_ex (NULL
 * means the plain operator: no ignore index, no z-loss):
 *   has_ignore_index  nonzero: rows whose target equals ignore_index get loss 0
 *                     and zero gradient and are left out of the mean.  Zero:
 *                     no row is ignored, and every target outside [0, N) --
 *                     INT64_MIN and INT64_MAX included -- gives NaN as in
 *                     qk_xent_fwd; ignore_index is then not read.
 *   ignore_index      the target value of ignored rows (any int64).
 *   z_loss            coefficient z of the term z * lse^2 added to each row's
 *                     loss (a penalty on the log-partition function; 0: none).
 * The article names cross-entropy loss only; these are the common training
 * variants of the same per-row definition, added in its epilogue.
 */
typedef struct {
  int32_t has_ignore_index;
  float z_loss;
  int64_t ignore_index;
} qk_xent_options;

/*
 * loss[i] = lse[i] - x[i, t_i] + z * lse[i]^2 (0 on ignored rows, NaN for a
 * target outside [0, N) that is not ignored); lse as in qk_xent_fwd.
 * mean_loss (may be NULL): one float32, the mean of loss over the rows that
 * are not ignored, summed in a fixed order (NaN when every row is ignored).
 * It must not overlap the other buffers.
 */
QK_API qk_status qk_xent_fwd_ex(const void* logits, const int64_t* targets, float* loss, float* lse,
                                float* mean_loss, int64_t M, int64_t N, qk_dtype dtype,
                                const qk_xent_options* options, void* stream);

/*
 * dlogits[i,j] = dloss_i * ((1 + 2 z lse_i) * exp(x[i,j] - lse_i) - [j == t_i]),
 * zero on ignored rows; otherwise as qk_xent_bwd.  For the gradient of the
 * mean, pass dloss_i = 1 / (number of rows not ignored).
 */
QK_API qk_status qk_xent_bwd_ex(const void* logits, const int64_t* targets, const float* lse,
                                const float* dloss, void* dlogits, int64_t M, int64_t N,
                                qk_dtype dtype, const qk_xent_options* options, void* stream);

/* Static English description of a status code; never NULL. */
QK_API const char* qk_status_string(qk_status s);

/*
 * Synchronises `stream`, then reads and clears the calling device's status
 * word.  Returns QK_OK when no kernel has reported a failure since the last
 * call, or the first failure recorded (QK_ERR_TIMEOUT).  A CUDA error from the
 * synchronisation itself is returned as QK_ERR_LAUNCH.
 */
QK_API qk_status qk_get_device_status(void* stream);

/* Largest N the operator accepts for `dtype` (rows longer than this return
 * QK_ERR_UNSUPPORTED).  The forward operators stream rows of any length on the
 * aligned path (INT64_MAX): softmax and RMSNorm rows longer than 1 MiB are read
 * twice (three HBM passes instead of two) -- only on the masked path, for
 * unaligned rows, are softmax and RMSNorm limited to 524,288 elements.  The
 * backward passes of softmax and RMSNorm hold rows of up to 512 KiB. */
QK_API int64_t qk_max_row_elements(qk_op op, qk_dtype dtype);

/*
 * Launch plan: how a call maps onto the GPU.  Reported by qk_get_plan() for
 * logging and benchmarks; qk_set_plan_override() pins one for tuning sweeps.
 *
 *   path            1 = TMA ring (aligned fast path), 2 = masked direct path,
 *                   3 = backward ring, 4 = two-pass ring (rows beyond 1 MiB;
 *                   an override with path 4 forces it for any row),
 *                   5 = masked backward, 6 = shifted ring (unaligned rows).
 *   threads         threads per CTA.
 *   row_threads     threads that share one row inside a CTA (rows per CTA
 *                   step = threads / row_threads).
 *   vec_per_thread  16-byte vectors each thread holds per row (or per chunk
 *                   for streamed rows); elements per thread on the masked path.
 *   cluster         CTAs of a thread-block cluster that split one row
 *                   (1 = no cluster); partial results meet in DSMEM.
 *   slots           shared-memory ring slots per CTA (TMA loads in flight).
 *   chunks          ring slots one row slice spans (> 1 only for streamed rows).
 *   ctas_per_sm     resident CTAs per SM the launch was sized for.
 *   grid            CTAs launched (persistent: each loops over its share).
 *   smem_bytes      dynamic shared memory per CTA.
 */
typedef struct {
  int32_t path;
  int32_t threads;
  int32_t row_threads;
  int32_t vec_per_thread;
  int32_t cluster;
  int32_t slots;
  int32_t chunks;
  int32_t ctas_per_sm;
  int32_t grid;
  int32_t smem_bytes;
} qk_plan;

/*
 * Fills *plan with what a call with these sizes would launch on the current
 * device (aligned pointers assumed).  Returns QK_ERR_UNSUPPORTED for rows that
 * are too long and QK_ERR_INVALID_ARG for bad sizes.
 */
QK_API qk_status qk_get_plan(qk_op op, qk_dtype dtype, int64_t M, int64_t N, qk_plan* plan);

/*
 * Tuning hook: every later aligned-path call of (op, dtype) uses `plan`'s
 * threads, row_threads, vec_per_thread, cluster, slots and chunks instead of
 * the built-in table (chunks and ctas_per_sm are recomputed; a zero slots
 * field keeps the table's rule; a positive grid caps the number of CTAs, which
 * makes each CTA walk more rows -- a test of the ring's reuse).  plan == NULL removes the override.
 * Returns QK_ERR_UNSUPPORTED when no compiled kernel matches the triple
 * (threads, row_threads, vec_per_thread).  Process-wide, not thread-safe
 * against concurrent calls of the same operator.
 */
QK_API qk_status qk_set_plan_override(qk_op op, qk_dtype dtype, const qk_plan* plan);

/*
 * Test hook for the device-side failure path.  Enqueues one CTA that waits on
 * a shared-memory barrier nobody completes, bounded by `timeout_ns`; when the
 * bound runs out the kernel records QK_ERR_TIMEOUT in the device status word
 * and returns normally (no trap, no fault).  qk_get_device_status() then
 * reports it.  timeout_ns must be in (0, 10 s].
 */
QK_API qk_status qk_test_wait_timeout(uint64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QK_H_ */
