/*
 * rnnt_gb300.h -- C ABI of the fused RNN-T (transducer) loss for GB300 (sm_103a).
 *
 * One call computes, for a batch of B utterances, the per-sample RNN-T loss
 * (negative log-likelihood summed over every alignment) and, optionally, its
 * gradient with respect to the joiner logits, with the semantics of
 * torchaudio.functional.rnnt_loss.  The operation and its arguments are the
 * ones of the rnnt-loss-ascend README ("optimized_transducer"):
 *   - section 参数说明 (parameter table): compact 2D logits, int32 targets and
 *     lengths, blank, clamp, fused_log_softmax, per-sample loss, grad with
 *     the shape of the logits;
 *   - section 约束说明 (constraints): float32/float16 logits (bfloat16 added
 *     here), blank in
 *     [-V, V-1] with -1 meaning V-1, sum of T_b*(U_b+1) equal to the number
 *     of logit rows, clamp <= 0 meaning no clipping;
 *   - section 架构设计 (architecture): a two-phase interface, workspace size
 *     first, then the fused launch;
 *   - section 核心梯度融合公式 / 精度保证: the gradient formula and the check that
 *     the alpha-side and beta-side losses agree.
 * Status codes follow the RNNTStatus convention of the ESPnet GPURNNT docs
 * (cost_and_grad returns success or RNNT_STATUS_INVALID_VALUE).
 *
 * Memory and streams: every pointer argument named "device" must point to
 * memory the current CUDA device can access.  The library allocates nothing
 * and keeps no state between calls other than per-device kernel attributes
 * (and, for rnnt_loss_fused_noalloc, its fixed scratch array); all work is
 * enqueued on `stream` and the host never synchronises.
 */
#ifndef RNNT_GB300_H
#define RNNT_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *rnnt_stream_t;

typedef enum {
    RNNT_OK = 0,
    RNNT_INVALID_VALUE = 1,       /* bad argument (host) or bad lengths/targets (device) */
    RNNT_WORKSPACE_TOO_SMALL = 2, /* workspace_bytes below rnnt_workspace_size()         */
    RNNT_LAUNCH_FAILED = 3,       /* a kernel launch returned a CUDA error               */
    RNNT_LOSS_MISMATCH = 4,       /* alpha-side and beta-side losses disagree (or NaN)   */
    RNNT_TIMEOUT = 5              /* a bounded device wait gave up                       */
} rnnt_status_t;

/* Storage type of the logits and the gradient (arithmetic is float32 for
 * every type; bfloat16 is this library's addition to the README's
 * float32/float16). */
typedef enum { RNNT_F32 = 0, RNNT_F16 = 1, RNNT_BF16 = 2 } rnnt_dtype_t;

typedef enum { RNNT_RED_NONE = 0, RNNT_RED_SUM = 1, RNNT_RED_MEAN = 2 } rnnt_reduction_t;

/* Largest supported target length (U_b <= RNNT_MAX_TARGET_LENGTH, so a lattice
 * is at most 1024 nodes wide). */
#define RNNT_MAX_TARGET_LENGTH 1023

/*
 * rnnt_workspace_size -- bytes of device scratch rnnt_loss_fused needs.
 * README 架构设计, first phase of the two-phase interface.
 *   B     number of samples (>= 1)
 *   rows  number of logit rows, sum over b of T_b*(U_b+1) (>= 1)
 *   V     vocabulary size including blank (>= 1)
 *   dt    logit element type
 *   bytes out: required size; about 36 bytes per logit row plus O(B).
 * Returns RNNT_INVALID_VALUE for a NULL `bytes` or out-of-range sizes.
 */
rnnt_status_t rnnt_workspace_size(int32_t B, int64_t rows, int32_t V, rnnt_dtype_t dt,
                                  size_t *bytes);

/*
 * rnnt_loss_fused -- loss and gradient of a batch in one call (README 架构设计,
 * second phase; 参数说明 for the arguments).
 *
 *   logits            device, (rows, V) row-major contiguous, dt.  Sample b owns
 *                     rows [off_b, off_b + T_b*(U_b+1)), off_b = sum_{i<b}
 *                     T_i*(U_i+1); inside a sample, row t*(U_b+1)+u holds the
 *                     joiner output for frame t after u emitted labels.
 *                     Must be 16-byte aligned.  Raw logits when
 *                     fused_log_softmax != 0, log-probabilities otherwise.
 *   targets           device int32, (B, targets_stride) row-major; row b holds
 *                     the U_b labels of sample b followed by ignored padding.
 *                     Labels must lie in [0, V) and differ from blank.
 *   targets_stride    1 <= targets_stride <= RNNT_MAX_TARGET_LENGTH, and
 *                     >= max_b U_b.
 *   logit_lengths     device int32 [B], T_b >= 1.
 *   target_lengths    device int32 [B], 0 <= U_b <= targets_stride.
 *   B                 batch size >= 1.
 *   blank             in [-V, V-1]; a negative value counts from the end.
 *   clamp             > 0 clips every gradient element to [-clamp, clamp]
 *                     before the reduction scale; <= 0 disables clipping.
 *   fused_log_softmax nonzero: the kernel applies log-softmax to each row.
 *   reduction         NONE / SUM / MEAN (mean over the batch).  It sets the
 *                     gradient scale (1/B for MEAN, else 1) and loss_reduced.
 *   loss              device float [B], required: per-sample loss.
 *   loss_reduced      device float [1] or NULL: sum (SUM, NONE) or mean (MEAN).
 *   grad              device (rows, V) in dt, or NULL for loss only.  It may
 *                     equal `logits` (the gradient then overwrites the
 *                     logits in place) but must not partly overlap it.  Must
 *                     be 16-byte aligned.
 *   workspace         device scratch of at least rnnt_workspace_size() bytes,
 *                     256-byte aligned, owned by the caller; it may be reused
 *                     by later calls on the same stream once this one is
 *                     enqueued (contents are rewritten every call).
 *   status_dev        device int32 [1] or NULL.  Receives RNNT_OK,
 *                     RNNT_INVALID_VALUE (device-detected: a T_b < 1, a U_b
 *                     out of range, a label out of range or equal to blank,
 *                     or rows != sum T_b*(U_b+1)) or RNNT_LOSS_MISMATCH
 *                     (alpha/beta losses differ by more than
 *                     1e-3*max(1,|loss|), or a loss is not finite).  When it
 *                     is not RNNT_OK, loss/grad contents are unspecified.
 *   stream            CUDA stream all kernels are enqueued on.
 *
 * Host-side return value: RNNT_INVALID_VALUE for NULL required pointers, bad
 * sizes/enums/blank, misaligned or partly overlapping buffers;
 * RNNT_WORKSPACE_TOO_SMALL; RNNT_LAUNCH_FAILED if a launch fails.  Nothing is
 * enqueued when a host-side check fails.
 */
rnnt_status_t rnnt_loss_fused(const void *logits, rnnt_dtype_t dt, int64_t rows, int32_t V,
                              const int32_t *targets, int32_t targets_stride,
                              const int32_t *logit_lengths, const int32_t *target_lengths,
                              int32_t B, int32_t blank, float clamp, int32_t fused_log_softmax,
                              rnnt_reduction_t reduction, float *loss, float *loss_reduced,
                              void *grad, void *workspace, size_t workspace_bytes,
                              int32_t *status_dev, rnnt_stream_t stream);

/*
 * Options of rnnt_loss_fused_ex.  A zero-initialised struct (or a NULL
 * pointer) gives the behaviour of rnnt_loss_fused.
 *
 *   fastemit_lambda   >= 0.  FastEmit weight (the fastemit_lambda argument of
 *                     the ESPnet GPURNNT docs and of compute_multiblank_grad_kernel,
 *                     after the FastEmit paper they cite): the gradient term of
 *                     every label-emission log-probability is multiplied by
 *                     1 + fastemit_lambda; blank terms and the loss are not
 *                     changed.  0 is the plain transducer gradient.
 *   padded            0: compact layout (rows = sum_b T_b*(U_b+1)).
 *                     1: padded layout of the GPURNNT docs (the activation
 *                     tensor of cost_and_grad, shape [B, T, U, V+1]; also the
 *                     torchaudio.functional.rnnt_loss layout): logits and grad are
 *                     (B, max_T, max_U + 1, V) row-major, rows must equal
 *                     B*max_T*(max_U+1), node (t, u) of sample b is row
 *                     (b*max_T + t)*(max_U+1) + u.  Rows outside a sample's
 *                     lattice (t >= T_b or u > U_b) are never read and get a
 *                     zero gradient.  T_b <= max_T and U_b <= max_U are
 *                     checked on the device (RNNT_INVALID_VALUE).
 *   max_T, max_U      padded layout only: max_T >= 1, 0 <= max_U <=
 *                     RNNT_MAX_TARGET_LENGTH, max_T*(max_U+1) < 2^31.
 *   num_big_blanks    0..RNNT_MAX_BIG_BLANKS.  Multi-blank transducer (ESPnet
 *                     compute_multiblank_grad_kernel docs and the multi-blank
 *                     paper they cite): besides `blank` (one frame), big blank
 *                     i is output big_blank_ids[i] (in [-V, V-1], negative
 *                     counting from the end; distinct, not blank, never a
 *                     label) and advances big_blank_durations[i] frames
 *                     (2..RNNT_MAX_BIG_BLANK_DURATION).  A path ends when a
 *                     blank-type step reaches frame T with every label
 *                     emitted; no step passes frame T.
 *   sigma             >= 0.  Logit under-normalisation of the same docs:
 *                     subtracted from every log-probability the lattice uses.
 *                     With num_big_blanks == 0 and sigma == 0 the call is the
 *                     standard transducer loss; otherwise it runs the
 *                     multi-blank kernels (workspace: rnnt_workspace_size_ex).
 */
#define RNNT_MAX_BIG_BLANKS 8
#define RNNT_MAX_BIG_BLANK_DURATION 16
typedef struct {
    float fastemit_lambda;
    int32_t padded;
    int32_t max_T;
    int32_t max_U;
    int32_t num_big_blanks;
    int32_t big_blank_ids[RNNT_MAX_BIG_BLANKS];
    int32_t big_blank_durations[RNNT_MAX_BIG_BLANKS];
    float sigma;
} rnnt_options_t;

/*
 * rnnt_workspace_size_ex -- workspace bytes of rnnt_loss_fused_ex with these
 * options (NULL: as rnnt_workspace_size).  The multi-blank kernels need 8
 * more bytes per big blank and lattice node.  RNNT_INVALID_VALUE as
 * rnnt_workspace_size, or for num_big_blanks outside 0..RNNT_MAX_BIG_BLANKS.
 */
rnnt_status_t rnnt_workspace_size_ex(int32_t B, int64_t rows, int32_t V, rnnt_dtype_t dt,
                                     const rnnt_options_t *options, size_t *bytes);

/*
 * rnnt_loss_fused_ex -- rnnt_loss_fused with options (FastEmit, padded
 * layout).  Same arguments, results and errors as rnnt_loss_fused, plus
 * `options` (NULL = defaults); RNNT_INVALID_VALUE for a negative or
 * non-finite fastemit_lambda or sigma, inconsistent padded sizes or invalid
 * big blanks.  The workspace is sized by rnnt_workspace_size_ex(B, rows, V,
 * dt, options) with the same `rows`.
 */
rnnt_status_t rnnt_loss_fused_ex(const void *logits, rnnt_dtype_t dt, int64_t rows, int32_t V,
                                 const int32_t *targets, int32_t targets_stride,
                                 const int32_t *logit_lengths, const int32_t *target_lengths,
                                 int32_t B, int32_t blank, float clamp, int32_t fused_log_softmax,
                                 rnnt_reduction_t reduction, float *loss, float *loss_reduced,
                                 void *grad, void *workspace, size_t workspace_bytes,
                                 int32_t *status_dev, rnnt_stream_t stream,
                                 const rnnt_options_t *options);

/*
 * rnnt_loss_fused_staged -- rnnt_loss_fused with stage timing (tracing aid).
 * Same arguments, plus stage_events: NULL, or an array of 7 cudaEvent_t
 * handles (entries may be NULL) that the call records on `stream` at its
 * stage boundaries: [0] start, [1] after offsets/schedule, [2] after the
 * row pass, [3] after the alpha/beta DP, [4] = [3] (the per-row gradient
 * coefficients are formed inside the gradient pass), [5] after the gradient
 * pass (whose last CTA also runs the loss check/reduction), [6] at the end.
 * A call that runs as one persistent kernel records [1]..[6] after it.
 * The caller creates and owns the events.
 */
rnnt_status_t rnnt_loss_fused_staged(const void *logits, rnnt_dtype_t dt, int64_t rows, int32_t V,
                                     const int32_t *targets, int32_t targets_stride,
                                     const int32_t *logit_lengths, const int32_t *target_lengths,
                                     int32_t B, int32_t blank, float clamp,
                                     int32_t fused_log_softmax, rnnt_reduction_t reduction,
                                     float *loss, float *loss_reduced, void *grad, void *workspace,
                                     size_t workspace_bytes, int32_t *status_dev,
                                     rnnt_stream_t stream, void *const *stage_events);

/*
 * rnnt_grad_scale -- multiply a gradient produced by rnnt_loss_fused by the
 * upstream gradient of the loss (the autograd backward step the README's
 * Python layer performs, section 架构设计 "Python 层").
 *   grad, dt, rows, V   the gradient buffer of a previous rnnt_loss_fused call
 *   B                   batch size of that call
 *   workspace           the workspace of that call, unmodified since (its
 *                       row offsets map rows to samples)
 *   factors             device float: factors[0] for the whole gradient
 *                       (per_sample == 0) or factors[b] for sample b's rows
 *                       (per_sample != 0).  Rows whose factor is exactly 1
 *                       are left untouched (no memory traffic).
 * The layout (compact or padded) is the one of that call; `rows` is the
 * gradient's row count passed to it.
 * Returns RNNT_INVALID_VALUE / RNNT_WORKSPACE_TOO_SMALL / RNNT_LAUNCH_FAILED
 * as rnnt_loss_fused does.
 */
rnnt_status_t rnnt_grad_scale(void *grad, rnnt_dtype_t dt, int64_t rows, int32_t V, int32_t B,
                              const void *workspace, size_t workspace_bytes,
                              const float *factors, int32_t per_sample, rnnt_stream_t stream);

/*
 * rnnt_plan -- how rnnt_loss_fused / rnnt_loss_fused_ex would run a call of
 * this shape on the current device, without running it (a planning and
 * measurement aid; no counterpart on the pages, whose README promises one
 * kernel launch per call, 价值说明 "Kernel 启动次数").
 *   B, rows, V, dt, targets_stride, fused_log_softmax   as for the call
 *   want_grad   nonzero when the call will pass a gradient buffer
 *   options     as for rnnt_loss_fused_ex, or NULL
 *   plan        out: persistent = 1 when one cooperative kernel runs the
 *               whole call (preparation, rows, recursions, gradient, check),
 *               0 for one kernel per stage; launches = kernels the call
 *               enqueues.
 * The call itself takes the per-stage kernels instead if the device
 * refuses the cooperative launch at that time.  Returns RNNT_INVALID_VALUE
 * for bad sizes, RNNT_LAUNCH_FAILED when no device is current.
 */
typedef struct {
    int32_t persistent;
    int32_t launches;
} rnnt_plan_t;

rnnt_status_t rnnt_plan(int32_t B, int64_t rows, int32_t V, rnnt_dtype_t dt,
                        int32_t targets_stride, int32_t fused_log_softmax, int32_t want_grad,
                        const rnnt_options_t *options, rnnt_plan_t *plan);

/*
 * rnnt_set_trace -- task tracing (a debugging aid; process-wide setting, not
 * thread-safe).  While a buffer is set, every rnnt_loss_fused call writes
 * records int4 {kind | sample << 2, SM id, start ns, end ns} (kind 0: row
 * chunk, 1: alpha/beta recursions of a sample, 2: gradient chunk; times
 * relative to the start of the call's preparation) at indices below
 * bytes/16.  A call that runs as one persistent kernel records every task:
 * for each sample (longest DP first) its row chunks, then every gradient
 * chunk (record = task index), and sample b's recursions at index
 * (task count + b).  A call on the per-stage kernels records the recursions
 * only: the forward and backward recursion of the i-th sample in DP order at
 * indices 2i and 2i + 1.  device_buffer must be 16-byte aligned
 * device memory that outlives the calls; NULL (or bytes < 16) turns tracing
 * off.
 */
rnnt_status_t rnnt_set_trace(void *device_buffer, size_t bytes);

/* Size of the fixed device scratch array rnnt_loss_fused_noalloc uses: 32 MiB,
 * enough for rnnt_workspace_size() up to about 900,000 logit rows. */
#define RNNT_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * rnnt_loss_fused_noalloc -- rnnt_loss_fused for callers that cannot hand
 * out device memory.  The paper has no counterpart: this is an interface of
 * this library only.
 *
 * Same arguments and results as rnnt_loss_fused without workspace and
 * workspace_bytes.  The scratch is a file-scope device array of
 * RNNT_NOALLOC_SCRATCH_BYTES bytes inside this library, one per device; the
 * call allocates nothing (no cudaMalloc/cudaFree, no allocating library
 * routine).  The first call on a device, made with that device current,
 * looks up the array's device address (cudaGetSymbolAddress) once and
 * caches it; make that first call before any stream capture.  The cached
 * address is that of the device's primary context at the time: a process
 * that destroys it (cudaDeviceReset) must not call this entry point on that
 * device afterwards.
 *
 * Every call on a device shares the one array and leaves its contents
 * behind; each call rewrites everything it reads before reading it.  Calls
 * whose kernels overlap on the GPU (other streams, other host threads)
 * race on the array and give undefined results: serialize them, e.g. on
 * one stream.  rnnt_grad_scale, which reads a caller workspace, does not
 * apply to this call's gradient.
 *
 * Returns RNNT_WORKSPACE_TOO_SMALL, before any device work, when
 * rnnt_workspace_size(B, rows, V, dt) exceeds RNNT_NOALLOC_SCRATCH_BYTES;
 * RNNT_LAUNCH_FAILED when the address lookup fails; otherwise what
 * rnnt_loss_fused returns.
 */
rnnt_status_t rnnt_loss_fused_noalloc(const void *logits, rnnt_dtype_t dt, int64_t rows,
                                      int32_t V, const int32_t *targets, int32_t targets_stride,
                                      const int32_t *logit_lengths,
                                      const int32_t *target_lengths, int32_t B, int32_t blank,
                                      float clamp, int32_t fused_log_softmax,
                                      rnnt_reduction_t reduction, float *loss,
                                      float *loss_reduced, void *grad, int32_t *status_dev,
                                      rnnt_stream_t stream);

/*
 * rnnt_selftest_wait_timeout -- diagnostic of the bounded device waits (no
 * counterpart on the pages).  Enqueues one kernel whose warp waits, with the
 * same helper the loss kernels use for their shared-memory row copies, on a
 * barrier that nothing completes; after `polls` (>= 1) polls the wait gives
 * up, and status_dev (device int32) receives RNNT_TIMEOUT, as a loss call's
 * status would.  Nothing faults, traps or stays in flight; the context stays
 * usable.  Returns RNNT_INVALID_VALUE (NULL status_dev, polls < 1) or
 * RNNT_LAUNCH_FAILED.
 */
rnnt_status_t rnnt_selftest_wait_timeout(int32_t *status_dev, int32_t polls, rnnt_stream_t stream);

/* Static English description of a status code. */
const char *rnnt_status_string(rnnt_status_t status);

/* ABI version of this header (major * 100 + minor). */
int32_t rnnt_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RNNT_GB300_H */
