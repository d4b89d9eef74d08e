/*
 * vce.h -- C ABI of the GB300 vocabulary cross-entropy library (libvce.so).
 *
 * Softmax cross-entropy over a [T, V] logits matrix that stays accurate at large
 * target margins, its gradient, the merge of vocabulary-chunked statistics, and a
 * fused linear cross-entropy (declared in vce_linear.h), as hand-written sm_103a
 * CUDA kernels.
 *
 * Sources of the operations (the web pages this library restates):
 *   [TT]  torchtitan PR #5723, "[loss] fix softmax collapse with improved ce perf":
 *         Numerics (target-excluded log-sum-exp and softplus NLL; the p_t = 1/4
 *         branch of the target gradient; ignored labels), Memory/perf (the
 *         compiled form: column mask, one read of the logits in forward, per-row
 *         statistics saved, the gradient rebuilt in one fused backward pass;
 *         bf16 input upcast inside the op).
 *   [MC]  Megatron-core API docs, core.tensor_parallel.cross_entropy:
 *         vocab_parallel_cross_entropy(vocab_parallel_logits, target,
 *         label_smoothing, tp_group) and the VocabParallelCrossEntropy helpers
 *         (calculate_logits_max, gather_predicted_logits: target mask, local
 *         target ids, predicted logit zero for targets owned elsewhere).
 *   [CCE] apple/ml-cross-entropy issue #14: linear_cross_entropy(e, c, targets)
 *         (classifier weight only, no bias), impl="cce_exact" (no gradient
 *         filtering) and use_kahan (compensated accumulation of dc and de).
 *
 * Conventions common to every call:
 *   - Every pointer is a DEVICE pointer owned by the caller unless stated "host".
 *     The library allocates and frees nothing; scratch space is an explicit
 *     caller-provided workspace where a call needs one.
 *   - Every call only enqueues work on the caller's stream `s` and returns; it
 *     never synchronises.  Inputs must stay valid until that work has run.
 *   - Logits are read only (const): the input is never written [TT, Memory/perf].
 *   - Matrices are row-major with a leading dimension `ld` (elements between the
 *     starts of consecutive rows, ld >= number of columns).  Rows need not be
 *     16-byte aligned; 16-byte aligned rows take the vectorised path.
 *   - Labels are int64.  A label equal to ignore_index marks an ignored row: its
 *     loss and gradient are exactly +0.0, whatever its logits hold (even +-inf).
 *     Any other label outside [0, V) is an error: the device writes VCE_ERR_LABEL
 *     into *status, that row's loss becomes NaN (and so does a reduced loss), its
 *     gradient is 0.  No call traps or asserts on the device.
 *   - Per-row losses and reduced losses are fp32 whatever the logits dtype.
 *   - Return value: VCE_OK, or a negative host-detected error (nothing was
 *     enqueued in that case).  Device-detected errors go to *status; read it after
 *     the stream has run (vce_get_status does that).  *status need not be cleared
 *     before a call: every call writes it.
 *   - The stage-ring kernels of ce_forward, ce_backward and ce_forward_backward
 *     share a launch slot of device words across their CTAs (dynamic row claims,
 *     the count of finished CTAs, the first error code), taken round-robin from
 *     1024 slots per kernel file and left zero by the launch's last CTA.  At most
 *     1024 launches of one of these kernels may therefore be in flight at once,
 *     across all streams and host threads of a process (a graph replays the slot
 *     it was captured with: do not run one graph's replays concurrently).
 */
#ifndef VCE_H
#define VCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* vce_stream_t; /* the same handle as cudaStream_t; NULL = legacy stream */

#define VCE_ABI_VERSION 1
#define VCE_ROW_STATS 4     /* floats per row of row_stats */
#define VCE_CHUNK_STATS 4   /* floats per (chunk, row) of chunk statistics */
#define VCE_MAX_CHUNKS 64   /* most column chunks ce_merge_chunks accepts */
#define VCE_NOALLOC_MAX_CHUNK_ROWS 262144   /* most k * T for ce_merge_chunks_noalloc (4 MiB) */

/* Exported entry points (the library is built with hidden symbol visibility otherwise). */
#if defined(__GNUC__)
#define VCE_API __attribute__((visibility("default")))
#else
#define VCE_API
#endif

typedef enum { VCE_F32 = 0, VCE_BF16 = 1 } vce_dtype;
typedef enum { VCE_RED_NONE = 0, VCE_RED_SUM = 1, VCE_RED_MEAN = 2 } vce_reduction;

enum {
    VCE_OK = 0,
    VCE_ERR_LABEL = 1,        /* device-detected: a label neither ignore_index nor in [0, V) */
    VCE_ERR_NULL = -1,        /* a required pointer is NULL */
    VCE_ERR_DTYPE = -2,       /* unknown or unsupported dtype / reduction */
    VCE_ERR_SHAPE = -3,       /* a size is negative, zero where it must not be, or overflows */
    VCE_ERR_LD = -4,          /* a leading dimension is smaller than the row length */
    VCE_ERR_ALIGN = -5,       /* a pointer is not aligned to its element size (16 B for stats) */
    VCE_ERR_WORKSPACE = -6,   /* workspace missing or smaller than required */
    VCE_ERR_CUDA = -7,        /* a CUDA runtime call failed (launch, memset, attribute query) */
    VCE_ERR_ARG = -8,         /* any other invalid argument (chunk count, chunk layout) */
    VCE_ERR_DEVICE = -9,      /* the current device is not an sm_100-family GPU */
    VCE_ERR_SCRATCH_LIMIT = -10 /* k * T exceeds VCE_NOALLOC_MAX_CHUNK_ROWS (ce_merge_chunks_noalloc) */
};

/* Library ABI version (VCE_ABI_VERSION of the build). */
VCE_API int vce_abi_version(void);

/* Static text for a status code; never NULL. */
VCE_API const char* vce_status_string(int status);

/* Floats per row of the row_stats buffer (= VCE_ROW_STATS). */
VCE_API size_t vce_row_stats_floats(void);

/*
 * Waits for stream `s`, then copies the device status word to *host_out.
 * Returns VCE_OK or VCE_ERR_CUDA / VCE_ERR_NULL.
 */
VCE_API int vce_get_status(const int32_t* status, vce_stream_t s, int32_t* host_out);

/*
 * vce_last_cuda_error -- the cudaError_t behind the most recent VCE_ERR_CUDA an entry point
 * returned on the calling host thread (0 if none), then cleared; vce_cuda_error_name gives
 * its name.  No page counterpart: a diagnostic.
 */
VCE_API int vce_last_cuda_error(void);
VCE_API const char* vce_cuda_error_name(int code);

/*
 * vce_debug_checks -- 1 if this library was built with device-side index checks
 * (python -m vocab_cross_entropy_gb300.build --debug-checks, which makes libvce_debug.so),
 * else 0.  No page counterpart: a debugging aid.
 */
VCE_API int vce_debug_checks(void);

/*
 * vce_debug_status -- in a build with device-side index checks: waits for the device
 * (cudaDeviceSynchronize), then writes to *host_out the code of the first index check that
 * failed since the last call (121 a row outside [0, T); 122 a column range outside its row
 * or chunk; 123 a chunk or segment index outside its table; 124 a stage or ring slot
 * outside the ring; 125 a GEMM output tile outside the output), or 0, and clears the record.
 * A kernel whose check fails skips that access (it never traps), so its outputs are then
 * incomplete.  In the release build it writes 0 and waits for nothing.  Returns VCE_OK,
 * VCE_ERR_NULL or VCE_ERR_CUDA.  No page counterpart: a debugging aid.
 */
VCE_API int vce_debug_status(int32_t* host_out);

/*
 * ce_forward -- per-row NLL and the statistics its gradient needs.  [TT, Numerics;
 * Memory/perf, compiled forward]  For row i with label t:
 *     L'_i = log sum_{j != t} exp(z_ij)          (target left out by a column test)
 *     x_i  = L'_i - z_it
 *     loss_rows[i] = softplus(x_i) = -log softmax(z_i)_t
 * in one read of the row (running max and rescaled sum-exp), fp32 arithmetic on
 * bf16 or fp32 input.  Reduction SUM writes sum_i loss_i to *loss_out; MEAN writes
 * that sum divided by N, the number of non-ignored rows (NaN when N = 0), summed
 * in a fixed order (bitwise reproducible); NONE leaves loss_out untouched (may be NULL).
 *
 *   logits     [T, ld] of dtype `dt` (VCE_F32 or VCE_BF16), element-aligned
 *   T, V, ld   rows, vocabulary size (>= 1), leading dimension (>= V); T may be 0
 *   labels     [T] int64;  ignore_index: label value of ignored rows (e.g. -100)
 *   loss_rows  [T] fp32, written
 *   loss_out   [1] fp32, written for SUM / MEAN
 *   row_stats  [T * VCE_ROW_STATS] fp32, 16-byte aligned, written; per row
 *              (L', sigmoid(x) = 1 - p_t, target-gradient coefficient, row weight).
 *              The target coefficient is p_t - 1 when p_t < 1/4 (x > ln 3), else
 *              -(1 - p_t) [TT, Numerics].  The row weight is 1/N (MEAN), 1 (SUM,
 *              NONE) or 0 (ignored / invalid row).  Consumed by ce_backward.
 *   status     [1] int32, set to 0 by this call, VCE_ERR_LABEL on a bad label, or
 *              105 / 106 / 108 / 110 when a bounded device-side wait gave up after 2 s
 *              (rows longer than 32 KB made of 16-byte vectors stream through a
 *              shared-memory stage ring: free stage, loaded stage, warp partials, free
 *              statistics slots; shorter rows take one warp per row and other layouts
 *              one block per row, which have no such waits), 112 when the ring's wait
 *              for the batch's label count gave up (SUM / MEAN, at most 65536 rows: the
 *              ring then reduces the losses itself), or 111 if the ring's consumer
 *              groups were given rows longer than two stages (not reachable from this
 *              call); the outputs are then undefined
 */
VCE_API int ce_forward(const void* logits, vce_dtype dt, int64_t T, int64_t V, int64_t ld,
               const int64_t* labels, int64_t ignore_index, vce_reduction red,
               float* loss_rows, float* loss_out, float* row_stats, int32_t* status,
               vce_stream_t s);

/*
 * ce_backward -- gradient of the reduced loss w.r.t. the logits, rebuilt in one
 * pass from the logits and row_stats.  [TT, Numerics; Memory/perf, compiled backward]
 *     grad_ij = c_i * exp(z_ij - L'_i) * sigmoid(x_i)          (j != t)
 *     grad_it = c_i * (p_t - 1) if p_t < 1/4, else -c_i * (1 - p_t)
 * with c_i = grad_output[0] * weight_i (SUM, MEAN) or grad_output[i] * weight_i
 * (NONE).  Ignored rows are written as +0.0.  fp32 math, bf16 output rounded to
 * nearest even.
 *
 *   logits, dt, T, V, ld, labels, ignore_index, red: as given to ce_forward
 *   row_stats    [T * VCE_ROW_STATS] from ce_forward (or ce_merge_chunks)
 *   grad_output  fp32 [1] (SUM, MEAN) or [T] (NONE)
 *   grad_logits  [T, ld_grad] of dtype grad_dt (VCE_F32 or VCE_BF16), written;
 *                it must not overlap the logits
 */
VCE_API int ce_backward(const void* logits, vce_dtype dt, int64_t T, int64_t V, int64_t ld,
                const int64_t* labels, int64_t ignore_index, vce_reduction red,
                const float* row_stats, const float* grad_output,
                void* grad_logits, vce_dtype grad_dt, int64_t ld_grad, vce_stream_t s);

/*
 * ce_forward_ls / ce_backward_ls -- ce_forward / ce_backward with label smoothing.
 * [MC, vocab_parallel_cross_entropy: label_smoothing, a factor in [0.0, 1.0), default 0]
 * The page gives the factor and its range only; the targets here are the one-hot mixed with
 * the uniform distribution over all V classes, q = (1 - eps) onehot(t) + eps / V:
 *     loss_i = (1 - eps) softplus(x_i) + eps (LSE(z_i) - mean_j z_ij)      (= -sum_j q_j log p_j)
 *     grad_ij = c_i (p_ij - eps / V),  grad_it = c_i (p_t - 1 + eps (1 - 1/V))
 * with the collapse-safe forms of softplus(x) = -log p_t and of p_t - 1 of ce_forward.  The
 * forward additionally sums each row's logits.  label_smoothing outside [0, 1) (or NaN)
 * returns VCE_ERR_ARG.  eps = 0 is exactly ce_forward / ce_backward.  Pass the same eps to
 * both calls.  Other arguments as ce_forward / ce_backward.
 */
VCE_API int ce_forward_ls(const void* logits, vce_dtype dt, int64_t T, int64_t V, int64_t ld,
                  const int64_t* labels, int64_t ignore_index, float label_smoothing,
                  vce_reduction red, float* loss_rows, float* loss_out, float* row_stats,
                  int32_t* status, vce_stream_t s);

VCE_API int ce_backward_ls(const void* logits, vce_dtype dt, int64_t T, int64_t V, int64_t ld,
                   const int64_t* labels, int64_t ignore_index, float label_smoothing,
                   vce_reduction red, const float* row_stats, const float* grad_output,
                   void* grad_logits, vce_dtype grad_dt, int64_t ld_grad, vce_stream_t s);

/*
 * ce_forward_backward -- ce_forward followed by ce_backward in one pass over the logits, for
 * callers that know grad_output when the forward runs (e.g. a mean loss seeded by 1).
 * [TT, Numerics; Memory/perf: the forward prepares the backward]  Same arguments, results
 * and per-row numerics as the two calls, with the row's sum of exponentials taken in another
 * fp32 order (so equal to the two calls up to that rounding, and bitwise reproducible from
 * run to run).  Each row is read from HBM once: where V, ld and ld_grad are multiples of 8
 * and logits and grad_logits are 16-byte aligned, a cluster of up to 8 CTAs holds the row in
 * shared memory between its two passes [MC, VocabParallelCrossEntropy: the vocabulary split
 * with a (max, sum-exp, target) exchange]; otherwise the gradient pass re-reads the row from
 * L2.  HBM moves V*e in and V*e_g out per row.  On the shared-memory path with SUM or MEAN
 * and at most 65536 rows, the kernel counts N and reduces the losses itself (the CTA that
 * finishes last sums them in a fixed order); otherwise, for MEAN, *loss_out holds 1/N while
 * the call's work runs and the mean loss when it is done.
 *
 *   logits, dt, T, V, ld, labels, ignore_index, red: as ce_forward
 *   grad_output  fp32 [1] (SUM, MEAN) or [T] (NONE), read on the device
 *   loss_rows, loss_out, row_stats: as ce_forward (row_stats carries the weights)
 *   status       as ce_forward, or 105..109 when a device-side wait of the shared-memory
 *                path gave up after 2 s (105 free stage, 106 loaded stage, 107 the cluster's
 *                row statistics, 108 the warps' partial statistics, 109 a row's gradient
 *                coefficients); the outputs are then undefined
 *   grad_logits  [T, ld_grad] of dtype grad_dt, written; must not overlap the logits
 */
VCE_API int ce_forward_backward(const void* logits, vce_dtype dt, int64_t T, int64_t V, int64_t ld,
                        const int64_t* labels, int64_t ignore_index, vce_reduction red,
                        const float* grad_output, float* loss_rows, float* loss_out,
                        float* row_stats, void* grad_logits, vce_dtype grad_dt, int64_t ld_grad,
                        int32_t* status, vce_stream_t s);

/*
 * ce_forward_backward_ls -- ce_forward_backward with label smoothing: the loss, statistics and
 * gradient of ce_forward_ls followed by ce_backward_ls (the targets q = (1 - eps) onehot(t) +
 * eps / V), in the same one pass over the logits.  label_smoothing outside [0, 1) (or NaN)
 * returns VCE_ERR_ARG; eps = 0 is exactly ce_forward_backward.  Other arguments as
 * ce_forward_backward.
 */
VCE_API int ce_forward_backward_ls(const void* logits, vce_dtype dt, int64_t T, int64_t V, int64_t ld,
                           const int64_t* labels, int64_t ignore_index, float label_smoothing,
                           vce_reduction red, const float* grad_output, float* loss_rows,
                           float* loss_out, float* row_stats, void* grad_logits, vce_dtype grad_dt,
                           int64_t ld_grad, int32_t* status, vce_stream_t s);

/*
 * vce_test_ce_fused_stall -- test hook for the give-up path of ce_forward_backward's
 * shared-memory kernel (no page counterpart).  Runs that kernel on bf16 logits [T, V]
 * (ld = V), ignore_index -100, reduction SUM, with its producer announcing 16 more bytes per
 * stage than its copies deliver, so no stage ever completes.  Every wait is bounded by wait_ns
 * (1 ms .. 2 s): the waiting warps give up and record their code, which the last CTA writes
 * to *status (105..109, see ce_forward_backward).  Each role stops at its next wait, the
 * producer lets its copies land (bounded) and the kernel returns; the context stays usable and
 * the launch slot is left zero.  loss_rows, row_stats and grad_logits are undefined afterwards.
 * Returns VCE_ERR_ARG, enqueuing nothing but the status reset, when [T, V] does not take the
 * shared-memory kernel (V not a multiple of 8, pointers not 16-byte aligned).
 */
VCE_API int vce_test_ce_fused_stall(const void* logits, int64_t T, int64_t V, const int64_t* labels,
                            const float* grad_output, float* loss_rows, float* row_stats,
                            void* grad_logits, uint64_t wait_ns, int32_t* status, vce_stream_t s);

/*
 * vce_test_ce_fwd_stall -- test hook for the give-up path of ce_forward's stage-ring kernel
 * (no page counterpart).  Runs that kernel on bf16 logits [T, V] (ld = V, 1 <= T <= 65536,
 * V * 2 > 32768 bytes), ignore_index -100, reduction SUM, with its producer announcing 16 more
 * bytes per stage than its copies deliver, so no stage ever completes.  Every wait is bounded
 * by wait_ns (1 ms .. 2 s): the waiting warps give up and record their code, which the last
 * CTA writes to *status (105, 106, 108, 110 or 112, see ce_forward) with no clearing before;
 * the kernel returns, the context stays usable and the launch slot is left zero.  loss_rows,
 * row_stats and *loss_out are undefined afterwards.  Returns VCE_ERR_ARG, enqueuing nothing,
 * when the rows do not take the stage ring (V not a multiple of 8, logits not 16-byte aligned,
 * rows of at most 32 KB).
 */
VCE_API int vce_test_ce_fwd_stall(const void* logits, int64_t T, int64_t V, const int64_t* labels,
                                  float* loss_rows, float* row_stats, float* loss_out, uint64_t wait_ns,
                                  int32_t* status, vce_stream_t s);

/*
 * ce_merge_chunks -- CE forward (+ backward) over logits held as k column chunks
 * in separate buffers, the single-GPU form of the vocabulary-parallel CE [MC,
 * vocab_parallel_cross_entropy; TT, Numerics: the owner of the target drops it].
 * Chunk c covers global columns [off_c, off_c + width[c]), off_c = sum of the
 * earlier widths, V = sum of all widths.  Three device steps:
 *   1. per chunk and row, over the chunk's non-target columns: the max m_c, the
 *      sum s_c of exp(z - m_c), and the target logit if the chunk owns the target
 *      (off_c <= t < off_c + width[c]); written to chunk_stats_ws as
 *      [k][T][VCE_CHUNK_STATS] = (m_c, s_c, z_t or 0, owner 1.0/0.0);
 *   2. per row: M = max_c m_c, S = sum_c s_c exp(m_c - M) (chunks with m_c = -inf
 *      skipped), then loss, row_stats and the reduction exactly as ce_forward;
 *   3. if chunk_grads != NULL: every chunk's gradient as ce_backward, with c_i from
 *      grad_output, read on the device when step 3 runs.
 *
 *   k                        1 .. VCE_MAX_CHUNKS
 *   chunk_logits             host array [k] of device pointers [T, chunk_ld[c]]
 *   chunk_width, chunk_ld    host arrays [k]: columns (>= 1) and leading dimensions
 *   chunk_grads              host array [k] of device pointers, or NULL (forward only)
 *   chunk_grad_ld            host array [k], or NULL for chunk_grad_ld = chunk_width
 *   chunk_stats_ws           [k * T * VCE_CHUNK_STATS] fp32, 16-byte aligned, scratch
 *   other arguments          as ce_forward / ce_backward
 */
VCE_API int ce_merge_chunks(int k, const void* const* chunk_logits, const int64_t* chunk_width,
                    const int64_t* chunk_ld, vce_dtype dt, int64_t T,
                    const int64_t* labels, int64_t ignore_index, vce_reduction red,
                    float* loss_rows, float* loss_out, float* row_stats,
                    const float* grad_output, void* const* chunk_grads,
                    const int64_t* chunk_grad_ld, vce_dtype grad_dt,
                    float* chunk_stats_ws, int32_t* status, vce_stream_t s);

/*
 * ce_merge_chunks_ls -- ce_merge_chunks with label smoothing (the targets and numerics of
 * ce_forward_ls / ce_backward_ls).  Step 1 also writes each (chunk, row)'s sum of logits to
 * chunk_sums_ws [k][T] fp32 (4-byte aligned scratch; required when label_smoothing > 0, may
 * be NULL otherwise); step 2 adds a row's chunk sums in chunk order.  label_smoothing outside
 * [0, 1) (or NaN) returns VCE_ERR_ARG; 0 is exactly ce_merge_chunks.  Other arguments as
 * ce_merge_chunks.
 */
VCE_API int ce_merge_chunks_ls(int k, const void* const* chunk_logits, const int64_t* chunk_width,
                       const int64_t* chunk_ld, vce_dtype dt, int64_t T,
                       const int64_t* labels, int64_t ignore_index, float label_smoothing,
                       vce_reduction red, float* loss_rows, float* loss_out, float* row_stats,
                       const float* grad_output, void* const* chunk_grads,
                       const int64_t* chunk_grad_ld, vce_dtype grad_dt,
                       float* chunk_stats_ws, float* chunk_sums_ws, int32_t* status, vce_stream_t s);

/*
 * ce_merge_chunks_noalloc -- ce_merge_chunks for callers that cannot allocate device memory.
 * None of the pages has a counterpart: this entry point exists for callers that have no
 * way to provide the per-call chunk_stats_ws scratch, such as a host program driving the
 * library through this C ABI without a device memory manager of its own, or an engine
 * whose device memory is a single arena reserved at start-up that no op may carve from.
 *
 * Same arguments, steps and results as ce_merge_chunks, without chunk_stats_ws: the
 * per-(chunk, row) statistics live in a fixed array in device memory that the library
 * defines (VCE_NOALLOC_MAX_CHUNK_ROWS entries of 16 bytes = 4 MiB, held on every GPU that
 * loads the library until the process exits).  The call allocates and frees nothing.
 *
 *   - k * T must not exceed VCE_NOALLOC_MAX_CHUNK_ROWS; larger sizes return
 *     VCE_ERR_SCRATCH_LIMIT and enqueue nothing.
 *   - The first call on each device looks up the array's device address on that device
 *     (cudaGetSymbolAddress, with that device current); make that first call before
 *     capturing any stream.  A failed lookup returns VCE_ERR_CUDA.  The address is kept
 *     with the unique id of the device's context: after a device reset (a new context,
 *     in which the library's module and its array are loaded anew) the next call looks it
 *     up again, and that call, too, belongs before any stream capture.
 *   - Every call on a device uses the same array and leaves its contents behind.  Calls
 *     whose work can overlap on the GPU (different streams without ordering, or different
 *     host threads) race on it and give undefined results; order them on one stream.
 */
VCE_API int ce_merge_chunks_noalloc(int k, const void* const* chunk_logits, const int64_t* chunk_width,
                            const int64_t* chunk_ld, vce_dtype dt, int64_t T,
                            const int64_t* labels, int64_t ignore_index, vce_reduction red,
                            float* loss_rows, float* loss_out, float* row_stats,
                            const float* grad_output, void* const* chunk_grads,
                            const int64_t* chunk_grad_ld, vce_dtype grad_dt,
                            int32_t* status, vce_stream_t s);

#ifdef __cplusplus
}
#endif

#endif /* VCE_H */
