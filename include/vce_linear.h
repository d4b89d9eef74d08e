/*
 * vce_linear.h -- fused linear cross-entropy of the GB300 vocabulary CE library.
 *
 * Source: apple/ml-cross-entropy issue #14 (Cut Cross-Entropy):
 * linear_cross_entropy(e, c, targets) computes the cross-entropy of softmax(e c^T)
 * from the embeddings e and the classifier weight c (no bias) without storing the
 * logits; impl="cce_exact" disables gradient filtering so the gradients are the plain
 * CE gradients; use_kahan keeps the accumulation of dc and de compensated.  The CE
 * numerics are those of ce_forward / ce_backward in vce.h (torchtitan PR #5723).
 *
 * Conventions as in vce.h: device pointers owned by the caller, asynchronous on the
 * caller's stream, negative return = host-detected argument error (nothing enqueued),
 * device-detected errors in *status.
 */
#ifndef VCE_LINEAR_H
#define VCE_LINEAR_H

#include "vce.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Bytes of workspace linear_ce_fwd_bwd needs for these sizes; 0 if the sizes are
 * invalid (T, V >= 1; D >= 8 and a multiple of 8).  For T=8192, D=4096, V=128256 it is
 * about 1.95 GB (per-tile statistics, one 32768-column vocabulary chunk of the gradient as
 * two bf16 halves, the compensated dE accumulator pair, the fp32 dW partial of one chunk,
 * and the gradient-filter bit tables of one chunk).
 */
VCE_API size_t linear_ce_workspace_bytes(int64_t T, int64_t D, int64_t V);

/*
 * linear_ce_fwd_bwd -- loss and gradients of CE(softmax(E W^T), labels) in one call.
 *   z = E W^T is formed 128 x 256 tiles at a time on the tensor cores (bf16 operands,
 *   fp32 accumulators) and never stored as a [T, V] matrix.
 *   loss_rows[i] = softplus(logsumexp_{j != t} z_ij - z_it), reduction as ce_forward.
 *   With G = dloss/dz (softmax - onehot scaled by c_i, the target entry by the p_t = 1/4
 *   branch, ignored rows 0):
 *       dE = G W   [T, D],       dW = G^T E   [V, D].
 *   G enters the two gradient GEMMs as an exact-to-16-bits pair of bf16 terms
 *   (G = G_hi + G_lo).  Each GEMM accumulates in fp32 on the tensor cores; dW is formed as
 *   two partial products over the halves of T and dE as one partial product per 32768-column
 *   vocabulary chunk, and the partials are merged with a two-sum compensated fp32 pair.
 *
 *   E            [T, D] bf16 row-major, 16-byte aligned
 *   W            [V, D] bf16 row-major, 16-byte aligned
 *   labels       [T] int64; ignore_index marks ignored rows
 *   red          VCE_RED_MEAN, VCE_RED_SUM or VCE_RED_NONE
 *   grad_output  fp32 [1] (SUM, MEAN) or [T] (NONE): upstream gradient of the loss
 *   loss_rows    [T] fp32, written;  loss_out [1] fp32, written for SUM / MEAN
 *   dE, dW       [T, D] and [V, D] of dtype grad_dt (VCE_BF16 or VCE_F32), 16-byte
 *                aligned, written (bf16 rounded to nearest even from fp32)
 *   workspace    >= linear_ce_workspace_bytes(T, D, V) bytes, 256-byte aligned,
 *                scratch owned by the caller, contents undefined on return
 *   status       [1] int32: 0, VCE_ERR_LABEL, or 100..104 when the GEMM pipeline gave up
 *                (100: the two CTAs of a pair got different tensor-memory columns; 101..104: a
 *                device-side wait ran out), the outputs then being undefined
 */
VCE_API int linear_ce_fwd_bwd(const void* E, const void* W, int64_t T, int64_t D, int64_t V,
                      const int64_t* labels, int64_t ignore_index, vce_reduction red,
                      const float* grad_output, float* loss_rows, float* loss_out,
                      void* dE, void* dW, vce_dtype grad_dt,
                      void* workspace, size_t workspace_bytes, int32_t* status, vce_stream_t s);

/*
 * linear_ce_fwd_bwd_filtered -- linear_ce_fwd_bwd with gradient filtering (Cut Cross-Entropy
 * issue #14: the filtering that impl="cce_exact" turns off; the page states no rule, this is
 * the rule taken here).
 *   G is cut into blocks of 128 rows by 128 vocabulary columns (aligned at 0).  A block is
 *   dropped -- its entries count as 0 in dE = G W and dW = G^T E -- when none of its valid
 *   rows has its target among the block's columns and every non-target probability p_ij of
 *   its valid rows is below filter_eps.  The dW and dE GEMMs skip the dropped blocks'
 *   K blocks (128 rows, resp. columns, is a whole number of their K blocks), so kept blocks
 *   keep exactly the unfiltered arithmetic and the work falls with the dropped fraction.
 *   The loss and row statistics are never filtered.  The filtered gradient GEMMs run on
 *   single CTAs; dW is one product over all of T (dE's chunks are still merged with the
 *   two-sum pair).
 *
 *   filter_eps   threshold on p_ij, finite and >= 0; 0 is exactly linear_ce_fwd_bwd (no
 *                block is dropped).  NaN, negative or infinite: VCE_ERR_ARG, nothing enqueued.
 *   kept_blocks  optional device uint64 (8-byte aligned, may be NULL): set to the number of
 *                (row block, column block) pairs kept, over all vocabulary chunks; 0 when
 *                filter_eps = 0 (the filter does not run)
 *   Every other argument as linear_ce_fwd_bwd; the workspace size is the same.
 */
VCE_API int linear_ce_fwd_bwd_filtered(const void* E, const void* W, int64_t T, int64_t D, int64_t V,
                               const int64_t* labels, int64_t ignore_index, vce_reduction red,
                               const float* grad_output, float* loss_rows, float* loss_out,
                               void* dE, void* dW, vce_dtype grad_dt, float filter_eps,
                               unsigned long long* kept_blocks, void* workspace, size_t workspace_bytes,
                               int32_t* status, vce_stream_t s);

/*
 * linear_ce_fwd_bwd_timed -- linear_ce_fwd_bwd_filtered with a CUDA event recorded on `s`
 * before and after each of its tensor-core GEMM launches (no page counterpart: it measures
 * the call for the benchmark).  The outputs are those of linear_ce_fwd_bwd_filtered (which
 * filter_eps = 0 makes linear_ce_fwd_bwd).  It waits for the stream, then writes to host
 * memory, per GEMM kind k (0 statistics GEMM, 1 gradient-tile GEMMs, 2 dW GEMMs, 3 dE
 * GEMMs), gemm_ms[k] = the summed milliseconds of its launches and gemm_launches[k] = their
 * number.  Blocking; the events are created and destroyed by the call.  NULL gemm_ms or
 * gemm_launches: VCE_ERR_NULL.
 */
VCE_API int linear_ce_fwd_bwd_timed(const void* E, const void* W, int64_t T, int64_t D, int64_t V,
                            const int64_t* labels, int64_t ignore_index, vce_reduction red,
                            const float* grad_output, float* loss_rows, float* loss_out,
                            void* dE, void* dW, vce_dtype grad_dt, float filter_eps,
                            unsigned long long* kept_blocks, void* workspace, size_t workspace_bytes,
                            int32_t* status, vce_stream_t s, float* gemm_ms, int* gemm_launches);

/*
 * vce_gemm_bf16 -- the tensor-core GEMM the linear-CE is built on, with a plain fp32 output:
 *     C[m][n] = sum_k A(m, k) B(n, k)
 * A is [M, K] row-major (a_mn = 0, K-major) or [K, M] row-major (a_mn = 1, MN-major); B is
 * [N, K] (b_mn = 0) or [K, N] (b_mn = 1).  bf16 operands, fp32 accumulation, tiles 256
 * columns wide, run on CTA pairs (256-row tiles) when ceil(M / 128) is even, else on single
 * CTAs (128-row tiles).  M, N, K multiples of 8; A, B, C 16-byte aligned; C [M, ldc] fp32,
 * ldc >= N and a multiple of 4.  No page counterpart: it exposes the building block for
 * testing.
 */
VCE_API int vce_gemm_bf16(const void* A, int a_mn, const void* B, int b_mn, int64_t M, int64_t N, int64_t K,
                  float* C, int64_t ldc, vce_stream_t s);

/*
 * vce_gemm_bf16_variant -- vce_gemm_bf16 in a chosen launch form (no page counterpart; for
 * testing and timing the forms the linear-CE uses): pair = 0 single CTAs, 128-row tiles;
 * pair = 1 CTA pairs issuing cta_group::2 MMAs, 256-row tiles (needs ceil(M / 128) even);
 * pair = 2 CTA pairs with two 64-column K blocks per pipeline stage (also needs
 * ceil(K / 64) even).  Any other pair, or a form the shape does not allow: VCE_ERR_ARG,
 * nothing enqueued.  Other arguments as vce_gemm_bf16.
 */
VCE_API int vce_gemm_bf16_variant(const void* A, int a_mn, const void* B, int b_mn, int64_t M, int64_t N, int64_t K,
                          float* C, int64_t ldc, int pair, vce_stream_t s);

/*
 * vce_test_gemm_stall -- test hook for the GEMM's give-up path (no page counterpart).
 * Runs vce_gemm_bf16's pipeline (A [M,K], B [N,K] K-major; CTA pairs when ceil(M / 128) is
 * even, else single CTAs) with its producer announcing 16 more bytes per stage than its
 * copies deliver, so no stage ever completes.  Every wait of the kernel is bounded by wait_ns
 * (1 ms .. 2 s): the waiting role gives up, writes its code to *status (101 empty-slot, 102
 * full-slot, 103 accumulator-free, 104 accumulator-full wait), the other roles (of both CTAs
 * of a pair) stop, copies in flight are drained, tensor memory is released and the kernel
 * returns; the context stays usable.  C's contents are undefined afterwards.
 */
VCE_API int vce_test_gemm_stall(const void* A, const void* B, int64_t M, int64_t N, int64_t K, float* C,
                        uint64_t wait_ns, int32_t* status, vce_stream_t s);

/*
 * vce_test_gemm_skip -- test hook for the GEMM's K-block skipping (no page counterpart; the
 * machinery gradient filtering uses).  As vce_gemm_bf16 with A [M, K], B [N, K] K-major, C
 * [M, N] fp32, except that M tile i (128 rows) adds only the 128-column K blocks b whose bit
 * b % 32 of skip[i * skip_ld + b / 32] is set:
 *     C[m][n] = sum over set blocks b of sum_{k in block b} A[m][k] B[n][k]
 * (0 where a tile has no set bit).  skip: device uint32 [ceil(M/128)][skip_ld], skip_ld >=
 * ceil(ceil(K/128) / 32); bits of blocks at or past ceil(K/128) must be clear (C is undefined
 * for a tile that sets only such bits).  It runs on single CTAs, as the filtered linear-CE's
 * gradient GEMMs do.  Bad skip_ld: VCE_ERR_ARG.
 */
VCE_API int vce_test_gemm_skip(const void* A, const void* B, int64_t M, int64_t N, int64_t K, const uint32_t* skip,
                       int64_t skip_ld, float* C, vce_stream_t s);

#ifdef __cplusplus
}
#endif

#endif /* VCE_LINEAR_H */
