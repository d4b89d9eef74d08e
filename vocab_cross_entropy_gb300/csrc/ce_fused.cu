// Cross-entropy forward and backward in one pass over the logits, for callers that know the
// upstream gradient when the forward runs (training with a mean loss seeded by 1).
//
// Method: torchtitan PR #5723 "[loss] fix softmax collapse with improved ce perf" — the same
// numerics as ce_forward / ce_backward (Numerics: target-excluded log-sum-exp, softplus NLL,
// the p_t = 1/4 branch; Memory/perf: "forward also prepares the backward").
//
// Rows whose layout suits 16-byte bulk copies go to the kernel in ce_ring.cu, which holds each
// row in shared memory between its passes.  The others come here: each block takes one row,
// the forward stream reads it from HBM with an evict-last L2 policy, the block reduces it to
// the row statistics, and the backward stream re-reads the same row (mostly an L2 hit) to
// write the gradient.  Measured at T=16384, V=128256 bf16: without the evict-last policy the
// step takes 12% longer; an evict-first policy on the re-read costs 1.4%.  HBM moves V*e bytes
// in and V*e_g out per row, instead of 2*V*e in and V*e_g out for the two separate calls.
//
//   k_ce_count_valid  one block: 1/N for the mean, parked in loss_out[0] until k_ce_reduce
//                     replaces it by the mean loss (unless the ring kernel counts N and reduces
//                     the losses itself: SUM / MEAN over at most 65536 rows)
//   k_ce_fused        one row per block iteration: forward stream, statistics, backward stream
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "ce_rows.cuh"
#include "ce_segments.h"
#include "vce.h"
#include "vce_device.cuh"
#include "vce_check.cuh"
#include "vce_host.h"

namespace vce {
namespace {

// The weight 1/N of the mean (N = the number of valid labels) into *inv_n, and the status word
// cleared for the kernels that follow on the stream.  Eight labels per thread are in flight
// before any is used.
template <int NT>
__global__ void __launch_bounds__(NT) k_ce_count_valid(const int64_t* __restrict__ labels, int64_t T, int64_t V,
                                                       int64_t ignore_index, float* inv_n, int32_t* status) {
    constexpr int U = 8;
    __shared__ long long sm_n[NT / 32];
    long long n = 0;
    for (int64_t i0 = threadIdx.x; i0 < T; i0 += (int64_t)NT * U) {
        int64_t t[U];
#pragma unroll
        for (int u = 0; u < U; ++u) t[u] = i0 + (int64_t)u * NT < T ? labels[i0 + (int64_t)u * NT] : ignore_index;
#pragma unroll
        for (int u = 0; u < U; ++u) n += (t[u] != ignore_index && t[u] >= 0 && t[u] < V) ? 1 : 0;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) n += __shfl_xor_sync(0xFFFFFFFFu, n, off);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (lane == 0) sm_n[wid] = n;
    __syncthreads();
    if (threadIdx.x == 0) {
        long long tot = 0;
        for (int w = 0; w < NT / 32; ++w) tot += sm_n[w];
        *inv_n = tot > 0 ? (float)(1.0 / (double)tot) : 0.f;   // the value k_ce_reduce computes
        *status = 0;
    }
}

// Two 512-thread blocks per SM: both streams inlined need ~60 registers (three blocks would spill).
// kSmooth: label smoothing eps > 0 (the row's sum of logits is reduced alongside the pair; the
// non-target gradient entries lose c eps / V).
template <typename S, typename O, int NT, bool kSmooth>
__global__ void __launch_bounds__(NT, 1024 / NT)
    k_ce_fused(const S* __restrict__ logits, int64_t T, int64_t V, int64_t ld, const int64_t* __restrict__ labels,
               int64_t ignore_index, int red, const float* __restrict__ grad_output, const float* __restrict__ inv_n,
               float* __restrict__ loss_rows, float4* __restrict__ row_stats, O* __restrict__ grad, int64_t ld_g,
               int32_t* status, float eps) {
    __shared__ float sm_m[NT / 32], sm_s[NT / 32], sm_sz[NT / 32];
    __shared__ float sm_zt, sm_coef, sm_bias, sm_gt, sm_shift;
    const float w_valid = (red == VCE_RED_MEAN) ? *inv_n : 1.f;
    for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
        const int64_t t = labels[row];
        if (!dbg::ok(row >= 0 && row < T && V <= ld && V <= ld_g, dbg::kRow)) continue;   // block-uniform
        const S* in = logits + row * ld;
        O* out = grad + row * ld_g;
        const bool ignored = (t == ignore_index);
        if (ignored || t < 0 || t >= V) {   // gradient +0.0 by selection; the logits are not read
            if (threadIdx.x == 0) {
                loss_rows[row] = ignored ? 0.f : __int_as_float(0x7FC00000);
                row_stats[row] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (!ignored) flag_label_error(status);
            }
            bwd_segment<S, O, NT>(in, out, V, -1, 0.f, 0.f, 0.f, true);
            continue;
        }
        float m = -kInf, s = 0.f, mb = 0.f, sz = 0.f;
        fwd_segment<S, NT, true, kLoadKeep, kSmooth>(in, V, t, m, s, mb, &sm_zt, threadIdx.x, &sz);
        if (kSmooth) {   // block sum of the logits (the barrier below publishes the warp sums)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sz += __shfl_xor_sync(0xFFFFFFFFu, sz, off);
            if ((threadIdx.x & 31) == 0) sm_sz[threadIdx.x >> 5] = sz;
        }
        ms_block_reduce<NT>(m, s, sm_m, sm_s);
        if (threadIdx.x == 0) {
            float loss;
            float4 st;
            if (kSmooth) {
                float tot = 0.f;
                for (int k = 0; k < NT / 32; ++k) tot += sm_sz[k];
                st = ce_row_finish_smoothed(m, s, sm_zt, tot, V, eps, &loss);
            } else {
                st = ce_row_finish(m, s, sm_zt, &loss);
            }
            st.w = w_valid;
            row_stats[row] = st;
            loss_rows[row] = loss;
            const float c = grad_output[red == VCE_RED_NONE ? row : 0] * w_valid;
            sm_coef = c * st.y;
            sm_bias = (st.x == -kInf) ? 0.f : st.x * kLog2e;
            sm_gt = c * st.z;
            sm_shift = kSmooth ? c * (eps / (float)V) : 0.f;
        }
        __syncthreads();
        bwd_segment<S, O, NT>(in, out, V, t, sm_coef, sm_bias, sm_gt, false, sm_shift);
        __syncthreads();   // sm_* are rewritten by the next row
    }
}

template <typename S, typename O, int NT>
cudaError_t launch_fused(const void* logits, int64_t T, int64_t V, int64_t ld, const int64_t* labels, int64_t ig,
                         int red, const float* go, const float* inv_n, float* loss_rows, float* row_stats, void* grad,
                         int64_t ld_g, int32_t* status, float eps, cudaStream_t s) {
    auto kern = eps > 0.f ? k_ce_fused<S, O, NT, true> : k_ce_fused<S, O, NT, false>;
    kern<<<grid_for(kern, NT, T), NT, 0, s>>>(reinterpret_cast<const S*>(logits), T, V, ld, labels, ig, red, go,
                                              inv_n, loss_rows, reinterpret_cast<float4*>(row_stats),
                                              reinterpret_cast<O*>(grad), ld_g, status, eps);
    return cudaGetLastError();
}

template <typename S, typename O>
cudaError_t dispatch_fused2(int nt, const void* logits, int64_t T, int64_t V, int64_t ld, const int64_t* labels,
                            int64_t ig, int red, const float* go, const float* inv_n, float* lr, float* rs, void* g,
                            int64_t ldg, int32_t* st, float eps, cudaStream_t s) {
    if (nt == 128)
        return launch_fused<S, O, 128>(logits, T, V, ld, labels, ig, red, go, inv_n, lr, rs, g, ldg, st, eps, s);
    if (nt == 256)
        return launch_fused<S, O, 256>(logits, T, V, ld, labels, ig, red, go, inv_n, lr, rs, g, ldg, st, eps, s);
    return launch_fused<S, O, 512>(logits, T, V, ld, labels, ig, red, go, inv_n, lr, rs, g, ldg, st, eps, s);
}

}  // namespace

VCE_DEBUG_READER(debug_word_ce_fused)

}  // namespace vce

using namespace vce;

extern "C" int ce_forward_backward_ls(const void* logits, vce_dtype dt, int64_t T, int64_t V, int64_t ld,
                                      const int64_t* labels, int64_t ignore_index, float label_smoothing,
                                      vce_reduction red, const float* grad_output, float* loss_rows, float* loss_out,
                                      float* row_stats, void* grad_logits, vce_dtype grad_dt, int64_t ld_grad,
                                      int32_t* status, vce_stream_t s) {
    if (dt != VCE_F32 && dt != VCE_BF16) return VCE_ERR_DTYPE;
    if (grad_dt != VCE_F32 && grad_dt != VCE_BF16) return VCE_ERR_DTYPE;
    if (red != VCE_RED_NONE && red != VCE_RED_SUM && red != VCE_RED_MEAN) return VCE_ERR_DTYPE;
    if (!(label_smoothing >= 0.f && label_smoothing < 1.f)) return VCE_ERR_ARG;
    if (T < 0 || V < 1) return VCE_ERR_SHAPE;
    if (ld < V || ld_grad < V) return VCE_ERR_LD;
    if (!status || (red != VCE_RED_NONE && !loss_out)) return VCE_ERR_NULL;
    const size_t es = dt == VCE_BF16 ? 2 : 4, gs = grad_dt == VCE_BF16 ? 2 : 4;
    if (T > 0) {
        if (!logits || !labels || !grad_output || !loss_rows || !row_stats || !grad_logits) return VCE_ERR_NULL;
        if (!fits_bytes(T, ld, es) || !fits_bytes(T, ld_grad, gs)) return VCE_ERR_SHAPE;
        if (!aligned(logits, es) || !aligned(grad_logits, gs) || !aligned(labels, 8) || !aligned(loss_rows, 4) ||
            !aligned(row_stats, 16) || !aligned(grad_output, 4))
            return VCE_ERR_ALIGN;
    }
    if (red != VCE_RED_NONE && !aligned(loss_out, 4)) return VCE_ERR_ALIGN;
    int rc = require_sm100();
    if (rc) return rc;
    // The ring kernel writes the status word itself (its launch slot carries the error code), and
    // it counts N and reduces the losses itself where it can (SUM / MEAN, at most 65536 rows).
    // Otherwise the mean's weight 1/N comes first (k_ce_count_valid, which also clears the
    // status word) and k_ce_reduce last; the L2 re-read kernel needs the status word cleared.
    const bool ring_ok = T > 0 && fused_ring_layout_ok(dt, T, V, ld, ld_grad, logits, grad_logits);
    const bool ring_reduces = ring_ok && fused_ring_reduces(red, T);
    auto count_first = [&]() {
        k_ce_count_valid<1024><<<1, 1024, 0, s>>>(labels, T, V, ignore_index, loss_out, status);
        return cudaGetLastError() == cudaSuccess;
    };
    auto clear_status = [&]() { return cudaMemsetAsync(status, 0, sizeof(int32_t), s) == cudaSuccess; };
    bool cleared = false;
    if (T > 0 && red == VCE_RED_MEAN && !ring_reduces) {
        if (!count_first()) return VCE_ERR_CUDA;
        cleared = true;
    } else if (!ring_ok) {
        if (!clear_status()) return VCE_ERR_CUDA;
        cleared = true;
    }
    bool reduced = false;
    if (T > 0) {
        const float eps = label_smoothing;
        // The row held in shared memory where the layout allows it, else the L2 re-read.
        bool launched = false;
        cudaError_t e = launch_fused_ring(dt, grad_dt, logits, T, V, ld, labels, ignore_index, red, grad_output,
                                          loss_out, loss_rows, row_stats, grad_logits, ld_grad, status, s, &launched,
                                          eps, 2000000000ull, 0, ring_reduces ? &reduced : nullptr, loss_out);
        // no cluster fitted after all: the fallback needs the mean's weight first, and a cleared
        // status word
        if (e == cudaSuccess && !launched && ring_reduces && red == VCE_RED_MEAN) {
            if (!count_first()) return VCE_ERR_CUDA;
            cleared = true;
        }
        if (e == cudaSuccess && !launched && !cleared && !clear_status()) return VCE_ERR_CUDA;
        if (e == cudaSuccess && !launched) {
            const int nt = pick_threads(V * (int64_t)es);
            if (dt == VCE_BF16 && grad_dt == VCE_BF16)
                e = dispatch_fused2<uint16_t, uint16_t>(nt, logits, T, V, ld, labels, ignore_index, red, grad_output,
                                                        loss_out, loss_rows, row_stats, grad_logits, ld_grad, status,
                                                        eps, s);
            else if (dt == VCE_BF16)
                e = dispatch_fused2<uint16_t, float>(nt, logits, T, V, ld, labels, ignore_index, red, grad_output,
                                                     loss_out, loss_rows, row_stats, grad_logits, ld_grad, status,
                                                     eps, s);
            else if (grad_dt == VCE_BF16)
                e = dispatch_fused2<float, uint16_t>(nt, logits, T, V, ld, labels, ignore_index, red, grad_output,
                                                     loss_out, loss_rows, row_stats, grad_logits, ld_grad, status,
                                                     eps, s);
            else
                e = dispatch_fused2<float, float>(nt, logits, T, V, ld, labels, ignore_index, red, grad_output,
                                                  loss_out, loss_rows, row_stats, grad_logits, ld_grad, status, eps, s);
        }
        if (e != cudaSuccess) return VCE_ERR_CUDA;
    }
    if (red != VCE_RED_NONE && !reduced &&
        launch_loss_reduce(loss_rows, labels, T, V, ignore_index, red, loss_out, row_stats, s) != cudaSuccess)
        return VCE_ERR_CUDA;
    return VCE_OK;
}

extern "C" int ce_forward_backward(const void* logits, vce_dtype dt, int64_t T, int64_t V, int64_t ld,
                                   const int64_t* labels, int64_t ignore_index, vce_reduction red,
                                   const float* grad_output, float* loss_rows, float* loss_out, float* row_stats,
                                   void* grad_logits, vce_dtype grad_dt, int64_t ld_grad, int32_t* status,
                                   vce_stream_t s) {
    return ce_forward_backward_ls(logits, dt, T, V, ld, labels, ignore_index, 0.f, red, grad_output, loss_rows,
                                  loss_out, row_stats, grad_logits, grad_dt, ld_grad, status, s);
}
