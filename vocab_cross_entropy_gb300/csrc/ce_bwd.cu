// Gradient of the softmax cross-entropy w.r.t. [T, V] logits, rebuilt in one pass from the
// logits and the per-row statistics of the forward.
//
// Method: torchtitan PR #5723 "[loss] fix softmax collapse with improved ce perf"
//   Numerics  - gradient softmax(z) - onehot(t) with the target entry p_t - 1 below p_t = 1/4
//               and -p_non_target above it; ignored labels zeroed by the label mask.
//   Memory/perf (compiled form) - the backward re-reads the saved bf16 input and the per-row
//               statistics and rebuilds the gradient in one fused kernel.
//
//   k_ce_bwd   one (chunk, row) segment per block iteration; 16-byte vector loads and
//              streaming stores on the aligned body of a row, scalar accesses on its head,
//              tail, or the whole row when input and output rows are out of phase.
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

// Items are (chunk, row) pairs, row-major over chunks so neighbouring blocks read the same row.
template <typename S, typename O, int NT>
__global__ void __launch_bounds__(NT) k_ce_bwd(const __grid_constant__ SegTable tab, const int64_t* __restrict__ labels,
                                               const float4* __restrict__ row_stats,
                                               const float* __restrict__ grad_output, int go_per_row,
                                               float eps_over_v) {
    const int64_t items = tab.T * tab.k;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int64_t row = it / tab.k;
        const int c = (int)(it - row * tab.k);
        if (!dbg::ok(c >= 0 && c < tab.k && row < tab.T, dbg::kChunk) ||
            !dbg::ok(tab.width[c] <= tab.ld_in[c] && tab.width[c] <= tab.ld_out[c], dbg::kCols))
            continue;   // block-uniform
        const float4 st = row_stats[row];
        const bool zero = (st.w == 0.f);   // ignored row or bad label: +0.0 by selection
        const float cg = zero ? 0.f : grad_output[go_per_row ? row : 0] * st.w;
        const float coef = cg * st.y;                      // c * (1 - p_t)
        const float bias = (st.x == -kInf) ? 0.f : st.x * kLog2e;
        const float gt = cg * st.z;
        const float shift = cg * eps_over_v;   // label smoothing: every non-target entry loses c eps / V
        const int64_t tl = zero ? -1 : labels[row] - tab.off[c];
        const S* in = reinterpret_cast<const S*>(tab.in[c]) + row * tab.ld_in[c];
        O* out = reinterpret_cast<O*>(tab.out[c]) + row * tab.ld_out[c];
        bwd_segment<S, O, NT>(in, out, tab.width[c], tl, coef, bias, gt, zero, shift);
    }
}

template <typename S, typename O, int NT>
cudaError_t launch_bwd(const SegTable& tab, const int64_t* labels, const float* row_stats, const float* go,
                       int go_per_row, float eps_over_v, cudaStream_t s) {
    auto kern = k_ce_bwd<S, O, NT>;
    kern<<<grid_for(kern, NT, tab.T * tab.k), NT, 0, s>>>(tab, labels, reinterpret_cast<const float4*>(row_stats), go,
                                                           go_per_row, eps_over_v);
    return cudaGetLastError();
}

template <typename S, typename O>
cudaError_t dispatch_bwd2(int nt, const SegTable& tab, const int64_t* labels, const float* rs, const float* go,
                          int per_row, float eov, cudaStream_t s) {
    if (nt == 128) return launch_bwd<S, O, 128>(tab, labels, rs, go, per_row, eov, s);
    if (nt == 256) return launch_bwd<S, O, 256>(tab, labels, rs, go, per_row, eov, s);
    return launch_bwd<S, O, 512>(tab, labels, rs, go, per_row, eov, s);
}

}  // namespace

VCE_DEBUG_READER(debug_word_ce_bwd)

cudaError_t launch_ce_bwd(vce_dtype dt, vce_dtype gdt, int nt, const SegTable& tab, const int64_t* labels,
                         const float* rs, const float* go, int per_row, cudaStream_t s, float eov) {
    if (dt == VCE_BF16 && gdt == VCE_BF16) return dispatch_bwd2<uint16_t, uint16_t>(nt, tab, labels, rs, go, per_row, eov, s);
    if (dt == VCE_BF16 && gdt == VCE_F32) return dispatch_bwd2<uint16_t, float>(nt, tab, labels, rs, go, per_row, eov, s);
    if (dt == VCE_F32 && gdt == VCE_BF16) return dispatch_bwd2<float, uint16_t>(nt, tab, labels, rs, go, per_row, eov, s);
    return dispatch_bwd2<float, float>(nt, tab, labels, rs, go, per_row, eov, s);
}


}  // namespace vce

using namespace vce;

extern "C" int ce_backward_ls(const void* logits, vce_dtype dt, int64_t T, int64_t V, int64_t ld,
                              const int64_t* labels, int64_t ignore_index, float label_smoothing, vce_reduction red, const float* row_stats, const float* grad_output,
                           void* grad_logits, vce_dtype grad_dt, int64_t ld_grad, vce_stream_t s) {
    (void)ignore_index;   // ignored rows carry weight 0 in row_stats
    int rc = VCE_OK;
    if (dt != VCE_F32 && dt != VCE_BF16) return VCE_ERR_DTYPE;
    if (red != VCE_RED_NONE && red != VCE_RED_SUM && red != VCE_RED_MEAN) return VCE_ERR_DTYPE;
    if (T < 0) return VCE_ERR_SHAPE;
    if (!(label_smoothing >= 0.f && label_smoothing < 1.f)) return VCE_ERR_ARG;
    if (grad_dt != VCE_F32 && grad_dt != VCE_BF16) return VCE_ERR_DTYPE;
    if (V < 1) return VCE_ERR_SHAPE;
    if (ld < V || ld_grad < V) return VCE_ERR_LD;
    if (T == 0) return VCE_OK;
    if (!logits || !labels || !row_stats || !grad_output || !grad_logits) return VCE_ERR_NULL;
    const size_t es = dt == VCE_BF16 ? 2 : 4, gs = grad_dt == VCE_BF16 ? 2 : 4;
    if (!fits_bytes(T, ld, es) || !fits_bytes(T, ld_grad, gs)) return VCE_ERR_SHAPE;
    if (!aligned(logits, es) || !aligned(grad_logits, gs) || !aligned(labels, 8) || !aligned(row_stats, 16) ||
        !aligned(grad_output, 4))
        return VCE_ERR_ALIGN;
    if ((rc = require_sm100())) return rc;
    SegTable tab{};
    tab.k = 1;
    tab.T = T;
    tab.in[0] = logits;
    tab.out[0] = grad_logits;
    tab.width[0] = V;
    tab.off[0] = 0;
    tab.ld_in[0] = ld;
    tab.ld_out[0] = ld_grad;
    // Rows streamed through shared memory where the layout allows it, else one block per row
    // with loads from global memory.
    const float eps_over_v = label_smoothing / (float)V;
    bool launched = false;
    cudaError_t e = launch_bwd_ring(dt, grad_dt, tab, labels, row_stats, grad_output, red == VCE_RED_NONE, eps_over_v,
                                    s, &launched);
    if (e == cudaSuccess && !launched) {
        const int nt = pick_threads(V * (int64_t)es);
        e = launch_ce_bwd(dt, grad_dt, nt, tab, labels, row_stats, grad_output, red == VCE_RED_NONE, s, eps_over_v);
    }
    if (e != cudaSuccess) return VCE_ERR_CUDA;
    return VCE_OK;
}


extern "C" int ce_backward(const void* logits, vce_dtype dt, int64_t T, int64_t V, int64_t ld, const int64_t* labels,
                           int64_t ignore_index, vce_reduction red, const float* row_stats, const float* grad_output,
                           void* grad_logits, vce_dtype grad_dt, int64_t ld_grad, vce_stream_t s) {
    return ce_backward_ls(logits, dt, T, V, ld, labels, ignore_index, 0.f, red, row_stats, grad_output, grad_logits,
                          grad_dt, ld_grad, s);
}
