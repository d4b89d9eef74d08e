// The loss reduction folded into the end of a ring kernel (ce_fwd_ring.cu: ce_forward;
// ce_ring.cu: ce_forward_backward), for SUM and MEAN over at most kMaxRows rows.
//
// Method: torchtitan PR #5723 "[loss] fix softmax collapse with improved ce perf" -- the loss is
// the sum of the rows' NLL, over the N rows with a valid label for MEAN (ignored rows weigh 0).
//
// Protocol.  Every CTA counts the batch's valid labels itself (count_valid_strided, while its
// first copies are in flight), so each row's weight 1/N is known where the row is finished.
// Within the kernel, error codes collect in a word of the CTA's shared memory.  At the end each
// CTA merges its code into its launch slot (ce_slots.cuh; the first code wins) and adds one to
// the slot's count of finished CTAs; the CTA that finds itself last sums every row's loss in a
// fixed order (thread i takes rows i, i + NT, ...; lanes, then warps, merged in order) as an
// fp32 (sum, compensation) pair with two-sum steps, as k_ce_reduce does, writes the reduced
// loss and the status word, and puts the slot back to zero.  The sum of an ignored row's +0
// loss adds nothing; a bad label's NaN makes the reduced loss NaN.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ce_slots.cuh"
#include "vce.h"

namespace vce {
namespace fold {

constexpr int64_t kMaxRows = 65536;   // every CTA reads every label: at most 512 KB of them

// s + x = t + e exactly (Knuth's TwoSum); e goes into the compensation c.
__device__ __forceinline__ void add(float& s, float& c, float x) {
    const float t = s + x;
    const float bp = t - s;
    c += (s - (t - bp)) + (x - bp);
    s = t;
}

// This thread's count of valid labels among rows first, first + step, ... (eight loads in
// flight).
__device__ __forceinline__ int count_valid_strided(const int64_t* labels, int64_t T, int64_t V,
                                                   int64_t ignore_index, int64_t first, int64_t step) {
    int n = 0;
#pragma unroll 8
    for (int64_t row = first; row < T; row += step) {
        const int64_t t = labels[row];
        n += (t != ignore_index && t >= 0 && t < V) ? 1 : 0;
    }
    return n;
}

// The last CTA's reduction: every row's loss summed in a fixed order (thread i takes rows i,
// i + NT, ...; lanes, then warps, merged in order) as an fp32 (sum, compensation) pair;
// thread 0 writes the reduced loss.  All NT threads call it.
template <int NT>
__device__ __forceinline__ void sum_losses(const float* loss_rows, int64_t T, long long n_all, int red,
                                           float* loss_out, float* sm_sum, float* sm_comp) {
    float sum = 0.f, comp = 0.f;
    // up to eight loads in flight ahead of the (serial) additions, which take the rows in the
    // same order as one at a time
    for (int64_t i = threadIdx.x; i < T; i += 8 * NT) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = i + u * NT < T ? __ldcg(loss_rows + i + u * NT) : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (i + u * NT < T) add(sum, comp, v[u]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float s2 = __shfl_xor_sync(0xFFFFFFFFu, sum, off);
        const float c2 = __shfl_xor_sync(0xFFFFFFFFu, comp, off);
        add(sum, comp, s2);
        comp += c2;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        sm_sum[warp] = sum;
        sm_comp[warp] = comp;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float s = 0.f, c = 0.f;
        for (int w = 0; w < NT / 32; ++w) {
            add(s, c, sm_sum[w]);
            c += sm_comp[w];
        }
        const double tot = isfinite(s) ? (double)s + (double)c : (double)s;
        *loss_out = red == VCE_RED_MEAN ? (float)(tot / (double)n_all) : (float)tot;   // 0/0: NaN
    }
}

// The end of a ring kernel, called by all NT threads of the block once every output of its rows
// is written (and, in a cluster, after the closing cluster barrier).  err: the CTA's error word
// in shared memory; n_all: the batch's valid labels; sm_sum, sm_comp: NT / 32 floats of shared
// memory; sm_last: one int of shared memory.  The last CTA reduces the losses if `reduce`,
// writes the status word (the first code, or 0) and puts the slot back to zero.  Every claim on
// the slot's row counter was made before its CTA got here.
template <int NT>
__device__ __forceinline__ void finish_slot(slots::LaunchSlot& slot, int32_t* status, const int* err, bool reduce,
                                            const float* loss_rows, int64_t T, long long n_all, int red,
                                            float* loss_out, float* sm_sum, float* sm_comp, int* sm_last) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        if (*err) atomicCAS(&slot.err, 0, *err);
        const int prev = atomicAdd(&slot.done, 1);
        *sm_last = prev == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (!*sm_last) return;
    __threadfence();
    // every CTA merged its code before it counted itself: the slot's word is final, and its
    // read overlaps the sum's loads
    int code = 0;
    if (threadIdx.x == 0) code = atomicExch(&slot.err, 0);
    if (reduce) sum_losses<NT>(loss_rows, T, n_all, red, loss_out, sm_sum, sm_comp);
    if (threadIdx.x == 0) {
        *status = code;
        atomicExch(&slot.done, 0);
        atomicExch(&slot.rows, 0u);
    }
}

}  // namespace fold
}  // namespace vce
