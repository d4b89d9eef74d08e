// The two row streams every CE kernel is built from: the forward (max, sum-exp) over a row
// segment with the target column left out, and the backward that rebuilds the gradient of a
// row segment.  Both split a segment into a scalar head up to the first 16-byte boundary,
// 16-byte vectors (four loads in flight per thread before use) and a scalar tail.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "vce_device.cuh"

namespace vce {

constexpr int kUnroll = 4;

// ------------------------------------------------------------------------------------------
// Row segment streaming (forward): thread-partial (m, s) over the segment's columns except
// the local target column `tl` (tl < 0 or >= w: no target here).  The thread that meets the
// target column stores its value to *zt_out.

// kLazy: sum against a lazily updated reference (ms_push_lazy); otherwise m ends as the exact
// maximum of the non-target values (ms_push), as the chunk statistics report it.
// kSumZ: also add every value of the segment (target included) into sz.
// kU: 16-byte loads in flight per thread before any is used.
template <typename S, int NT, bool kLazy, int kLoad = kLoadStream, bool kSumZ = false, int kU = kUnroll>
__device__ __forceinline__ void fwd_segment(const S* __restrict__ row, int64_t w, int64_t tl, float& m,
                                            float& s, float& mb, float* zt_out, const int tid,
                                            float* sz = nullptr) {
    constexpr int G = Elt<S>::kGroup;
    const uintptr_t a = reinterpret_cast<uintptr_t>(row);
    int64_t h = (int64_t)(((16 - (a & 15)) & 15) / sizeof(S));   // elements before 16-B alignment
    if (h > w) h = w;
    const int64_t nvec = (w - h) / G;
    const int64_t tail0 = h + nvec * G;

    // unaligned head and tail, one element per thread
    for (int64_t j = tid; j < h; j += NT) {
        float v = Elt<S>::load1(row + j);
        if (kSumZ) *sz += v;
        if (j == tl) { *zt_out = v; v = -kInf; }
        ms_push1(v, m, s, mb);
    }
    for (int64_t j = tail0 + tid; j < w; j += NT) {
        float v = Elt<S>::load1(row + j);
        if (kSumZ) *sz += v;
        if (j == tl) { *zt_out = v; v = -kInf; }
        ms_push1(v, m, s, mb);
    }

    const uint4* vp = reinterpret_cast<const uint4*>(row + h);
    const uint64_t pol = l2_policy<kLoad>();
    for (int64_t v0 = tid; v0 < nvec; v0 += (int64_t)NT * kU) {
        uint4 r[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t vi = v0 + (int64_t)u * NT;
            if (vi < nvec) r[u] = ld16<kLoad>(vp + vi, pol);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t vi = v0 + (int64_t)u * NT;
            if (vi < nvec) {
                float v[G];
                Elt<S>::unpack(r[u], v);
                if (kSumZ) {
                    float q[G];
#pragma unroll
                    for (int k = 0; k < G; ++k) q[k] = v[k];
#pragma unroll
                    for (int wd = 1; wd < G; wd *= 2)
#pragma unroll
                        for (int k = 0; k + wd < G; k += 2 * wd) q[k] += q[k + wd];
                    *sz += q[0];
                }
                const uint64_t rel = (uint64_t)(tl - (h + vi * G));
                if (rel < (uint64_t)G) {   // the target's group: mask it out (column test)
#pragma unroll
                    for (int k = 0; k < G; ++k)
                        if (rel == (uint64_t)k) { *zt_out = v[k]; v[k] = -kInf; }
                }
                if (kLazy)
                    ms_push_lazy<G>(v, m, s, mb);
                else
                    ms_push<G>(v, m, s, mb);
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
// Backward: one row segment.  grad = coef * 2^(z*log2e - bias) off target, gt at the target.

// Non-target entries are coef * 2^(z log2 e - bias) - shift (shift = c * eps / V under label
// smoothing, 0 otherwise: fmaf with a zero addend rounds exactly as the product).
template <typename S, typename O, int NT, int kLoad = kLoadStream>
__device__ __forceinline__ void bwd_segment(const S* __restrict__ row, O* __restrict__ grow, int64_t w, int64_t tl,
                                            float coef, float bias, float gt, bool zero, float shift = 0.f) {
    constexpr int G = Elt<S>::kGroup;
    const int tid = threadIdx.x;
    const uintptr_t a = reinterpret_cast<uintptr_t>(row);
    int64_t h = (int64_t)(((16 - (a & 15)) & 15) / sizeof(S));
    if (h > w) h = w;
    const bool out_ok = ((reinterpret_cast<uintptr_t>(grow + h)) % GroupStore<O, G>::kAlign) == 0;
    if (!out_ok) h = w;   // input and output phases differ: the whole segment goes scalar
    const int64_t nvec = (w - h) / G;
    const int64_t tail0 = h + nvec * G;

    auto one = [&](int64_t j) {
        float g = 0.f;
        if (!zero) {
            const float z = Elt<S>::load1(row + j);
            g = (j == tl) ? gt : fmaf(coef, ex2(fmaf(z, kLog2e, -bias)), -shift);
        }
        Elt<O>::store1(grow + j, g);
    };
    for (int64_t j = tid; j < h; j += NT) one(j);
    for (int64_t j = tail0 + tid; j < w; j += NT) one(j);

    const uint4* vp = reinterpret_cast<const uint4*>(row + h);
    O* gp = grow + h;
    if (zero) {
        const float g[G] = {};
        for (int64_t vi = tid; vi < nvec; vi += NT) GroupStore<O, G>::run(gp + vi * G, g);
        return;
    }
    const uint64_t pol = l2_policy<kLoad>();
    for (int64_t v0 = tid; v0 < nvec; v0 += (int64_t)NT * kUnroll) {
        uint4 r[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t vi = v0 + (int64_t)u * NT;
            if (vi < nvec) r[u] = ld16<kLoad>(vp + vi, pol);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t vi = v0 + (int64_t)u * NT;
            if (vi < nvec) {
                float v[G];
                Elt<S>::unpack(r[u], v);
#pragma unroll
                for (int k = 0; k < G; ++k) v[k] = fmaf(coef, ex2(fmaf(v[k], kLog2e, -bias)), -shift);
                const uint64_t rel = (uint64_t)(tl - (h + vi * G));
                if (rel < (uint64_t)G) {
#pragma unroll
                    for (int k = 0; k < G; ++k)
                        if (rel == (uint64_t)k) v[k] = gt;
                }
                GroupStore<O, G>::run(gp + vi * G, v);
            }
        }
    }
}

// Block-wide merge of the thread pairs; the result is valid in thread 0.
template <int NT>
__device__ __forceinline__ void ms_block_reduce(float& m, float& s, float* sm_m, float* sm_s) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    ms_warp_reduce(m, s);
    if (lane == 0) { sm_m[wid] = m; sm_s[wid] = s; }
    __syncthreads();
    if (wid == 0) {
        m = lane < NW ? sm_m[lane] : -kInf;
        s = lane < NW ? sm_s[lane] : 0.f;
        ms_warp_reduce(m, s);
    }
}

__device__ __forceinline__ void flag_label_error(int32_t* status) {
    if (status) atomicCAS(status, 0, (int32_t)VCE_ERR_LABEL);
}

}  // namespace vce
