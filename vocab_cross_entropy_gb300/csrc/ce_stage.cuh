// Per-stage row work of the kernels that stream rows through a shared-memory stage ring
// (ce_ring.cu: one-pass forward + gradient; ce_fwd_ring.cu: forward).  NT consumer threads
// share a stage; thread tid takes its 16-byte vectors tid + u * NT (u < U).  rel0 is the
// target's column minus the column of the thread's first vector of the stage.  kFull: the
// stage is whole (U * NT vectors), so no vector needs a bound check.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "vce_async.cuh"
#include "vce_device.cuh"

namespace vce {
namespace stage {

// 16 bytes of -inf in the storage format (vectors past a partial stage's end).
template <typename S>
__device__ __forceinline__ uint4 neg_inf16();
template <>
__device__ __forceinline__ uint4 neg_inf16<uint16_t>() {
    return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
}
template <>
__device__ __forceinline__ uint4 neg_inf16<float>() {
    return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
}

// Whether the target column falls in one of this thread's vectors of the stage.
template <typename S, int NT, int U>
__device__ __forceinline__ bool holds_target(int rel0) {
    constexpr int G = Elt<S>::kGroup, Span = NT * G;
    return rel0 >= 0 && rel0 < U * Span && (rel0 % Span) < G;
}

// The thread's U vectors of a loaded stage (vectors past a partial stage's end read as -inf).
template <typename S, int NT, int U, bool kFull>
__device__ __forceinline__ void load_stage(const uint4* buf, int nvec, int tid, uint4 (&r)[U]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int vi = tid + u * NT;
        r[u] = (kFull || vi < nvec) ? tc::lds16(buf + vi) : neg_inf16<S>();
    }
}

// Forward over the thread's U vectors of a stage: the (max, sum-exp) pair takes its U * G
// values at once (one reference check, one overflow check).  kTarget: this thread holds the
// target, whose value goes to *zt and is left out of the sum.  kSumZ: the stage's values
// (target included) are also added to *sz.
template <typename S, int NT, int U, bool kFull, bool kTarget, bool kSumZ = false>
__device__ __forceinline__ void fwd_vectors(const uint4 (&r)[U], int nvec, int rel0, int tid, float& m, float& s,
                                            float& mb, float* zt, float* sz = nullptr) {
    constexpr int G = Elt<S>::kGroup;
    float v[U][G];
#pragma unroll
    for (int u = 0; u < U; ++u) Elt<S>::unpack(r[u], v[u]);
    if (kSumZ) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (kFull || tid + u * NT < nvec) {
                float q[G];
#pragma unroll
                for (int k = 0; k < G; ++k) q[k] = v[u][k];
#pragma unroll
                for (int w = 1; w < G; w *= 2)
#pragma unroll
                    for (int k = 0; k + w < G; k += 2 * w) q[k] += q[k + w];
                *sz += q[0];
            }
        }
    }
    if (kTarget) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t rel = (uint32_t)(rel0 - u * NT * G);
#pragma unroll
            for (int k = 0; k < G; ++k)
                if (rel == (uint32_t)k) { *zt = v[u][k]; v[u][k] = -kInf; }
        }
    }
    ms_push_lazy_batch<U, G>(v, m, s, mb);
}

// Forward over one loaded stage (load_stage, then fwd_vectors); r keeps the loaded vectors.
template <typename S, int NT, int U, bool kFull, bool kTarget, bool kSumZ = false>
__device__ __forceinline__ void fwd_stage(const uint4* buf, int nvec, int rel0, int tid, float& m, float& s,
                                          float& mb, float* zt, float* sz, uint4 (&r)[U]) {
    load_stage<S, NT, U, kFull>(buf, nvec, tid, r);
    fwd_vectors<S, NT, U, kFull, kTarget, kSumZ>(r, nvec, rel0, tid, m, s, mb, zt, sz);
}

// The forward of a stage, choosing the instantiation for this thread and stage.  nvec may
// exceed U * NT (a later batch of the same stage follows); only the first U * NT are summed.
// r: the thread's loaded vectors (for a caller that keeps them).
template <typename S, int NT, int U, bool kSumZ = false>
__device__ __forceinline__ void fwd_stage_any(const uint4* buf, int nvec, int rel0, int tid, float& m, float& s,
                                              float& mb, float* zt, float* sz, uint4 (&r)[U]) {
    const bool full = nvec >= U * NT;
    if (holds_target<S, NT, U>(rel0)) {
        if (full) fwd_stage<S, NT, U, true, true, kSumZ>(buf, nvec, rel0, tid, m, s, mb, zt, sz, r);
        else fwd_stage<S, NT, U, false, true, kSumZ>(buf, nvec, rel0, tid, m, s, mb, zt, sz, r);
    } else {
        if (full) fwd_stage<S, NT, U, true, false, kSumZ>(buf, nvec, rel0, tid, m, s, mb, zt, sz, r);
        else fwd_stage<S, NT, U, false, false, kSumZ>(buf, nvec, rel0, tid, m, s, mb, zt, sz, r);
    }
}
template <typename S, int NT, int U, bool kSumZ = false>
__device__ __forceinline__ void fwd_stage_any(const uint4* buf, int nvec, int rel0, int tid, float& m, float& s,
                                              float& mb, float* zt, float* sz = nullptr) {
    uint4 r[U];
    fwd_stage_any<S, NT, U, kSumZ>(buf, nvec, rel0, tid, m, s, mb, zt, sz, r);
}

// Gradient of the thread's U vectors of a held stage (bwd_vectors: from registers the caller
// loaded; bwd_stage: read from the shared-memory stage): coef * 2^(z log2 e - bias) for every
// column, less shift = c eps / V
// under label smoothing (kShift), then the thread holding the target overwrites that entry with
// gt (its own later store to the same address).  Without kShift the entries are the plain
// product (an FMA with a zero addend rounds the same, but measured 1.2% slower in the one-pass
// kernel).  kPacked: the exponent arguments and the products two at a time (fma/mul .f32x2, the
// same rounding as the scalar forms); measured 1.1% + 1.0% faster in the one-pass kernel, and no
// faster in the backward alone.  Packed sums in the forward (even and odd columns summed apart)
// measured 0.3% slower in the one-pass kernel than the scalar tree.
template <typename S, typename O, int NT, int U, bool kFull, bool kShift = false, bool kPacked = false>
__device__ __forceinline__ void bwd_vectors(const uint4 (&r)[U], int nvec, O* gcol, int rel0, int tid, float coef,
                                            float bias, float gt, float shift) {
    constexpr int G = Elt<S>::kGroup;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int vi = tid + u * NT;
        if (kFull || vi < nvec) {
            float v[G];
            Elt<S>::unpack(r[u], v);
#pragma unroll
            for (int k = 0; k < G; k += 2) {
                float a0, a1;
                if (kPacked) {
                    ffma2(v[k], v[k + 1], kLog2e, -bias, a0, a1);
                } else {
                    a0 = fmaf(v[k], kLog2e, -bias);
                    a1 = fmaf(v[k + 1], kLog2e, -bias);
                }
                const float e0 = ex2(a0), e1 = ex2(a1);
                if (kPacked && kShift) {
                    ffma2(e0, e1, coef, -shift, v[k], v[k + 1]);
                } else if (kPacked) {
                    fmul2(e0, e1, coef, v[k], v[k + 1]);
                } else {
                    v[k] = kShift ? fmaf(coef, e0, -shift) : coef * e0;
                    v[k + 1] = kShift ? fmaf(coef, e1, -shift) : coef * e1;
                }
            }
            GroupStore<O, G>::run(gcol + vi * G, v);
        }
    }
    if (holds_target<S, NT, U>(rel0)) Elt<O>::store1(gcol + tid * G + rel0, gt);
}

template <typename S, typename O, int NT, int U, bool kFull, bool kShift = false, bool kPacked = false>
__device__ __forceinline__ void bwd_stage(const uint4* buf, int nvec, O* gcol, int rel0, int tid, float coef,
                                          float bias, float gt, float shift) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int vi = tid + u * NT;
        if (kFull || vi < nvec) r[u] = tc::lds16(buf + vi);
    }
    bwd_vectors<S, O, NT, U, kFull, kShift, kPacked>(r, nvec, gcol, rel0, tid, coef, bias, gt, shift);
}

}  // namespace stage
}  // namespace vce
