// Device helpers shared by the library's kernels: storage decoding, streaming
// memory access, the hardware base-2 exponential, and the (max, sum-exp) pair
// arithmetic of a one-pass log-sum-exp.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "vce.h"

namespace vce {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn3 = 1.0986122886681098f;   // p_t < 1/4  <=>  x = L' - z_t > ln 3
constexpr float kInf = __builtin_huge_valf();

// MUFU.EX2: 2^x, denormal results flushed to zero (the terms it feeds are summed
// against a leading 1, so values below 2^-126 do not matter).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 16-byte streaming load that bypasses L1 (every byte of the logits is used once per pass).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// 16-byte loads with an L2 policy: kLoadStream as ld_stream16; kLoadKeep marks the lines
// evict-last (the same row is read again shortly, by the one-pass forward+backward).
enum { kLoadStream = 0, kLoadKeep = 1 };

template <int kLoad>
__device__ __forceinline__ uint64_t l2_policy() {
    uint64_t pol = 0;
    if (kLoad == kLoadKeep) asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

template <int kLoad>
__device__ __forceinline__ uint4 ld16(const void* p, uint64_t pol) {
    if (kLoad == kLoadStream) return ld_stream16(p);
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p), "l"(pol));
    return r;
}

// Streaming (evict-first) stores for gradients that are not read back by this pass.
__device__ __forceinline__ void st_stream16(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_stream8(void* p, uint2 v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values to a packed bf16 pair, round to nearest even (lo in bits 0..15).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint16_t to_bf16(float v) {
    return (uint16_t)(pack_bf16x2(v, 0.f) & 0xFFFFu);
}

// ---- storage element traits -------------------------------------------------------------

template <typename S>
struct Elt;

template <>
struct Elt<float> {
    static constexpr int kGroup = 4;   // elements per 16-byte vector
    __device__ __forceinline__ static void unpack(uint4 r, float (&v)[4]) {
        v[0] = __uint_as_float(r.x);
        v[1] = __uint_as_float(r.y);
        v[2] = __uint_as_float(r.z);
        v[3] = __uint_as_float(r.w);
    }
    __device__ __forceinline__ static float load1(const float* p) { return __ldg(p); }
    __device__ __forceinline__ static void store1(float* p, float v) { *p = v; }
};

template <>
struct Elt<uint16_t> {   // bf16 storage bits
    static constexpr int kGroup = 8;
    __device__ __forceinline__ static void unpack(uint4 r, float (&v)[8]) {
        v[0] = bf16_lo(r.x);
        v[1] = bf16_hi(r.x);
        v[2] = bf16_lo(r.y);
        v[3] = bf16_hi(r.y);
        v[4] = bf16_lo(r.z);
        v[5] = bf16_hi(r.z);
        v[6] = bf16_lo(r.w);
        v[7] = bf16_hi(r.w);
    }
    __device__ __forceinline__ static float load1(const uint16_t* p) {
        return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p)) << 16);
    }
    __device__ __forceinline__ static void store1(uint16_t* p, float v) { *p = to_bf16(v); }
};

// Store G consecutive fp32 values (G = 4 or 8) at an aligned output address.
template <typename O, int G>
struct GroupStore;

template <>
struct GroupStore<uint16_t, 8> {   // 16 B
    __device__ __forceinline__ static void run(uint16_t* p, const float (&g)[8]) {
        st_stream16(p, make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]),
                                  pack_bf16x2(g[4], g[5]), pack_bf16x2(g[6], g[7])));
    }
    static constexpr int kAlign = 16;
};
template <>
struct GroupStore<uint16_t, 4> {   // 8 B
    __device__ __forceinline__ static void run(uint16_t* p, const float (&g)[4]) {
        st_stream8(p, make_uint2(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3])));
    }
    static constexpr int kAlign = 8;
};
template <>
struct GroupStore<float, 4> {      // 16 B
    __device__ __forceinline__ static void run(float* p, const float (&g)[4]) {
        st_stream16(p, make_uint4(__float_as_uint(g[0]), __float_as_uint(g[1]), __float_as_uint(g[2]),
                                  __float_as_uint(g[3])));
    }
    static constexpr int kAlign = 16;
};
template <>
struct GroupStore<float, 8> {      // 2 x 16 B
    __device__ __forceinline__ static void run(float* p, const float (&g)[8]) {
        st_stream16(p, make_uint4(__float_as_uint(g[0]), __float_as_uint(g[1]), __float_as_uint(g[2]),
                                  __float_as_uint(g[3])));
        st_stream16(p + 4, make_uint4(__float_as_uint(g[4]), __float_as_uint(g[5]), __float_as_uint(g[6]),
                                      __float_as_uint(g[7])));
    }
    static constexpr int kAlign = 16;
};

// Two fp32 FMAs, (a0, a1) * b + c, in one packed instruction (each lane rounds as fmaf).
__device__ __forceinline__ void ffma2(float a0, float a1, float b, float c, float& d0, float& d1) {
    asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %4};\n\tmov.b64 pc, {%5, %5};\n\t"
        "fma.rn.f32x2 pd, pa, pb, pc;\n\tmov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

// (d0, d1) = (a0 * b, a1 * b), two products in one packed fp32 instruction; each rounds as the
// scalar product a * b does.
__device__ __forceinline__ void fmul2(float a0, float a1, float b, float& d0, float& d1) {
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %4};\n\t"
        "mul.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b));
}

// ---- (max, sum-exp) pairs ------------------------------------------------------------------
//
// A pair (m, s) stands for the multiset sum  s * e^m = sum_k e^{v_k}, with m one of the v_k
// (the largest, for ms_push; a running reference within ~22 of the largest, for
// ms_push_lazy), so s >= 1 and no term overflows.  The empty set (or a set of -inf only) is
// (-inf, 0).

// Merge (m2, s2) into (m, s), rescaling both sums to the larger reference.
__device__ __forceinline__ void ms_merge(float& m, float& s, float m2, float s2) {
    const float M = fmaxf(m, m2);
    const float a = (m == M) ? 1.f : ex2((m - M) * kLog2e);    // also covers m = m2 = -inf
    const float b = (m2 == M) ? 1.f : ex2((m2 - M) * kLog2e);
    s = s * a + s2 * b;
    m = M;
}

// Add G values.  mb caches m * log2(e) (0 while m = -inf, so -inf values give e^-inf = 0).
template <int G>
__device__ __forceinline__ void ms_push(const float (&v)[G], float& m, float& s, float& mb) {
    float vm = v[0];
#pragma unroll
    for (int k = 1; k < G; ++k) vm = fmaxf(vm, v[k]);
    if (vm > m) {   // a new running maximum: rare after the first few groups of a row
        s *= ex2((m - vm) * kLog2e);
        m = vm;
        mb = m * kLog2e;
    }
    float e[G];
#pragma unroll
    for (int k = 0; k < G; ++k) e[k] = ex2(fmaf(v[k], kLog2e, -mb));
#pragma unroll
    for (int w = 1; w < G; w *= 2)
#pragma unroll
        for (int k = 0; k + w < G; k += 2 * w) e[k] += e[k + w];
    s += e[0];
}

// Add G values against a lazily updated reference.  The pair (m, s) only needs m to be one
// of the values seen (so s >= 1) and no term to overflow, not m to be the exact maximum:
// the first group of a thread sets m to that group's maximum, and later groups are summed
// against it unless a term reaches 2^32 (a value ~22 above m), which triggers a rescale to
// the new maximum.  This drops the per-group max (G-1 FMNMX + a compare) from the common
// path; the result is the same sum, s rounded in the same fp32 steps up to the reference.
template <int G>
__device__ __forceinline__ void ms_push_lazy(const float (&v)[G], float& m, float& s, float& mb) {
    if (m == -kInf) {   // first finite group of this thread: take its exact maximum as reference
        float vm = v[0];
#pragma unroll
        for (int k = 1; k < G; ++k) vm = fmaxf(vm, v[k]);
        if (vm == -kInf) return;
        m = vm;
        mb = m * kLog2e;
    }
    float e[G];
#pragma unroll
    for (int k = 0; k < G; ++k) e[k] = ex2(fmaf(v[k], kLog2e, -mb));
#pragma unroll
    for (int w = 1; w < G; w *= 2)
#pragma unroll
        for (int k = 0; k + w < G; k += 2 * w) e[k] += e[k + w];
    if (e[0] < 4294967296.f) {   // 2^32: no term can have overflowed
        s += e[0];
        return;
    }
    ms_push<G>(v, m, s, mb);   // rare: a value far above the reference; redo this group exactly
}

// ms_push_lazy over U groups at once: one reference check and one overflow check for all
// U * G values, so the U groups' exponentials and sums form one block of independent work.
template <int U, int G>
__device__ __forceinline__ void ms_push_lazy_batch(const float (&v)[U][G], float& m, float& s, float& mb) {
    if (m == -kInf) {   // first finite batch of this thread: its exact maximum is the reference
        float vm = -kInf;
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int k = 0; k < G; ++k) vm = fmaxf(vm, v[u][k]);
        if (vm == -kInf) return;
        m = vm;
        mb = m * kLog2e;
    }
    float t[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        float e[G];
#pragma unroll
        for (int k = 0; k < G; ++k) e[k] = ex2(fmaf(v[u][k], kLog2e, -mb));
#pragma unroll
        for (int w = 1; w < G; w *= 2)
#pragma unroll
            for (int k = 0; k + w < G; k += 2 * w) e[k] += e[k + w];
        t[u] = e[0];
    }
#pragma unroll
    for (int w = 1; w < U; w *= 2)
#pragma unroll
        for (int u = 0; u + w < U; u += 2 * w) t[u] += t[u + w];
    if (t[0] < 4294967296.f) {   // 2^32: no term can have overflowed
        s += t[0];
        return;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) ms_push<G>(v[u], m, s, mb);   // rare: redo exactly
}

__device__ __forceinline__ void ms_push1(float v, float& m, float& s, float& mb) {
    if (v > m) {
        s *= ex2((m - v) * kLog2e);
        m = v;
        mb = m * kLog2e;
    }
    s += ex2(fmaf(v, kLog2e, -mb));
}

__device__ __forceinline__ void ms_warp_reduce(float& m, float& s) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, off);
        const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, off);
        ms_merge(m, s, m2, s2);
    }
}

// ---- the per-row finish of the forward ----------------------------------------------------

__device__ __forceinline__ float softplus_f(float x) {
    return x > 0.f ? x + log1pf(expf(-x)) : log1pf(expf(x));
}

// From the target-excluded pair (M, S) and the target logit zt:
//   L' = M + log S, x = L' - z_t, loss = softplus(x) = -log p_t,
//   stats = (L', 1 - p_t = sigmoid(x), target coefficient, weight 1).
// The target coefficient is p_t - 1 when p_t < 1/4 and -(1 - p_t) otherwise, each a
// single rounding from sigmoid (torchtitan PR #5723, Numerics).  All three functions of x come
// from one exponential e = exp(-|x|):  sigmoid(|x|) = 1 / (1 + e),  sigmoid(-|x|) = e / (1 + e),
// softplus(x) = max(x, 0) + log1p(e)  (each the value of the textbook branch form: 1 / (1 + e^-x)
// or e^x / (1 + e^x) by the sign of x, and x + log1p(e^-x) or log1p(e^x)).
__device__ __forceinline__ float4 ce_row_finish(float M, float S, float zt, float* loss) {
    float lse, x;
    if (S > 0.f) {
        const float lnS = logf(S);
        lse = M + lnS;
        x = (M - zt) + lnS;   // M - z_t is exact for bf16 inputs of similar size
    } else {                   // no finite non-target logit: p_t = 1
        lse = -kInf;
        x = -kInf;
    }
    const float e = expf(-fabsf(x));
    const float d = 1.f + e;
    const float s_abs = 1.f / d, s_neg = e / d;
    const float pnt = (x >= 0.f) ? s_abs : s_neg;                 // sigmoid(x)
    *loss = (x > 0.f ? x : 0.f) + log1pf(e);
    const float dt = (x > kLn3) ? (s_neg - 1.f) : -pnt;           // x > ln 3 > 0: sigmoid(-x) = s_neg
    return make_float4(lse, pnt, dt, 1.f);
}

// Label smoothing eps (targets q = (1 - eps) onehot + eps / V): from the same (M, S, z_t) and
// the row's sum of all logits,
//   loss = (1 - eps) softplus(x) + eps (LSE(z) - sum_z / V),  LSE(z) = max(z_t, L') + softplus(-|x|),
// and the target coefficient gains eps (1 - 1/V) (the non-target shift -eps/V is applied by
// the backward).
__device__ __forceinline__ float4 ce_row_finish_smoothed(float M, float S, float zt, float sum_z, int64_t V,
                                                         float eps, float* loss) {
    float nll;
    float4 st = ce_row_finish(M, S, zt, &nll);
    const float L = st.x;
    float lse_all;
    if (L == -kInf) lse_all = zt;
    else if (zt == -kInf) lse_all = L;
    else lse_all = fmaxf(zt, L) + softplus_f(-fabsf(L - zt));
    const float inv_v = 1.f / (float)V;
    *loss = (1.f - eps) * nll + eps * (lse_all - sum_z * inv_v);
    st.z += eps * (1.f - inv_v);
    return st;
}

}  // namespace vce
