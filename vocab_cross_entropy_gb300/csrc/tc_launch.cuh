// Host side of the tensor-core GEMM (tc_gemm.cuh): TMA maps over row-major bf16 matrices, the
// launch of one GEMM as single CTAs or as CTA pairs, and the plain store epilogue (fp32 or
// bf16 output).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "tc_gemm.cuh"
#include "vce_device.cuh"
#include "vce_host.h"

namespace vce {
namespace tc {

// A row-major bf16 matrix [outer, inner] with row pitch ld elements, as a GEMM operand.
struct Mat {
    const void* base;
    int64_t inner, outer, ld;
};

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 f = fn.load();
    if (!f) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
            fn.store(f);
        }
    }
    return f;
}

// 2-D map over m with boxes of 64 inner elements (128 B, the swizzle span) x box_rows rows,
// 128-byte swizzle.  Loads past the extents read zeros.
inline bool make_map(CUtensorMap* map, const Mat& m, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)m.inner, (cuuint64_t)m.outer};
    cuuint64_t strides[1] = {(cuuint64_t)(m.ld * 2)};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(m.base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The kernel's shared-memory opt-in, set once per device (the attribute belongs to the
// function in the current device's context), and the number of 2-CTA clusters that fit on the
// device at once (0: none).  ready: the caller's per-kernel cache, per device 0 (unknown) or
// 1 + the clusters that fit.
template <class K>
cudaError_t prepare_kernel(K kern, int smem, bool pair, std::atomic<int> (&ready)[kMaxDevices], int* clusters) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int r = ready[dev].load();
    if (r == 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        int fit = 0;
        if (pair) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(2 * (device_sm_count() / 2));
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = smem;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&fit, kern, &cfg) != cudaSuccess) {
                (void)cudaGetLastError();
                fit = 0;
            }
        }
        r = 1 + fit;
        ready[dev].store(r);
    }
    *clusters = r - 1;
    return cudaSuccess;
}

template <class Epi, bool kAmn, bool kBmn, bool kCta2, bool kDualA, bool kK2 = false>
cudaError_t launch_gemm_as(const Mat& a0, const Mat& a1, const Mat& b, const GemmArgs& g,
                           const typename Epi::Params& ep, cudaStream_t s) {
    using C = Cfg<kCta2, kDualA, kK2, Epi::kScratch>;
    CUtensorMap ma0, ma1, mb;
    if (!make_map(&ma0, a0, kAmn ? 64 : BM) || !make_map(&ma1, a1, kAmn ? 64 : BM) ||
        !make_map(&mb, b, kBmn ? 64 : C::kBRows))
        return record_cuda(cudaErrorInvalidValue);
    auto kern = k_tc_gemm<Epi, kAmn, kBmn, kCta2, kDualA, kK2>;
    static std::atomic<int> ready[kMaxDevices];   // one cache per kernel instantiation
    int clusters = 0;
    cudaError_t e = prepare_kernel(kern, C::kSmem, kCta2, ready, &clusters);
    if (e != cudaSuccess) return record_cuda(e);
    if (kCta2) {
        if (clusters < 1 || g.tiles_m % 2) return record_cuda(cudaErrorInvalidConfiguration);
        const int64_t tiles = (int64_t)(g.tiles_m / 2) * g.tiles_n;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3((unsigned)(2 * std::max<int64_t>(1, std::min<int64_t>(tiles, clusters))));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = C::kSmem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return record_cuda(cudaLaunchKernelEx(&cfg, kern, ma0, ma1, mb, g, ep));
    }
    const int64_t tiles = (int64_t)g.tiles_m * g.tiles_n;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, device_sm_count()));
    kern<<<grid, kThreads, C::kSmem, s>>>(ma0, ma1, mb, g, ep);
    return record_cuda(cudaGetLastError());
}

// One GEMM, as CTA pairs (pair: tiles_m must be even and there must be no skip bits) or as
// single CTAs.  kDualA: acc = (A0 + A1) B^T over nk_a0 K blocks, both A tiles of a block in one
// stage (no skip bits).  kK2: two consecutive K blocks per stage (one A operand: nk == nk_a0, an
// even nk, no skip bits; the same accumulation order as one block per stage).
template <class Epi, bool kAmn, bool kBmn, bool kDualA = false, bool kK2 = false>
cudaError_t launch_gemm(const Mat& a0, const Mat& a1, const Mat& b, const GemmArgs& g,
                        const typename Epi::Params& ep, bool pair, cudaStream_t s) {
    if (pair && (g.tiles_m % 2 || g.skip)) return record_cuda(cudaErrorInvalidConfiguration);
    if (kDualA && g.skip) return record_cuda(cudaErrorInvalidConfiguration);
    if (kK2 && (g.skip || g.nk % 2 || g.nk != g.nk_a0)) return record_cuda(cudaErrorInvalidConfiguration);
    return pair ? launch_gemm_as<Epi, kAmn, kBmn, true, kDualA, kK2>(a0, a1, b, g, ep, s)
                : launch_gemm_as<Epi, kAmn, kBmn, false, kDualA, kK2>(a0, a1, b, g, ep, s);
}

// Output tile rows into [rows, cols] at row offset row_off with row pitch ld (bf16 rounded to
// nearest even from fp32, or fp32), evict-first: nothing in a call reads them back.
struct EpiStore {
    static constexpr int kScratch = 0;
    struct Params {
        void* out;
        int64_t ld, rows, cols, row_off;
        int bf16;
    };
    struct Row {};
    __device__ __forceinline__ static void begin(const Params&, Row&, int, int) {}
    __device__ __forceinline__ static void consume(const Params& p, Row&, int row, int col0, const uint32_t (&acc)[32]) {
        if (row >= p.rows || col0 >= p.cols) return;
        const int64_t base = (p.row_off + row) * p.ld + col0;
        const int n = (p.cols - col0) < 32 ? (int)(p.cols - col0) : 32;
        if (p.bf16) {
            uint16_t* o = reinterpret_cast<uint16_t*>(p.out) + base;
            if (n == 32) {
                uint32_t w[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(__uint_as_float(acc[2 * k]), __uint_as_float(acc[2 * k + 1]));
                uint4* d = reinterpret_cast<uint4*>(o);
#pragma unroll
                for (int q = 0; q < 4; ++q) st_stream16(d + q, make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
            } else {
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    if (k < n) o[k] = to_bf16(__uint_as_float(acc[k]));
            }
        } else {
            float* o = reinterpret_cast<float*>(p.out) + base;
            if (n == 32) {
                uint4* d = reinterpret_cast<uint4*>(o);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    st_stream16(d + q, make_uint4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]));
            } else {
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    if (k < n) o[k] = __uint_as_float(acc[k]);
            }
        }
    }
    __device__ __forceinline__ static void end(const Params&, Row&, int, int) {}
};

}  // namespace tc
}  // namespace vce
