// The tensor-core GEMM as a plain fp32-output product, and its test hooks: the two launch
// forms the linear-CE runs (single CTAs or CTA pairs), the give-up path of the pipeline's
// bounded waits, and K-block skipping.
// No page counterpart: they expose the building block of the linear-CE for testing.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tc_launch.cuh"
#include "vce_check.cuh"
#include "vce.h"
#include "vce_host.h"
#include "vce_linear.h"

namespace vce {
namespace {

using tc::BK;
using tc::BM;
using tc::BN;
using tc::Mat;

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool sizes_ok(int64_t M, int64_t N, int64_t K, int64_t lim) {
    return M >= 1 && N >= 1 && K >= 1 && M % 8 == 0 && N % 8 == 0 && K % 8 == 0 && M <= lim && N <= lim && K <= lim;
}

// C[M, ldc] = op(A) op(B)^T with the given layouts, on CTA pairs or single CTAs.
// k2: two K blocks per stage (needs an even number of K blocks).
template <bool kK2>
cudaError_t gemm_as(const Mat& ma, const Mat& mb, int a_mn, int b_mn, const tc::GemmArgs& g,
                    const tc::EpiStore::Params& ep, bool pair, cudaStream_t s) {
    if (a_mn && b_mn) return tc::launch_gemm<tc::EpiStore, true, true, false, kK2>(ma, ma, mb, g, ep, pair, s);
    if (a_mn) return tc::launch_gemm<tc::EpiStore, true, false, false, kK2>(ma, ma, mb, g, ep, pair, s);
    if (b_mn) return tc::launch_gemm<tc::EpiStore, false, true, false, kK2>(ma, ma, mb, g, ep, pair, s);
    return tc::launch_gemm<tc::EpiStore, false, false, false, kK2>(ma, ma, mb, g, ep, pair, s);
}

int gemm(const void* A, int a_mn, const void* B, int b_mn, int64_t M, int64_t N, int64_t K, float* C, int64_t ldc,
         bool pair, bool k2, cudaStream_t s) {
    const Mat ma = a_mn ? Mat{A, M, K, M} : Mat{A, K, M, K};
    const Mat mb = b_mn ? Mat{B, N, K, N} : Mat{B, K, N, K};
    const int nk = (int)cdiv(K, BK);
    tc::GemmArgs g{(int)cdiv(M, BM), (int)cdiv(N, BN), nk, nk, 0, 0, 0, 0, nullptr};
    tc::EpiStore::Params ep{C, ldc, M, N, 0, 0};
    const cudaError_t e = k2 ? gemm_as<true>(ma, mb, a_mn, b_mn, g, ep, pair, s)
                             : gemm_as<false>(ma, mb, a_mn, b_mn, g, ep, pair, s);
    return e == cudaSuccess ? VCE_OK : VCE_ERR_CUDA;
}

}  // namespace

VCE_DEBUG_READER(debug_word_gemm_hooks)

}  // namespace vce

using namespace vce;

extern "C" int vce_gemm_bf16(const void* A, int a_mn, const void* B, int b_mn, int64_t M, int64_t N, int64_t K,
                             float* C, int64_t ldc, vce_stream_t s) {
    if (!A || !B || !C) return VCE_ERR_NULL;
    if (!sizes_ok(M, N, K, 1 << 30)) return VCE_ERR_SHAPE;
    if (ldc < N) return VCE_ERR_LD;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || (ldc % 4)) return VCE_ERR_ALIGN;
    int rc = require_sm100();
    if (rc) return rc;
    return gemm(A, a_mn, B, b_mn, M, N, K, C, ldc, cdiv(M, BM) % 2 == 0, false, s);
}

extern "C" int vce_gemm_bf16_variant(const void* A, int a_mn, const void* B, int b_mn, int64_t M, int64_t N, int64_t K,
                                     float* C, int64_t ldc, int pair, vce_stream_t s) {
    if (!A || !B || !C) return VCE_ERR_NULL;
    if (!sizes_ok(M, N, K, 1 << 30)) return VCE_ERR_SHAPE;
    if (ldc < N) return VCE_ERR_LD;
    if (pair < 0 || pair > 2 || (pair && cdiv(M, BM) % 2) || (pair == 2 && cdiv(K, BK) % 2)) return VCE_ERR_ARG;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || (ldc % 4)) return VCE_ERR_ALIGN;
    int rc = require_sm100();
    if (rc) return rc;
    return gemm(A, a_mn, B, b_mn, M, N, K, C, ldc, pair != 0, pair == 2, s);
}

extern "C" int vce_test_gemm_stall(const void* A, const void* B, int64_t M, int64_t N, int64_t K, float* C,
                                   uint64_t wait_ns, int32_t* status, vce_stream_t s) {
    if (!A || !B || !C || !status) return VCE_ERR_NULL;
    if (!sizes_ok(M, N, K, 1 << 20)) return VCE_ERR_SHAPE;
    if (wait_ns < 1000000ull || wait_ns > 2000000000ull) return VCE_ERR_ARG;   // 1 ms .. 2 s
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16)) return VCE_ERR_ALIGN;
    int rc = require_sm100();
    if (rc) return rc;
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return VCE_ERR_CUDA;
    const int nk = (int)cdiv(K, BK);
    tc::GemmArgs g{(int)cdiv(M, BM), (int)cdiv(N, BN), nk, nk, 0, 0, 0, 0, status, 16u, wait_ns};
    tc::EpiStore::Params ep{C, N, M, N, 0, 0};
    const Mat ma{A, K, M, K}, mb{B, K, N, K};
    return tc::launch_gemm<tc::EpiStore, false, false>(ma, ma, mb, g, ep, cdiv(M, BM) % 2 == 0, s) == cudaSuccess
               ? VCE_OK
               : VCE_ERR_CUDA;
}

extern "C" int vce_test_gemm_skip(const void* A, const void* B, int64_t M, int64_t N, int64_t K, const uint32_t* skip,
                                  int64_t skip_ld, float* C, vce_stream_t s) {
    if (!A || !B || !C || !skip) return VCE_ERR_NULL;
    if (!sizes_ok(M, N, K, 1 << 20)) return VCE_ERR_SHAPE;
    if (skip_ld < cdiv(cdiv(K, 128), 32) || skip_ld > (1 << 20)) return VCE_ERR_ARG;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(skip, 4)) return VCE_ERR_ALIGN;
    int rc = require_sm100();
    if (rc) return rc;
    const int nk = (int)cdiv(K, BK);
    tc::GemmArgs g{(int)cdiv(M, BM), (int)cdiv(N, BN), nk, nk, 0, 0, 0, 0, nullptr};
    g.skip = skip;
    g.skip_ld = (int)skip_ld;
    tc::EpiStore::Params ep{C, N, M, N, 0, 0};
    const Mat ma{A, K, M, K}, mb{B, K, N, K};
    return tc::launch_gemm<tc::EpiStore, false, false>(ma, ma, mb, g, ep, false, s) == cudaSuccess
               ? VCE_OK
               : VCE_ERR_CUDA;
}
