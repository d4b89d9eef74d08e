// Device-side index checks of the debug build.
//
// Built with -DVCE_DEBUG_CHECKS (python -m vocab_cross_entropy_gb300.build --debug-checks,
// which makes libvce_debug.so), every dbg::ok(cond, code) in the kernels tests an index the
// kernel is about to turn into a global address -- a row against T, a column range against
// the row's extent, a chunk, stage or tile index against its table -- and, when the test
// fails, records `code` in the translation unit's debug word (first failure wins) and returns
// false, so the caller skips the access.  Nothing traps.  The host reads and clears the words
// with vce_debug_status().  In the release build dbg::ok is the constant true and the checks
// compile away.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace vce {
namespace dbg {

enum {
    kRow = 121,      // a row index outside [0, T)
    kCols = 122,     // a column range outside the row (or the chunk) it belongs to
    kChunk = 123,    // a chunk / segment index outside its table
    kStage = 124,    // a shared-memory stage or ring slot outside the ring
    kTile = 125,     // a GEMM output tile row or column outside the output
};

#ifdef VCE_DEBUG_CHECKS
// One word per translation unit (the library is built without relocatable device code).
static __device__ int32_t g_word;

__device__ __forceinline__ bool ok(bool cond, int code) {
    if (!cond) atomicCAS(&g_word, 0, (int32_t)code);
    return cond;
}

// Host reader of this translation unit's word: copies it to *out and clears it.
#define VCE_DEBUG_READER(fn)                                                               \
    int fn(int32_t* out) {                                                                 \
        const int32_t zero = 0;                                                            \
        if (cudaMemcpyFromSymbol(out, ::vce::dbg::g_word, sizeof(int32_t)) != cudaSuccess) \
            return -1;                                                                     \
        return cudaMemcpyToSymbol(::vce::dbg::g_word, &zero, sizeof(int32_t)) == cudaSuccess ? 0 : -1; \
    }
#else
__device__ __forceinline__ constexpr bool ok(bool, int) { return true; }

#define VCE_DEBUG_READER(fn) \
    int fn(int32_t* out) {   \
        *out = 0;            \
        return 0;            \
    }
#endif

constexpr bool kEnabled =
#ifdef VCE_DEBUG_CHECKS
    true;
#else
    false;
#endif

}  // namespace dbg
}  // namespace vce
