// Host-side helpers shared by the library's entry points: argument checks and cached
// device properties.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace vce {

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// rows * ld * esize bytes (the extent of a [rows, ld] matrix) fits in int64.
inline bool fits_bytes(int64_t rows, int64_t ld, size_t esize) {
    if (rows < 0 || ld < 0) return false;
    if (rows == 0 || ld == 0) return true;
    const int64_t lim = INT64_MAX / (int64_t)esize;
    return ld <= lim / rows;
}

// Per-device caches hold this many devices; calls on a device beyond it report an error
// (or skip the cached fast path where one exists).
constexpr int kMaxDevices = 64;

int device_sm_count();     // SMs of the current device (cached per device)

// Remembers a failed CUDA runtime result for vce_last_cuda_error (per host thread); returns e.
cudaError_t record_cuda(cudaError_t e);
int require_sm100();       // VCE_OK when the current device is an sm_100-family GPU

// Per-row merge of k partial (max, sum-exp, target, owner) statistics laid out [k][T] as
// float4, then the row finish (loss, row_stats); and the fixed-order loss reduction.
cudaError_t launch_stats_merge(const float* part, int k, int64_t T, int64_t V, const int64_t* labels,
                               int64_t ignore_index, float* loss_rows, float* row_stats, int32_t* status,
                               cudaStream_t s);
cudaError_t launch_loss_reduce(const float* loss_rows, const int64_t* labels, int64_t T, int64_t V,
                               int64_t ignore_index, int red, float* loss_out, float* row_stats, cudaStream_t s);

// Debug-build index checks (vce_check.cuh): each translation unit with checks reads and clears
// its own debug word (0 in the release build).
int debug_word_ce_fwd(int32_t* out);
int debug_word_ce_bwd(int32_t* out);
int debug_word_ce_fwd_ring(int32_t* out);
int debug_word_ce_bwd_ring(int32_t* out);
int debug_word_ce_ring(int32_t* out);
int debug_word_ce_fused(int32_t* out);
int debug_word_lce(int32_t* out);
int debug_word_gemm_hooks(int32_t* out);

}  // namespace vce
