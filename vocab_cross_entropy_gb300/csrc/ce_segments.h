// Row segments shared by the CE kernels: a table of up to VCE_MAX_CHUNKS column chunks
// (input pointer, output pointer, width, global column offset, leading dimensions), passed
// to kernels by value as a __grid_constant__ parameter, and the launch-shape helpers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "vce.h"
#include "vce_host.h"

namespace vce {

struct SegTable {
    int k;
    int64_t T;
    const void* in[VCE_MAX_CHUNKS];
    void* out[VCE_MAX_CHUNKS];
    int64_t width[VCE_MAX_CHUNKS];
    int64_t off[VCE_MAX_CHUNKS];
    int64_t ld_in[VCE_MAX_CHUNKS];
    int64_t ld_out[VCE_MAX_CHUNKS];
};

inline int pick_threads(int64_t row_bytes) {
    if (row_bytes <= 8 * 1024) return 128;
    if (row_bytes <= 64 * 1024) return 256;
    return 512;
}

template <typename K>
inline int grid_for(K kernel, int nt, int64_t items) {
    const int sms = device_sm_count();
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, nt, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int64_t g = std::min<int64_t>(items, (int64_t)sms * per_sm);
    return (int)std::max<int64_t>(g, 1);
}

// The gradient of every (chunk, row) segment of `tab` (ce_bwd.cu).
// eps_over_v: label smoothing eps / V (0 without smoothing).
cudaError_t launch_ce_bwd(vce_dtype dt, vce_dtype gdt, int nt, const SegTable& tab, const int64_t* labels,
                          const float* row_stats, const float* grad_output, int go_per_row, cudaStream_t s,
                          float eps_over_v = 0.f);

// One-pass forward+backward with each row held in shared memory between its two passes
// (ce_ring.cu).  Sets *launched when it enqueued the kernel; leaves it false, enqueuing
// nothing, when the shape or layout does not fit (fused_ring_layout_ok false, or no cluster
// fits).  eps: label smoothing (0: none).  wait_ns bounds every wait of the kernel; tx_extra > 0
// (tests only) announces that many bytes more per stage than each copy delivers, so no stage
// completes and the waits give up.  reduced != null asks the kernel to reduce the losses into
// *loss_out itself (SUM / MEAN over at most 65536 rows; inv_n is then unused) and reports whether
// it does.  The kernel writes *status itself at its end (the launch's first error code, or 0):
// it needs no clearing before.
cudaError_t launch_fused_ring(vce_dtype dt, vce_dtype gdt, const void* logits, int64_t T, int64_t V, int64_t ld,
                              const int64_t* labels, int64_t ignore_index, int red, const float* grad_output,
                              const float* inv_n, float* loss_rows, float* row_stats, void* grad, int64_t ld_g,
                              int32_t* status, cudaStream_t s, bool* launched, float eps = 0.f,
                              uint64_t wait_ns = 2000000000ull, uint32_t tx_extra = 0, bool* reduced = nullptr,
                              float* loss_out = nullptr);

// Whether launch_fused_ring takes this layout: rows and leading dimensions of whole 16-byte
// vectors, both buffers 16-byte aligned, rows short enough for an 8-CTA cluster; and whether
// it reduces the losses itself for `red` over T rows.
bool fused_ring_layout_ok(vce_dtype dt, int64_t T, int64_t V, int64_t ld, int64_t ld_g, const void* logits,
                          const void* grad);
bool fused_ring_reduces(int red, int64_t T);

// The gradient of every (chunk, row) segment of `tab` with each segment streamed through a
// shared-memory stage ring (ce_bwd_ring.cu; items claimed at run time, ce_slots.cuh): the same
// entries as launch_ce_bwd.  Leaves
// *launched false, enqueuing nothing, unless every input and output chunk row is whole 16-byte
// vectors on a 16-byte boundary.
cudaError_t launch_bwd_ring(vce_dtype dt, vce_dtype gdt, const SegTable& tab, const int64_t* labels,
                            const float* row_stats, const float* grad_output, int go_per_row, float eps_over_v,
                            cudaStream_t s, bool* launched);

// CE forward with each row streamed through a shared-memory stage ring (ce_fwd_ring.cu); eps:
// label smoothing (0: none).  Sets *launched when it enqueued the kernel; leaves it false,
// enqueuing nothing, when the layout does not fit (rows or leading dimension not multiples of
// 8 elements, logits not 16-byte aligned).  For red SUM / MEAN and at most 65536 rows the
// kernel also reduces the losses into *loss_out and writes the rows' weights, and sets
// *reduced.  The kernel writes *status itself at its end (the launch's first error code, or 0):
// it needs no clearing before.  wait_ns bounds every wait of the kernel; tx_extra > 0 (test hook only) announces that many
// more bytes per stage than its copies deliver, so no stage completes.
cudaError_t launch_fwd_ring(vce_dtype dt, const void* logits, int64_t T, int64_t V, int64_t ld, const int64_t* labels,
                            int64_t ignore_index, float eps, int red, float* loss_rows, float* loss_out,
                            float* row_stats, int32_t* status, cudaStream_t s, bool* launched, bool* reduced,
                            uint64_t wait_ns = 2000000000ull, uint32_t tx_extra = 0);

}  // namespace vce
