// Softmax cross-entropy over [T, V] logits: forward row statistics, the reduction, the
// rebuilt gradient, and the vocabulary-chunked variant with its on-device merge.
//
// Method: torchtitan PR #5723 "[loss] fix softmax collapse with improved ce perf"
//   Numerics  - NLL = softplus(logsumexp_{j != t} z_j - z_t), the target dropped before
//               the sum; target gradient p_t - 1 below p_t = 1/4, else -p_non_target;
//               ignored labels finite, then zeroed by the label mask.
//   Memory/perf (compiled form) - the target removed by a column test so the sum is one
//               read of the logits; only per-row statistics saved; the gradient rebuilt
//               in one fused backward pass; bf16 input upcast inside the op.
// Vocabulary chunks: Megatron-core core.tensor_parallel.cross_entropy (per-shard
//   calculate_logits_max / gather_predicted_logits, all-reduce over the TP group),
//   here merged on one device.
//
// Kernels (all stream the rows once, 16-byte vector accesses on the aligned body of
// each row, scalar accesses on an unaligned head and tail):
//   k_ce_fwd        one row per block iteration: (max, sum-exp) over j != t, z_t,
//                   then loss and row statistics
//   k_ce_reduce     one block: fixed-order compensated fp32 sum of the losses, N, and 1/N weights
//   k_ce_bwd        (ce_bwd.cu) one (chunk, row) segment per block iteration: the gradient
//   k_ce_chunk_fwd  one (chunk, row) segment per warp: chunk statistics
//   k_ce_merge      one row per thread: merge the chunk statistics, then as k_ce_fwd
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "vce.h"
#include "vce_device.cuh"
#include "vce_check.cuh"
#include "vce_host.h"
#include "ce_rows.cuh"
#include "ce_segments.h"

namespace vce {
namespace {

// ------------------------------------------------------------------------------------------

// Three blocks of 512 threads per SM (registers capped at 42): the row stream is issue- and
// latency-bound, and 48 resident warps per SM measured 10% faster than 32 at T=16384, V=128256 bf16.
// kSmooth: label smoothing eps > 0 (the row's sum of all logits is reduced alongside; two
// blocks per SM, since the extra sum does not fit in 42 registers).
template <typename S, int NT, bool kSmooth>
__global__ void __launch_bounds__(NT, (kSmooth ? 1024 : 1536) / NT)
    k_ce_fwd(const S* __restrict__ logits, int64_t T, int64_t V, int64_t ld,
                                               const int64_t* __restrict__ labels, int64_t ignore_index,
                                               float eps, float* __restrict__ loss_rows,
                                               float4* __restrict__ row_stats, int32_t* status) {
    __shared__ float sm_m[NT / 32], sm_s[NT / 32], sm_sz[NT / 32];
    __shared__ float sm_zt;
    for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
        const int64_t t = labels[row];
        const bool ignored = (t == ignore_index);
        if (ignored || t < 0 || t >= V) {   // no read of the row: loss 0 (ignored) or NaN (bad label)
            if (threadIdx.x == 0) {
                loss_rows[row] = ignored ? 0.f : __int_as_float(0x7FC00000);
                row_stats[row] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (!ignored) flag_label_error(status);
            }
            continue;
        }
        if (!dbg::ok(row >= 0 && row < T && V <= ld, dbg::kRow)) continue;   // block-uniform
        float m = -kInf, s = 0.f, mb = 0.f, sz = 0.f;
        fwd_segment<S, NT, true, kLoadStream, kSmooth>(logits + row * ld, V, t, m, s, mb, &sm_zt, threadIdx.x, &sz);
        if (kSmooth) {   // block sum of the logits (the barrier below publishes the warp sums)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sz += __shfl_xor_sync(0xFFFFFFFFu, sz, off);
            if ((threadIdx.x & 31) == 0) sm_sz[threadIdx.x >> 5] = sz;
        }
        ms_block_reduce<NT>(m, s, sm_m, sm_s);   // contains the barrier that publishes sm_zt
        if (threadIdx.x == 0) {
            float loss;
            if (kSmooth) {
                float tot = 0.f;
                for (int w = 0; w < NT / 32; ++w) tot += sm_sz[w];
                row_stats[row] = ce_row_finish_smoothed(m, s, sm_zt, tot, V, eps, &loss);
            } else {
                row_stats[row] = ce_row_finish(m, s, sm_zt, &loss);
            }
            loss_rows[row] = loss;
        }
        __syncthreads();
    }
}

// One warp per row, for rows of at most 64 KB: each lane streams its share of the row with
// eight 16-byte loads in flight (six with label smoothing, whose row sum needs registers) and
// the warp reduces with shuffles only, so no block barrier sits between rows and every
// resident warp keeps its loads in flight.  24 warps per SM (80 registers).
constexpr int kWarpRowThreads = 256;

template <typename S, bool kSmooth>
__global__ void __launch_bounds__(kWarpRowThreads, 3)
    k_ce_fwd_warp(const S* __restrict__ logits, int64_t T, int64_t V, int64_t ld, const int64_t* __restrict__ labels,
                  int64_t ignore_index, float eps, float* __restrict__ loss_rows, float4* __restrict__ row_stats,
                  int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kWarpRowThreads / 32);
    for (int64_t row = (int64_t)blockIdx.x * (kWarpRowThreads / 32) + (threadIdx.x >> 5); row < T; row += warps) {
        const int64_t t = labels[row];
        const bool ignored = (t == ignore_index);
        if (ignored || t < 0 || t >= V) {   // no read of the row: loss 0 (ignored) or NaN (bad label)
            if (lane == 0) {
                loss_rows[row] = ignored ? 0.f : __int_as_float(0x7FC00000);
                row_stats[row] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (!ignored) flag_label_error(status);
            }
            continue;
        }
        if (!dbg::ok(row >= 0 && row < T && V <= ld, dbg::kRow)) continue;   // warp-uniform
        float m = -kInf, s = 0.f, mb = 0.f, sz = 0.f;
        float zt_found = kInf;   // stays +inf except in the lane that meets the target
        fwd_segment<S, 32, true, kLoadStream, kSmooth, kSmooth ? 6 : 8>(logits + row * ld, V, t, m, s, mb, &zt_found,
                                                                        lane, &sz);
        ms_warp_reduce(m, s);
        if (kSmooth) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sz += __shfl_xor_sync(0xFFFFFFFFu, sz, off);
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, zt_found != kInf);
        const float zt = hit ? __shfl_sync(0xFFFFFFFFu, zt_found, __ffs(hit) - 1) : 0.f;
        if (lane == 0) {
            float loss;
            row_stats[row] = kSmooth ? ce_row_finish_smoothed(m, s, zt, sz, V, eps, &loss) : ce_row_finish(m, s, zt, &loss);
            loss_rows[row] = loss;
        }
    }
}

// Fixed-order reduction of the per-row losses (one block).  Rows with a bad label add NaN.
// MEAN also writes each valid row's weight 1/N into its statistics.  Thread tid takes rows
// tid + NT (8 j + u), u < 8: eight rows' label and loss loads are in flight before any is
// used, and the validity of up to 64 rows stays in a register mask for the weight pass (longer
// inputs reread their labels there).  The partition is fixed, so the sum is bitwise
// reproducible.
//
// The sum is an fp32 pair (s, c) carried with error-free two-sum steps (Knuth's TwoSum: s + x
// = t + e exactly), so s + c holds the exact sum of the terms up to rounding of the
// compensation itself, far below the fp32 rounding of the result; the pairs merge the same
// way across lanes and warps.  (This device runs fp64 arithmetic at a small fraction of its
// fp32 rate: fp64 partials made this one-block kernel take 17 us at T = 16384.)  Only the
// final division is done in fp64.  A non-finite sum (an inf loss row, or NaN) is s alone.

__device__ __forceinline__ void two_sum_add(float& s, float& c, float x) {
    const float t = s + x;
    const float bp = t - s;
    c += (s - (t - bp)) + (x - bp);
    s = t;
}
__device__ __forceinline__ void two_sum_merge(float& s, float& c, float s2, float c2) {
    two_sum_add(s, c, s2);
    c += c2;
}

template <int NT>
__global__ void __launch_bounds__(NT) k_ce_reduce(const float* __restrict__ loss_rows, const int64_t* __restrict__ labels,
                                                  int64_t T, int64_t V, int64_t ignore_index, int red,
                                                  float* loss_out, float4* row_stats) {
    constexpr int U = 8;
    __shared__ float sm_s[NT / 32], sm_c[NT / 32];
    __shared__ long long sm_n[NT / 32];
    __shared__ float sm_inv;
    float acc = 0.f, comp = 0.f;
    long long n = 0;
    uint64_t valid_mask = 0;   // bit j * U + u: row tid + NT (U j + u) is valid (j < 8)
    int j = 0;
    for (int64_t i0 = threadIdx.x; i0 < T; i0 += (int64_t)NT * U, ++j) {
        int64_t t[U];
        float l[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + (int64_t)u * NT;
            t[u] = i < T ? labels[i] : ignore_index;
            l[u] = i < T ? loss_rows[i] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (t[u] != ignore_index) {
                two_sum_add(acc, comp, l[u]);
                const bool ok = t[u] >= 0 && t[u] < V;
                n += ok ? 1 : 0;
                if (ok && j < 8) valid_mask |= 1ull << (j * U + u);
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float s2 = __shfl_xor_sync(0xFFFFFFFFu, acc, off);
        const float c2 = __shfl_xor_sync(0xFFFFFFFFu, comp, off);
        two_sum_merge(acc, comp, s2, c2);
        n += __shfl_xor_sync(0xFFFFFFFFu, n, off);
    }
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (lane == 0) { sm_s[wid] = acc; sm_c[wid] = comp; sm_n[wid] = n; }
    __syncthreads();
    if (wid == 0) {
        acc = lane < NT / 32 ? sm_s[lane] : 0.f;
        comp = lane < NT / 32 ? sm_c[lane] : 0.f;
        n = lane < NT / 32 ? sm_n[lane] : 0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float s2 = __shfl_xor_sync(0xFFFFFFFFu, acc, off);
            const float c2 = __shfl_xor_sync(0xFFFFFFFFu, comp, off);
            two_sum_merge(acc, comp, s2, c2);
            n += __shfl_xor_sync(0xFFFFFFFFu, n, off);
        }
        if (lane == 0) {
            const double sum = isfinite(acc) ? (double)acc + (double)comp : (double)acc;
            if (red == VCE_RED_MEAN) {
                *loss_out = (float)(sum / (double)n);   // 0/0 = NaN when every row is ignored
                sm_inv = n > 0 ? (float)(1.0 / (double)n) : 0.f;
            } else {
                *loss_out = (float)sum;
            }
        }
    }
    if (red != VCE_RED_MEAN) return;
    __syncthreads();
    const float inv = sm_inv;
    j = 0;
    for (int64_t i0 = threadIdx.x; i0 < T; i0 += (int64_t)NT * U, ++j) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + (int64_t)u * NT;
            if (i >= T) break;
            bool ok;
            if (j < 8) {
                ok = (valid_mask >> (j * U + u)) & 1ull;
            } else {
                const int64_t t = labels[i];
                ok = t != ignore_index && t >= 0 && t < V;
            }
            if (ok) row_stats[i].w = inv;
        }
    }
}

// ------------------------------------------------------------------------------------------
// Vocabulary chunks: per-(chunk, row) statistics, then a per-row merge.

// One warp per (chunk, row) item, items row-major over chunks: a chunk row (32 KB for 8
// chunks of a 128256-entry bf16 row) is too short to amortise block barriers, so each warp streams its item
// and reduces with shuffles only.  The maximum is exact (ms_push), as the statistics report it.
constexpr int kChunkThreads = 512;

// kSumZ (label smoothing): also each item's sum of logits into chunk_sums [k][T].
template <typename S, bool kSumZ>
__global__ void __launch_bounds__(kChunkThreads, 2) k_ce_chunk_fwd(const __grid_constant__ SegTable tab,
                                                                   const int64_t* __restrict__ labels,
                                                                   int64_t ignore_index,
                                                                   float4* __restrict__ chunk_stats,
                                                                   float* __restrict__ chunk_sums) {
    const int lane = threadIdx.x & 31;
    const int64_t items = tab.T * tab.k;
    const int64_t warps = (int64_t)gridDim.x * (kChunkThreads / 32);
    for (int64_t it = (int64_t)blockIdx.x * (kChunkThreads / 32) + (threadIdx.x >> 5); it < items; it += warps) {
        const int64_t row = it / tab.k;
        const int c = (int)(it - row * tab.k);
        if (!dbg::ok(c >= 0 && c < tab.k && row < tab.T, dbg::kChunk) ||
            !dbg::ok(tab.width[c] <= tab.ld_in[c], dbg::kCols))
            continue;   // warp-uniform
        const int64_t t = labels[row];
        const int64_t w = tab.width[c];
        const int64_t tl = (t == ignore_index) ? -1 : t - tab.off[c];
        const bool owner = (tl >= 0 && tl < w);
        float m = -kInf, s = 0.f, mb = 0.f, zt = 0.f;
        float zt_found = kInf;   // stays +inf except in the lane that meets the target
        float sz = 0.f;
        fwd_segment<S, 32, false, kLoadStream, kSumZ>(reinterpret_cast<const S*>(tab.in[c]) + row * tab.ld_in[c], w,
                                                      owner ? tl : -1, m, s, mb, &zt_found, lane, &sz);
        ms_warp_reduce(m, s);
        if (kSumZ) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sz += __shfl_xor_sync(0xFFFFFFFFu, sz, off);
            if (lane == 0) chunk_sums[(int64_t)c * tab.T + row] = sz;
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, zt_found != kInf);
        if (hit) zt = __shfl_sync(0xFFFFFFFFu, zt_found, __ffs(hit) - 1);
        if (lane == 0)
            chunk_stats[(int64_t)c * tab.T + row] = make_float4(m, s, owner ? zt : 0.f, owner ? 1.f : 0.f);
    }
}

// chunk_sums != NULL: label smoothing eps; the row's sum of logits is the chunks' sums added in
// chunk order.
__global__ void k_ce_merge(const float4* __restrict__ chunk_stats, int k, int64_t T, int64_t V,
                           const int64_t* __restrict__ labels, int64_t ignore_index, float* __restrict__ loss_rows,
                           float4* __restrict__ row_stats, int32_t* status, const float* __restrict__ chunk_sums,
                           float eps) {
    for (int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; row < T; row += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = labels[row];
        const bool ignored = (t == ignore_index);
        if (ignored || t < 0 || t >= V) {
            loss_rows[row] = ignored ? 0.f : __int_as_float(0x7FC00000);
            row_stats[row] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (!ignored) flag_label_error(status);
            continue;
        }
        float M = -kInf, S = 0.f, zt = 0.f;
        for (int c = 0; c < k; ++c) {
            const float4 cs = chunk_stats[(int64_t)c * T + row];
            ms_merge(M, S, cs.x, cs.y);
            if (cs.w != 0.f) zt = cs.z;
        }
        float loss;
        if (chunk_sums) {
            float tot = 0.f;
            for (int c = 0; c < k; ++c) tot += chunk_sums[(int64_t)c * T + row];
            row_stats[row] = ce_row_finish_smoothed(M, S, zt, tot, V, eps, &loss);
        } else {
            row_stats[row] = ce_row_finish(M, S, zt, &loss);
        }
        loss_rows[row] = loss;
    }
}

// The merge for many partials per row (the linear-CE's per-tile statistics, 501 tiles at V =
// 128256): one thread per row merges its k partials one after another, and 8192 rows keep only
// 32 SMs busy (0.146 ms per call).  Here a block takes 32 consecutive rows (one per lane) and
// its kSeg warps split the partials into contiguous ranges, so each load instruction reads
// 32 consecutive rows' partials of one tile; warp 0 then merges the kSeg ranges in order and
// finishes the row.  The partition is fixed, so the result is reproducible.
constexpr int kMergeSeg = 8;

__global__ void __launch_bounds__(32 * kMergeSeg) k_ce_merge_seg(const float4* __restrict__ chunk_stats, int k,
                                                                int64_t T, int64_t V,
                                                                const int64_t* __restrict__ labels,
                                                                int64_t ignore_index, float* __restrict__ loss_rows,
                                                                float4* __restrict__ row_stats, int32_t* status) {
    __shared__ float4 part[kMergeSeg][32];   // (m, s, z_t, owner) of each range, per row
    const int lane = threadIdx.x & 31, seg = threadIdx.x >> 5;
    const int c0 = (int)((int64_t)k * seg / kMergeSeg), c1 = (int)((int64_t)k * (seg + 1) / kMergeSeg);
    for (int64_t base = (int64_t)blockIdx.x * 32; base < T; base += (int64_t)gridDim.x * 32) {
        const int64_t row = base + lane;
        const int64_t t = row < T ? labels[row] : ignore_index;
        const bool valid = row < T && t != ignore_index && t >= 0 && t < V;
        float M = -kInf, S = 0.f, zt = 0.f, own = 0.f;
        if (valid) {
            int c = c0;
            for (; c + 4 <= c1; c += 4) {   // four partials in flight before any is merged
                float4 cs[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) cs[u] = chunk_stats[(int64_t)(c + u) * T + row];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    ms_merge(M, S, cs[u].x, cs[u].y);
                    if (cs[u].w != 0.f) { zt = cs[u].z; own = 1.f; }
                }
            }
            for (; c < c1; ++c) {
                const float4 cs = chunk_stats[(int64_t)c * T + row];
                ms_merge(M, S, cs.x, cs.y);
                if (cs.w != 0.f) { zt = cs.z; own = 1.f; }
            }
        }
        part[seg][lane] = make_float4(M, S, zt, own);
        __syncthreads();
        if (seg == 0 && row < T) {
            if (!valid) {
                loss_rows[row] = (t == ignore_index) ? 0.f : __int_as_float(0x7FC00000);
                row_stats[row] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (t != ignore_index) flag_label_error(status);
            } else {
                float Mr = -kInf, Sr = 0.f, ztr = 0.f;
#pragma unroll
                for (int g = 0; g < kMergeSeg; ++g) {
                    const float4 pg = part[g][lane];
                    ms_merge(Mr, Sr, pg.x, pg.y);
                    if (pg.w != 0.f) ztr = pg.z;
                }
                float loss;
                row_stats[row] = ce_row_finish(Mr, Sr, ztr, &loss);
                loss_rows[row] = loss;
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------------------------------
// host side

template <typename S, int NT>
cudaError_t launch_fwd(const void* logits, int64_t T, int64_t V, int64_t ld, const int64_t* labels, int64_t ig,
                       float eps, float* loss_rows, float* row_stats, int32_t* status, cudaStream_t s) {
    auto kern = eps > 0.f ? k_ce_fwd<S, NT, true> : k_ce_fwd<S, NT, false>;
    kern<<<grid_for(kern, NT, T), NT, 0, s>>>(reinterpret_cast<const S*>(logits), T, V, ld, labels, ig, eps,
                                              loss_rows, reinterpret_cast<float4*>(row_stats), status);
    return cudaGetLastError();
}

template <typename S>
cudaError_t launch_fwd_warp(const void* logits, int64_t T, int64_t V, int64_t ld, const int64_t* labels, int64_t ig,
                            float eps, float* loss_rows, float* row_stats, int32_t* status, cudaStream_t s) {
    auto kern = eps > 0.f ? k_ce_fwd_warp<S, true> : k_ce_fwd_warp<S, false>;
    const int64_t blocks = (T + kWarpRowThreads / 32 - 1) / (kWarpRowThreads / 32);
    kern<<<grid_for(kern, kWarpRowThreads, blocks), kWarpRowThreads, 0, s>>>(
        reinterpret_cast<const S*>(logits), T, V, ld, labels, ig, eps, loss_rows, reinterpret_cast<float4*>(row_stats),
        status);
    return cudaGetLastError();
}

template <typename S>
cudaError_t launch_chunk_fwd(const SegTable& tab, const int64_t* labels, int64_t ig, float* ws, float* sums,
                             cudaStream_t s) {
    auto kern = sums ? k_ce_chunk_fwd<S, true> : k_ce_chunk_fwd<S, false>;
    const int64_t blocks_needed = (tab.T * tab.k + kChunkThreads / 32 - 1) / (kChunkThreads / 32);
    kern<<<grid_for(kern, kChunkThreads, blocks_needed), kChunkThreads, 0, s>>>(tab, labels, ig,
                                                                               reinterpret_cast<float4*>(ws), sums);
    return cudaGetLastError();
}

template <typename S>
cudaError_t dispatch_fwd(int nt, const void* logits, int64_t T, int64_t V, int64_t ld, const int64_t* labels,
                         int64_t ig, float eps, float* lr, float* rs, int32_t* st, cudaStream_t s) {
    if (nt == 128) return launch_fwd<S, 128>(logits, T, V, ld, labels, ig, eps, lr, rs, st, s);
    if (nt == 256) return launch_fwd<S, 256>(logits, T, V, ld, labels, ig, eps, lr, rs, st, s);
    return launch_fwd<S, 512>(logits, T, V, ld, labels, ig, eps, lr, rs, st, s);
}


cudaError_t launch_reduce(const float* loss_rows, const int64_t* labels, int64_t T, int64_t V, int64_t ig, int red,
                          float* loss_out, float* row_stats, cudaStream_t s) {
    k_ce_reduce<1024><<<1, 1024, 0, s>>>(loss_rows, labels, T, V, ig, red, loss_out,
                                         reinterpret_cast<float4*>(row_stats));
    return cudaGetLastError();
}

int check_common(vce_dtype dt, vce_reduction red, int64_t T) {
    if (dt != VCE_F32 && dt != VCE_BF16) return VCE_ERR_DTYPE;
    if (red != VCE_RED_NONE && red != VCE_RED_SUM && red != VCE_RED_MEAN) return VCE_ERR_DTYPE;
    if (T < 0) return VCE_ERR_SHAPE;
    return VCE_OK;
}

}  // namespace

VCE_DEBUG_READER(debug_word_ce_fwd)

cudaError_t launch_stats_merge(const float* part, int k, int64_t T, int64_t V, const int64_t* labels,
                               int64_t ignore_index, float* loss_rows, float* row_stats, int32_t* status,
                               cudaStream_t s) {
    if (k >= 4 * kMergeSeg) {   // many partials per row: ranges of them per warp
        const int64_t blocks = (T + 31) / 32;
        const int mg = (int)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)device_sm_count() * 8));
        k_ce_merge_seg<<<mg, 32 * kMergeSeg, 0, s>>>(reinterpret_cast<const float4*>(part), k, T, V, labels,
                                                      ignore_index, loss_rows, reinterpret_cast<float4*>(row_stats),
                                                      status);
        return cudaGetLastError();
    }
    const int mt = 256;
    const int mg = (int)std::max<int64_t>(1, std::min<int64_t>((T + mt - 1) / mt, (int64_t)device_sm_count() * 8));
    k_ce_merge<<<mg, mt, 0, s>>>(reinterpret_cast<const float4*>(part), k, T, V, labels, ignore_index, loss_rows,
                                 reinterpret_cast<float4*>(row_stats), status, nullptr, 0.f);
    return cudaGetLastError();
}

cudaError_t launch_loss_reduce(const float* loss_rows, const int64_t* labels, int64_t T, int64_t V,
                               int64_t ignore_index, int red, float* loss_out, float* row_stats, cudaStream_t s) {
    return launch_reduce(loss_rows, labels, T, V, ignore_index, red, loss_out, row_stats, s);
}

}  // namespace vce

using namespace vce;

extern "C" int ce_forward_ls(const void* logits, vce_dtype dt, int64_t T, int64_t V, int64_t ld,
                             const int64_t* labels, int64_t ignore_index, float label_smoothing, vce_reduction red, float* loss_rows, float* loss_out, float* row_stats,
                          int32_t* status, vce_stream_t s) {
    int rc = check_common(dt, red, T);
    if (rc) return rc;
    if (!(label_smoothing >= 0.f && label_smoothing < 1.f)) return VCE_ERR_ARG;
    if (V < 1) return VCE_ERR_SHAPE;
    if (ld < V) return VCE_ERR_LD;
    if (!status || (red != VCE_RED_NONE && !loss_out)) return VCE_ERR_NULL;
    const size_t es = dt == VCE_BF16 ? 2 : 4;
    if (T > 0) {
        if (!logits || !labels || !loss_rows || !row_stats) return VCE_ERR_NULL;
        if (!fits_bytes(T, ld, es)) return VCE_ERR_SHAPE;
        if (!aligned(logits, es) || !aligned(labels, 8) || !aligned(loss_rows, 4) || !aligned(row_stats, 16))
            return VCE_ERR_ALIGN;
    }
    if (red != VCE_RED_NONE && !aligned(loss_out, 4)) return VCE_ERR_ALIGN;
    if ((rc = require_sm100())) return rc;
    bool reduced = false;   // the ring kernel reduced the losses itself
    // The ring kernel writes the status word itself (its launch slot carries the error code);
    // every other path clears it first and merges codes into it.
    auto clear_status = [&]() { return cudaMemsetAsync(status, 0, sizeof(int32_t), s) == cudaSuccess; };
    if (T == 0 && !clear_status()) return VCE_ERR_CUDA;
    if (T > 0) {
        // Rows of at most 32 KB: one warp per row (k_ce_fwd_warp; 8192 x 16000 bf16: 0.070 ms,
        // against 0.080 on the stage ring and 0.102 on the ring's four consumer groups).  Longer
        // rows of whole 16-byte vectors stream through the shared-memory stage ring (rows of
        // two stages with its consumers in two groups: 4096 x 32000 bf16, 0.052 ms back to back,
        // against 0.0613 on one block per row), other layouts one block per row with global loads.
        bool launched = false;
        const int64_t row_bytes = V * (int64_t)es;
        cudaError_t e = cudaSuccess;
        if (row_bytes <= 32768) {
            if (!clear_status()) return VCE_ERR_CUDA;
            e = dt == VCE_BF16 ? launch_fwd_warp<uint16_t>(logits, T, V, ld, labels, ignore_index, label_smoothing,
                                                           loss_rows, row_stats, status, s)
                               : launch_fwd_warp<float>(logits, T, V, ld, labels, ignore_index, label_smoothing,
                                                        loss_rows, row_stats, status, s);
            launched = true;
        } else {
            e = launch_fwd_ring(dt, logits, T, V, ld, labels, ignore_index, label_smoothing, red, loss_rows, loss_out,
                                row_stats, status, s, &launched, &reduced);
        }
        if (e == cudaSuccess && !launched) {
            if (!clear_status()) return VCE_ERR_CUDA;
            const int nt = pick_threads(row_bytes);
            e = dt == VCE_BF16 ? dispatch_fwd<uint16_t>(nt, logits, T, V, ld, labels, ignore_index, label_smoothing,
                                                        loss_rows, row_stats, status, s)
                               : dispatch_fwd<float>(nt, logits, T, V, ld, labels, ignore_index, label_smoothing,
                                                     loss_rows, row_stats, status, s);
        }
        if (e != cudaSuccess) return VCE_ERR_CUDA;
    }
    if (red != VCE_RED_NONE && !reduced &&
        launch_reduce(loss_rows, labels, T, V, ignore_index, red, loss_out, row_stats, s) != cudaSuccess)
        return VCE_ERR_CUDA;
    return VCE_OK;
}

extern "C" int ce_forward(const void* logits, vce_dtype dt, int64_t T, int64_t V, int64_t ld, const int64_t* labels,
                          int64_t ignore_index, vce_reduction red, float* loss_rows, float* loss_out, float* row_stats,
                          int32_t* status, vce_stream_t s) {
    return ce_forward_ls(logits, dt, T, V, ld, labels, ignore_index, 0.f, red, loss_rows, loss_out, row_stats, status, s);
}

extern "C" int ce_merge_chunks_ls(int k, const void* const* chunk_logits, const int64_t* chunk_width,
                                  const int64_t* chunk_ld, vce_dtype dt, int64_t T, const int64_t* labels,
                                  int64_t ignore_index, float label_smoothing, vce_reduction red, float* loss_rows,
                                  float* loss_out, float* row_stats, const float* grad_output,
                                  void* const* chunk_grads, const int64_t* chunk_grad_ld, vce_dtype grad_dt,
                                  float* chunk_stats_ws, float* chunk_sums_ws, int32_t* status, vce_stream_t s) {
    int rc = check_common(dt, red, T);
    if (rc) return rc;
    if (!(label_smoothing >= 0.f && label_smoothing < 1.f)) return VCE_ERR_ARG;
    const bool smooth = label_smoothing > 0.f;
    if (k < 1 || k > VCE_MAX_CHUNKS) return VCE_ERR_ARG;
    if (!chunk_logits || !chunk_width || !chunk_ld || !status) return VCE_ERR_NULL;
    if (red != VCE_RED_NONE && !loss_out) return VCE_ERR_NULL;
    if (chunk_grads && grad_dt != VCE_F32 && grad_dt != VCE_BF16) return VCE_ERR_DTYPE;
    const size_t es = dt == VCE_BF16 ? 2 : 4, gs = grad_dt == VCE_BF16 ? 2 : 4;
    SegTable tab{};
    tab.k = k;
    tab.T = T;
    int64_t V = 0, max_w = 0;
    for (int c = 0; c < k; ++c) {
        const int64_t w = chunk_width[c];
        if (w < 1) return VCE_ERR_SHAPE;
        if (chunk_ld[c] < w) return VCE_ERR_LD;
        const int64_t gld = chunk_grad_ld ? chunk_grad_ld[c] : w;
        if (chunk_grads && gld < w) return VCE_ERR_LD;
        if (T > 0) {
            if (!chunk_logits[c] || (chunk_grads && !chunk_grads[c])) return VCE_ERR_NULL;
            if (!fits_bytes(T, chunk_ld[c], es) || (chunk_grads && !fits_bytes(T, gld, gs))) return VCE_ERR_SHAPE;
            if (!aligned(chunk_logits[c], es) || (chunk_grads && !aligned(chunk_grads[c], gs))) return VCE_ERR_ALIGN;
        }
        tab.in[c] = chunk_logits[c];
        tab.out[c] = chunk_grads ? chunk_grads[c] : nullptr;
        tab.width[c] = w;
        tab.off[c] = V;
        tab.ld_in[c] = chunk_ld[c];
        tab.ld_out[c] = gld;
        if (V > INT64_MAX - w) return VCE_ERR_SHAPE;
        V += w;
        max_w = std::max(max_w, w);
    }
    if (T > 0) {
        if (!labels || !loss_rows || !row_stats || !chunk_stats_ws || (chunk_grads && !grad_output))
            return VCE_ERR_NULL;
        if (smooth && !chunk_sums_ws) return VCE_ERR_NULL;
        if (!aligned(labels, 8) || !aligned(loss_rows, 4) || !aligned(row_stats, 16) || !aligned(chunk_stats_ws, 16) ||
            (smooth && !aligned(chunk_sums_ws, 4)))
            return VCE_ERR_ALIGN;
        if (!fits_bytes(T, (int64_t)k * VCE_CHUNK_STATS, 4)) return VCE_ERR_SHAPE;
    }
    if ((rc = require_sm100())) return rc;
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return VCE_ERR_CUDA;
    if (T > 0) {
        float* sums = smooth ? chunk_sums_ws : nullptr;
        cudaError_t e = dt == VCE_BF16 ? launch_chunk_fwd<uint16_t>(tab, labels, ignore_index, chunk_stats_ws, sums, s)
                                       : launch_chunk_fwd<float>(tab, labels, ignore_index, chunk_stats_ws, sums, s);
        if (e != cudaSuccess) return VCE_ERR_CUDA;
        const int mt = 256;
        const int mg = (int)std::min<int64_t>((T + mt - 1) / mt, (int64_t)device_sm_count() * 8);
        k_ce_merge<<<mg, mt, 0, s>>>(reinterpret_cast<const float4*>(chunk_stats_ws), k, T, V, labels, ignore_index,
                                     loss_rows, reinterpret_cast<float4*>(row_stats), status, sums, label_smoothing);
        if (cudaGetLastError() != cudaSuccess) return VCE_ERR_CUDA;
    }
    if (red != VCE_RED_NONE &&
        launch_reduce(loss_rows, labels, T, V, ignore_index, red, loss_out, row_stats, s) != cudaSuccess)
        return VCE_ERR_CUDA;
    if (chunk_grads && T > 0) {
        // Chunk rows streamed through shared memory where every chunk's layout allows it.
        const float eps_over_v = label_smoothing / (float)V;
        bool launched = false;
        cudaError_t e = launch_bwd_ring(dt, grad_dt, tab, labels, row_stats, grad_output, red == VCE_RED_NONE,
                                        eps_over_v, s, &launched);
        if (e == cudaSuccess && !launched) {
            const int nt = pick_threads(max_w * (int64_t)es);
            e = launch_ce_bwd(dt, grad_dt, nt, tab, labels, row_stats, grad_output, red == VCE_RED_NONE, s, eps_over_v);
        }
        if (e != cudaSuccess) return VCE_ERR_CUDA;
    }
    return VCE_OK;
}

extern "C" int ce_merge_chunks(int k, const void* const* chunk_logits, const int64_t* chunk_width,
                               const int64_t* chunk_ld, vce_dtype dt, int64_t T, const int64_t* labels,
                               int64_t ignore_index, vce_reduction red, float* loss_rows, float* loss_out,
                               float* row_stats, const float* grad_output, void* const* chunk_grads,
                               const int64_t* chunk_grad_ld, vce_dtype grad_dt, float* chunk_stats_ws,
                               int32_t* status, vce_stream_t s) {
    return ce_merge_chunks_ls(k, chunk_logits, chunk_width, chunk_ld, dt, T, labels, ignore_index, 0.f, red,
                              loss_rows, loss_out, row_stats, grad_output, chunk_grads, chunk_grad_ld, grad_dt,
                              chunk_stats_ws, nullptr, status, s);
}
