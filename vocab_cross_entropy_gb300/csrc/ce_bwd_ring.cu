// CE backward (ce_backward, and the gradient step of ce_merge_chunks) for rows that suit bulk
// copies: each row, or each chunk of a row, streams through a shared-memory stage ring and its
// gradient is written from there.
//
// Method: torchtitan PR #5723 "[loss] fix softmax collapse with improved ce perf" (Numerics:
// the gradient rebuilt from the logits and the row statistics, the p_t = 1/4 branch) — the same
// per-element arithmetic as k_ce_bwd (grad = coef * 2^(z log2 e - bias), the target entry gt).
//
// Items are (row, chunk) pairs of a segment table, row-major over its k chunks (k = 1 for a
// [T, V] matrix).  One CTA per SM walks the items blockIdx.x, blockIdx.x + gridDim.x, ... with
// three roles:
//   producer warp   reads the row statistics of 32 items at a time (one per lane); lane 0
//                   publishes each weighted item's row, chunk, coefficients (coef, bias, target
//                   gradient, smoothing shift) and target column, and streams the item into a
//                   ring of seven 32 KB stages with bulk asynchronous copies (cp.async.bulk)
//   consumer warps  per stage, a thread's 4 x 16-byte vectors to gradient entries stored with
//                   16-byte streaming stores (stage::bwd_stage); the stage goes back to the
//                   producer right away
//   zero warp       writes +0.0 over the gradient of items of weight 0 (ignored or invalid
//                   labels), whose logits are not read
// Every wait is bounded (2 s).  A wait that gives up sets the CTA's abort flag; every role then
// keeps its arrivals but skips the work and later waits.  ce_backward has no status word, so
// the gradient is then undefined without a report.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "ce_segments.h"
#include "ce_stage.cuh"
#include "vce.h"
#include "vce_async.cuh"
#include "vce_device.cuh"
#include "vce_check.cuh"
#include "vce_host.h"

namespace vce {
namespace bring {

constexpr int kChunk = 32768;          // bytes per stage (one bulk copy)
constexpr int kStages = 7;
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps, kZeroWarp = kConsumerWarps + 1;
constexpr int kThreads = kConsumers + 64;
constexpr int kVecPerThread = kChunk / 16 / kConsumers;
constexpr int kInfoSlots = 16;         // > the rows the producer can run ahead (kStages, at one stage a row)
static_assert(kVecPerThread * kConsumers * 16 == kChunk, "every consumer takes the same whole vectors of a stage");

// A weighted item of the CTA's sequence: where its gradient goes and how it is formed.
struct RowInfo {
    int64_t row;
    int tl;                            // target column within the chunk (-1: not in it)
    int c;                             // chunk
    float coef, bias, gt, shift;
};

struct alignas(16) Ctl {
    RowInfo info[kInfoSlots];          // by the row's index in the sequence, mod kInfoSlots
    uint64_t full[kStages];            // stage loaded
    uint64_t empty[kStages];           // stage released (one arrival per consumer warp)
    int abort;
};
constexpr int kSmemBytes = kStages * kChunk + (int)sizeof(Ctl);

struct Args {
    const int64_t* labels;
    const float4* row_stats;           // (L', 1 - p_t, target coefficient, weight); weight 0: no gradient
    const float* grad_output;
    int go_per_row;
    float eps_over_v;                  // label smoothing eps / V (0: none)
    uint64_t wait_ns;
};

template <typename S, typename O, bool kShift>
__global__ void __launch_bounds__(kThreads, 1) k_ce_bwd_ring(const __grid_constant__ Args a,
                                                             const __grid_constant__ SegTable tab) {
    constexpr int G = Elt<S>::kGroup;
    constexpr int64_t es = sizeof(S);
    extern __shared__ __align__(128) uint8_t smem[];
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem + kStages * kChunk);
    volatile int* abort_flag = &ctl.abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t stride = gridDim.x, items = tab.T * tab.k;
    auto stages_of = [&](int c) { return (int)((tab.width[c] * es + kChunk - 1) / kChunk); };

    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; ++st) {
            tc::mbar_init(&ctl.full[st], 1);
            tc::mbar_init(&ctl.empty[st], kConsumerWarps);
        }
        for (int i = 0; i < kInfoSlots; ++i) ctl.info[i] = RowInfo{-1, -1, 0, 0.f, 0.f, 0.f, 0.f};
        ctl.abort = 0;
        tc::fence_mbar_init();
    }
    __syncthreads();

    // The number of items of this CTA with a nonzero weight (each warp counts for itself).
    auto count_valid = [&]() {
        int n = 0;
#pragma unroll 4
        for (int64_t it = blockIdx.x + (int64_t)lane * stride; it < items; it += 32 * stride)
            n += a.row_stats[it / tab.k].w != 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) n += __shfl_xor_sync(0xFFFFFFFFu, n, off);
        return n;
    };

    if (warp == kProducerWarp) {
        // ---------------- producer ----------------
        uint32_t q = 0, e = 0;
        bool stop = false;
        for (int64_t base = blockIdx.x; base < items && !stop; base += 32 * stride) {
            const int64_t my = base + (int64_t)lane * stride;
            const float4 st_my = my < items ? a.row_stats[my / tab.k] : make_float4(0.f, 0.f, 0.f, 0.f);
            uint32_t todo = __ballot_sync(0xFFFFFFFFu, st_my.w != 0.f);
            while (todo && !stop) {
                const int b = __ffs(todo) - 1;
                todo &= todo - 1;
                const float sx = __shfl_sync(0xFFFFFFFFu, st_my.x, b), sy = __shfl_sync(0xFFFFFFFFu, st_my.y, b);
                const float sz = __shfl_sync(0xFFFFFFFFu, st_my.z, b), sw = __shfl_sync(0xFFFFFFFFu, st_my.w, b);
                if (lane == 0) {
                    const int64_t it = base + (int64_t)b * stride;
                    const int64_t row = it / tab.k;
                    const int c = (int)(it - row * tab.k);
                    const int64_t t = a.labels[row], off = tab.off[c], w = tab.width[c];
                    const float cg = a.grad_output[a.go_per_row ? row : 0] * sw;
                    // the item's coefficients, published with its first stage
                    ctl.info[e % kInfoSlots] = RowInfo{row, (t >= off && t < off + w) ? (int)(t - off) : -1, c,
                                                       cg * sy, (sx == -kInf) ? 0.f : sx * kLog2e, cg * sz,
                                                       cg * a.eps_over_v};
                    const char* src = static_cast<const char*>(tab.in[c]) + row * tab.ld_in[c] * es;
                    const int64_t bytes = w * es;
                    const int nchunk = stages_of(c);
                    for (int j = 0; j < nchunk; ++j) {
                        const int st = (int)(q % kStages);
                        if (!tc::mbar_wait(&ctl.empty[st], ((q / kStages) & 1) ^ 1, abort_flag, nullptr, 0,
                                           a.wait_ns)) {
                            stop = true;
                            break;
                        }
                        const uint32_t nb = (uint32_t)std::min<int64_t>(kChunk, bytes - (int64_t)j * kChunk);
                        if (!dbg::ok(row < tab.T && c < tab.k && (int64_t)j * kChunk + nb <= bytes &&
                                         w <= tab.ld_in[c],
                                     dbg::kCols)) {
                            *abort_flag = 1;   // no copy: the other roles stop at their next wait
                            stop = true;
                            break;
                        }
                        tc::mbar_arrive_expect_tx(&ctl.full[st], nb);
                        tc::bulk_load(smem + st * kChunk, src + (int64_t)j * kChunk, nb, &ctl.full[st]);
                        ++q;
                    }
                    ++e;
                    stop = stop || *abort_flag;
                }
                stop = __shfl_sync(0xFFFFFFFFu, stop, 0);
            }
        }
        if (lane == 0) {   // copies still in flight (only after an abort) land before the CTA may exit
            int never = 0;
            for (uint32_t p = q > (uint32_t)kStages ? q - kStages : 0; p < q; ++p)
                tc::mbar_wait(&ctl.full[p % kStages], (p / kStages) & 1, &never, nullptr, 0, a.wait_ns);
        }
        __syncwarp();
    } else if (warp == kZeroWarp) {
        // ---------------- items of weight 0: gradient +0.0 by selection ----------------
        for (int64_t base = blockIdx.x; base < items; base += 32 * stride) {
            const int64_t my = base + (int64_t)lane * stride;
            uint32_t bad = __ballot_sync(0xFFFFFFFFu, my < items && a.row_stats[my / tab.k].w == 0.f);
            while (bad) {
                const int b = __ffs(bad) - 1;
                bad &= bad - 1;
                const int64_t it = base + (int64_t)b * stride;
                const int64_t row = it / tab.k;
                const int c = (int)(it - row * tab.k);
                if (!dbg::ok(row < tab.T && c < tab.k && tab.width[c] <= tab.ld_out[c], dbg::kCols)) continue;
                O* grow = static_cast<O*>(tab.out[c]) + row * tab.ld_out[c];
                const float zero[G] = {};
                for (int64_t vi = lane; vi < tab.width[c] / G; vi += 32) GroupStore<O, G>::run(grow + vi * G, zero);
            }
        }
    } else {
        // ---------------- consumers ----------------
        const int tid = threadIdx.x;
        const int nv = count_valid();
        uint32_t q = 0;   // ring chunk of the current item's first stage
        for (int e = 0; e < nv; ++e) {
            RowInfo ri{-1, -1, 0, 0.f, 0.f, 0.f, 0.f};
            O* grow = nullptr;
            int nchunk = 1;
            int64_t bytes = 0;
            for (int j = 0; j < nchunk; ++j) {
                const uint32_t p = q + j;
                const int st = (int)(p % kStages);
                const bool ok = tc::mbar_wait(&ctl.full[st], (p / kStages) & 1, abort_flag, nullptr, 0, a.wait_ns);
                if (j == 0) {   // the item is known once its first stage has landed
                    ri = ctl.info[e % kInfoSlots];
                    const bool in_range = ri.row >= 0 && ri.row < tab.T && ri.c >= 0 && ri.c < tab.k;   // else: aborted
                    const int c = in_range ? ri.c : 0;
                    grow = in_range ? static_cast<O*>(tab.out[c]) + ri.row * tab.ld_out[c] : nullptr;
                    bytes = tab.width[c] * es;
                    nchunk = stages_of(c);
                }
                if (ok && grow && !*abort_flag) {
                    const uint4* buf = reinterpret_cast<const uint4*>(smem + st * kChunk);
                    const int nvec = (int)(std::min<int64_t>(kChunk, bytes - (int64_t)j * kChunk) / 16);
                    const int col0 = j * (kChunk / (int)sizeof(S));
                    const int rel0 = ri.tl - (col0 + tid * G);
                    if (!dbg::ok((int64_t)col0 + (int64_t)nvec * G <= bytes / es && nvec <= kChunk / 16, dbg::kCols))
                        ;   // the stage's columns would leave the item's row: no store
                    else if (nvec == kVecPerThread * kConsumers)
                        stage::bwd_stage<S, O, kConsumers, kVecPerThread, true, kShift>(
                            buf, nvec, grow + col0, rel0, tid, ri.coef, ri.bias, ri.gt, ri.shift);
                    else
                        stage::bwd_stage<S, O, kConsumers, kVecPerThread, false, kShift>(
                            buf, nvec, grow + col0, rel0, tid, ri.coef, ri.bias, ri.gt, ri.shift);
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&ctl.empty[st]);
            }
            q += nchunk;
        }
    }
}

template <typename S, typename O>
cudaError_t launch(const Args& args, const SegTable& tab, cudaStream_t s) {
    auto kern = args.eps_over_v > 0.f ? k_ce_bwd_ring<S, O, true> : k_ce_bwd_ring<S, O, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(device_sm_count(), tab.T * tab.k);
    kern<<<grid, kThreads, kSmemBytes, s>>>(args, tab);
    return cudaGetLastError();
}

}  // namespace bring

VCE_DEBUG_READER(debug_word_ce_bwd_ring)

cudaError_t launch_bwd_ring(vce_dtype dt, vce_dtype gdt, const SegTable& tab, const int64_t* labels,
                            const float* row_stats, const float* grad_output, int go_per_row, float eps_over_v,
                            cudaStream_t s, bool* launched) {
    using namespace bring;
    *launched = false;
    const int64_t es = dt == VCE_BF16 ? 2 : 4, gs = gdt == VCE_BF16 ? 2 : 4;
    if (tab.T < 1) return cudaSuccess;
    // every input and output chunk row starts on a 16-byte boundary and is whole 16-byte vectors
    for (int c = 0; c < tab.k; ++c)
        if (tab.width[c] % 8 || tab.ld_in[c] % 8 || tab.ld_out[c] % 8 || !aligned(tab.in[c], 16) ||
            !aligned(tab.out[c], 16) || tab.width[c] > ((int64_t)1 << 30) / std::max(es, gs))
            return cudaSuccess;
    const Args args{labels, reinterpret_cast<const float4*>(row_stats), grad_output, go_per_row, eps_over_v,
                    tc::kWaitNs};
    cudaError_t e;
    if (dt == VCE_BF16 && gdt == VCE_BF16) e = launch<uint16_t, uint16_t>(args, tab, s);
    else if (dt == VCE_BF16) e = launch<uint16_t, float>(args, tab, s);
    else if (gdt == VCE_BF16) e = launch<float, uint16_t>(args, tab, s);
    else e = launch<float, float>(args, tab, s);
    if (e == cudaSuccess) *launched = true;
    return e;
}

}  // namespace vce
