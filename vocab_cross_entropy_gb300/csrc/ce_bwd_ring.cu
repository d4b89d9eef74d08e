// CE backward (ce_backward, and the gradient step of ce_merge_chunks) for rows that suit bulk
// copies: each row, or each chunk of a row, streams through a shared-memory stage ring and its
// gradient is written from there.
//
// Method: torchtitan PR #5723 "[loss] fix softmax collapse with improved ce perf" (Numerics:
// the gradient rebuilt from the logits and the row statistics, the p_t = 1/4 branch) — the same
// per-element arithmetic as k_ce_bwd (grad = coef * 2^(z log2 e - bias), the target entry gt).
//
// Items are (row, chunk) pairs of a segment table, row-major over its k chunks (k = 1 for a
// [T, V] matrix).  One CTA per SM.  A CTA takes the items blockIdx.x + i gridDim.x, i < kPre,
// and then claims items one at a time from its launch slot's counter (ce_slots.cuh), so the
// CTAs end within about an item of each other instead of each owning a fixed share whose
// weighted items vary.  Three roles:
//   producer warp   lane 0 publishes each weighted item's row, chunk, coefficients (coef, bias,
//                   target gradient, smoothing shift) and target column, and streams the item
//                   into a ring of seven 32 KB stages with bulk asynchronous copies
//                   (cp.async.bulk); after the last item, an end marker
//   consumer warps  per stage, a thread's 4 x 16-byte vectors to gradient entries stored with
//                   16-byte streaming stores (stage::bwd_stage); the stage goes back to the
//                   producer right away
//   zero warp       writes +0.0 over the gradient of the items of weight 0 (ignored or invalid
//                   labels) among blockIdx.x, blockIdx.x + gridDim.x, ..., whose logits are not
//                   read
// Every wait is bounded (2 s).  A wait that gives up sets the CTA's abort flag; every role then
// stops at its next wait, and the producer lets its copies in flight land (bounded).
// ce_backward has no status word, so the gradient is then undefined without a report.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "ce_segments.h"
#include "ce_slots.cuh"
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
constexpr int kPre = 4;                // fixed items per CTA before the claimed ones
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
    int64_t last_claim;                // the producer's last claim, stored once its reply is in
};
constexpr int kSmemBytes = kStages * kChunk + (int)sizeof(Ctl);

struct Args {
    const int64_t* labels;
    const float4* row_stats;           // (L', 1 - p_t, target coefficient, weight); weight 0: no gradient
    const float* grad_output;
    int go_per_row;
    float eps_over_v;                  // label smoothing eps / V (0: none)
    uint64_t wait_ns;
    int slot;                          // this launch's slot (ce_slots.cuh)
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

    slots::LaunchSlot& slot = slots::g_launch_slots[a.slot];

    if (warp == kProducerWarp) {
        // ---------------- producer ----------------
        // The fixed items' statistics and labels are loaded by the warp at once, so lane 0
        // issues them back to back and the ring fills without waiting on anything.  Then the
        // claim of the item after next and the statistics and label of the next item are in
        // flight while this item's copies wait for free stages.
        uint32_t q = 0, e = 0, q_copies = 0;   // ring positions used; of them, by copies (lane 0)
        bool stop = false;
        auto issue = [&](int64_t it, float4 st, int64_t t) {   // lane 0: a weighted item
            const int64_t row = it / tab.k;
            const int c = (int)(it - row * tab.k);
            const int64_t off = tab.off[c], w = tab.width[c];
            const float cg = a.grad_output[a.go_per_row ? row : 0] * st.w;
            // the item's coefficients, published with its first stage
            ctl.info[e % kInfoSlots] = RowInfo{row, (t >= off && t < off + w) ? (int)(t - off) : -1, c, cg * st.y,
                                               (st.x == -kInf) ? 0.f : st.x * kLog2e, cg * st.z, cg * a.eps_over_v};
            const char* src = static_cast<const char*>(tab.in[c]) + row * tab.ld_in[c] * es;
            const int64_t bytes = w * es;
            const int nchunk = stages_of(c);
            for (int j = 0; j < nchunk; ++j) {
                const int st_i = (int)(q % kStages);
                if (!tc::mbar_wait(&ctl.empty[st_i], ((q / kStages) & 1) ^ 1, abort_flag, nullptr, 0, a.wait_ns)) {
                    stop = true;
                    return;
                }
                const uint32_t nb = (uint32_t)std::min<int64_t>(kChunk, bytes - (int64_t)j * kChunk);
                if (!dbg::ok(row < tab.T && c < tab.k && (int64_t)j * kChunk + nb <= bytes && w <= tab.ld_in[c],
                             dbg::kCols)) {
                    *abort_flag = 1;   // no copy: the other roles stop at their next wait
                    stop = true;
                    return;
                }
                tc::mbar_arrive_expect_tx(&ctl.full[st_i], nb);
                tc::bulk_load(smem + st_i * kChunk, src + (int64_t)j * kChunk, nb, &ctl.full[st_i]);
                q_copies = ++q;
            }
            ++e;
            stop = stop || *abort_flag;
        };
        unsigned int c1 = 0, c2 = 0;
        if (lane == 0) {
            c1 = atomicAdd(&slot.rows, 1u);
            c2 = atomicAdd(&slot.rows, 1u);
        }
        const int64_t my = blockIdx.x + (int64_t)lane * stride;
        const bool mine = lane < kPre && my < items;
        const float4 st_my = mine ? a.row_stats[my / tab.k] : make_float4(0.f, 0.f, 0.f, 0.f);
        const int64_t t_my = mine ? a.labels[my / tab.k] : 0;
        const uint32_t pre = __ballot_sync(0xFFFFFFFFu, mine && st_my.w != 0.f);
#pragma unroll
        for (int k = 0; k < kPre; ++k) {
            const float4 st = make_float4(__shfl_sync(0xFFFFFFFFu, st_my.x, k), __shfl_sync(0xFFFFFFFFu, st_my.y, k),
                                          __shfl_sync(0xFFFFFFFFu, st_my.z, k), __shfl_sync(0xFFFFFFFFu, st_my.w, k));
            const int64_t t = __shfl_sync(0xFFFFFFFFu, t_my, k);
            if (lane == 0 && ((pre >> k) & 1u) && !stop) issue(blockIdx.x + (int64_t)k * stride, st, t);
        }
        if (lane == 0) {
            const int64_t base = (int64_t)kPre * stride;
            const float4 none = make_float4(0.f, 0.f, 0.f, 0.f);
            int64_t i0 = base + c1, i1 = base + c2;
            float4 s0 = i0 < items ? a.row_stats[i0 / tab.k] : none;
            int64_t t0 = i0 < items ? a.labels[i0 / tab.k] : 0;
            while (i0 < items && !stop) {
                const int64_t i2 = base + atomicAdd(&slot.rows, 1u);
                const float4 s1 = i1 < items ? a.row_stats[i1 / tab.k] : none;
                const int64_t t1 = i1 < items ? a.labels[i1 / tab.k] : 0;
                if (s0.w != 0.f) issue(i0, s0, t0);
                i0 = i1;
                s0 = s1;
                t0 = t1;
                i1 = i2;
            }
            // Wait for the last claim's reply: every claim on the slot's counter has landed before
            // this CTA counts itself finished, so the last CTA's reset of it comes after them all.
            *reinterpret_cast<volatile int64_t*>(&ctl.last_claim) = i1;
            if (!stop) {   // the end marker: the next item's first stage completes without data
                const int st_i = (int)(q % kStages);
                if (tc::mbar_wait(&ctl.empty[st_i], ((q / kStages) & 1) ^ 1, abort_flag, nullptr, 0, a.wait_ns)) {
                    ctl.info[e % kInfoSlots] = RowInfo{-1, -1, 0, 0.f, 0.f, 0.f, 0.f};
                    tc::mbar_arrive(&ctl.full[st_i]);
                    ++q;
                }
            }
            // After an abort, copies still in flight land before the CTA may exit.  Only the last
            // kStages positions can hold one, and only those the marker did not refill.
            if (*abort_flag) {
                int never = 0;
                const uint32_t lo = q > (uint32_t)kStages ? q - kStages : 0;
                for (uint32_t p = q_copies > (uint32_t)kStages ? q_copies - kStages : 0; p < q_copies; ++p)
                    if (p >= lo)
                        tc::mbar_wait(&ctl.full[p % kStages], (p / kStages) & 1, &never, nullptr, 0, a.wait_ns);
            }
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
        uint32_t q = 0;   // ring chunk of the current item's first stage
        for (int e = 0;; ++e) {   // until the end marker
            // the item is known once its first stage (or the end marker) has landed
            const bool ok0 = tc::mbar_wait(&ctl.full[q % kStages], (q / kStages) & 1, abort_flag, nullptr, 0,
                                           a.wait_ns);
            if (!__all_sync(0xFFFFFFFFu, ok0)) break;
            const RowInfo ri = ctl.info[e % kInfoSlots];
            if (ri.row < 0) break;
            const bool in_range = ri.row < tab.T && ri.c >= 0 && ri.c < tab.k;
            const int c = in_range ? ri.c : 0;
            O* grow = in_range ? static_cast<O*>(tab.out[c]) + ri.row * tab.ld_out[c] : nullptr;
            const int64_t bytes = tab.width[c] * es;
            const int nchunk = stages_of(c);
            for (int j = 0; j < nchunk; ++j) {
                const uint32_t p = q + j;
                const int st = (int)(p % kStages);
                const bool ok = j == 0 || tc::mbar_wait(&ctl.full[st], (p / kStages) & 1, abort_flag, nullptr, 0,
                                                        a.wait_ns);
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

    // ---------------- the launch's end: the launch slot goes back to zero ----------------
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&slot.done, 1) == (int)gridDim.x - 1) {
            __threadfence();
            atomicExch(&slot.rows, 0u);
            atomicExch(&slot.done, 0);
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
                    tc::kWaitNs, slots::next_slot()};
    cudaError_t e;
    if (dt == VCE_BF16 && gdt == VCE_BF16) e = launch<uint16_t, uint16_t>(args, tab, s);
    else if (dt == VCE_BF16) e = launch<uint16_t, float>(args, tab, s);
    else if (gdt == VCE_BF16) e = launch<float, uint16_t>(args, tab, s);
    else e = launch<float, float>(args, tab, s);
    if (e == cudaSuccess) *launched = true;
    return e;
}

}  // namespace vce
