// CE forward (ce_forward) for rows that suit bulk copies: each row streams through a
// shared-memory stage ring, so no thread holds global loads in flight.
//
// Method: torchtitan PR #5723 "[loss] fix softmax collapse with improved ce perf" (Numerics:
// target-excluded log-sum-exp, softplus NLL) — the same per-row statistics as k_ce_fwd.
//
// One CTA per SM.  A CTA starts on row blockIdx.x and then claims rows one at a time from its
// launch slot's counter (ce_slots.cuh): at 4096 x 32000 bf16 a fixed share of rows b, b +
// gridDim.x, ... had the CTAs end their rows between 33.8 and 42.7 us (5% of the rows are
// ignored and unevenly spread, and SMs do not all stream equally fast).  Three roles:
//   producer warp   one lane claims the rows and streams each valid one into a ring of seven
//                   32 KB stages with bulk asynchronous copies (cp.async.bulk), completion
//                   counted on per-stage mbarriers, and publishes each row's index and target
//                   column; after the last row, an end marker per consumer group
//   consumer warps  in kGroups groups (1 or 2), group g taking the CTA's rows g, g + kGroups, ...; per
//                   stage, a thread's 16-byte vectors summed four at a time into its (max,
//                   sum-exp) pair (stage::fwd_stage); the stage goes back to the producer right
//                   away; at the end of a row each warp of the group publishes its pair
//   stats warp      merges the warps' pairs, finishes the row (loss, row statistics) and frees
//                   the row's slots; it also writes the outputs of the ignored and invalid rows
//                   among blockIdx.x, blockIdx.x + gridDim.x, ...
// Row hand-offs go through kSlots mbarrier-guarded slots, by the row's index in the CTA's
// sequence mod kSlots; consumers wait for the stats warp to free a slot before writing it
// again, kSlots rows later.  The bf16 row stream of k_ce_fwd is issue-bound (a thread keeps
// four 16-byte loads in flight and sums them one vector at a time); here the copies need no
// registers and the sum takes fewer instructions per element.
//
// Groups: a row costs each warp that touches it a fixed amount of work (its stage waits and
// releases, the shuffle merge of its lanes, the hand-off), so rows of two stages run with the
// consumers in 2 groups: each thread then takes twice the columns of a row for the same
// per-row work.  Each group holds one stage at a time, so 2 stages are being summed and 5 are
// loading ahead.  (4096 x 32000 bf16: 0.0592 ms for the call, against 0.0654 without groups
// and 0.0613 on one block per row.  Rows of one stage in 4 groups lost to one warp per row:
// 8192 x 16000, 0.102 against 0.070 ms.)
//
// The CTA that finishes last writes the status word (the launch's first error code, or 0) and
// puts the launch slot back to zero, so the caller's status word needs no clearing beforehand.
// The loss reduction folded in (Args::fold, for SUM / MEAN with at most fold::kMaxRows rows;
// ce_fold.cuh): the consumer warps count every valid label of the batch at the start, while the
// first copies are in flight, so the stats warp writes each row's weight 1/N itself, and the
// last CTA also sums the rows' losses.  No separate reduction launch.
//
// Every wait is bounded (2 s); a wait that gives up records its code (105 free stage, 106
// loaded stage, 108 warp partials, 110 free slots) and sets the CTA's abort flag, after which
// every role stops at its next wait.  111: consumer groups asked for rows too long for them
// (the kernel writes the status word and returns before any wait).  112: the stats warp's wait
// for the consumer warps' label counts (folded reduction) gave up.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "ce_segments.h"
#include "ce_fold.cuh"
#include "ce_stage.cuh"
#include "vce.h"
#include "vce_async.cuh"
#include "vce_device.cuh"
#include "vce_check.cuh"
#include "vce_host.h"

namespace vce {
namespace fring {

constexpr int kChunk = 32768;          // bytes per stage (one bulk copy)
constexpr int kStages = 7;
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps, kStatsWarp = kConsumerWarps + 1;
constexpr int kThreads = kConsumers + 64;
constexpr int kVecPerThread = kChunk / 16 / kConsumers;   // per 4-vector batch of a stage
constexpr uint32_t kSuspendNs = 0;       // plain polls (a suspend hint measured no faster here)
constexpr int kSlots = 4;                // hand-off slots: consumers run up to kSlots rows ahead of the stats warp
constexpr int kInfoSlots = 16;           // > the rows the producer can run ahead of the stats warp (kStages + kSlots)
constexpr int kPre = 4;                  // fixed rows per CTA before the claimed ones
static_assert(kVecPerThread * kConsumers * 16 == kChunk, "every consumer takes the same whole vectors of a stage");
static_assert((kConsumerWarps & (kConsumerWarps - 1)) == 0 && kConsumerWarps <= 32, "warp pairs merge in one warp");
enum { kErrEmpty = 105, kErrFull = 106, kErrPartials = 108, kErrSlots = 110, kErrGroups = 111, kErrCount = 112 };

struct RowInfo {
    int64_t row;
    int tl;   // target column
    int pad;
};

struct alignas(16) Ctl {
    RowInfo info[kInfoSlots];          // by the row's index in the sequence, mod kInfoSlots
    float red_m[kSlots][kConsumerWarps], red_s[kSlots][kConsumerWarps], red_z[kSlots][kConsumerWarps];
    float zt[kSlots];
    uint64_t full[kStages];            // stage loaded
    uint64_t empty[kStages];           // stage released (one arrival per consumer warp)
    uint64_t rbar[kSlots];             // warp pairs published (one arrival per consumer warp)
    uint64_t fbar[kSlots];             // the slot read by the stats warp
    uint64_t nbar;                     // the consumer warps' label counts published (folded reduction)
    int nwarp[kConsumerWarps];         // each consumer warp's count of the batch's valid labels
    long long n_all;                   // the batch's valid labels (stats warp)
    float red_sum[kThreads / 32], red_comp[kThreads / 32];   // the last CTA's loss sum, per warp
    int err;                           // first error code of the CTA (folded reduction)
    int last;                          // this CTA finished last (folded reduction)
    int abort;
    int64_t last_claim;                // the producer's last claim, stored once its reply is in
};
constexpr int kSmemBytes = kStages * kChunk + (int)sizeof(Ctl);

struct Args {
    const void* logits;
    int64_t T, V, ld;
    const int64_t* labels;
    int64_t ignore_index;
    float* loss_rows;
    float4* row_stats;
    int32_t* status;
    float eps;                         // label smoothing (k_ce_fwd_ring<S, true> only)
    uint64_t wait_ns;
    int fold;                          // reduce the losses in this kernel (SUM / MEAN)
    int red;                           // vce_reduction
    float* loss_out;                   // the reduced loss (fold)
    int slot;                          // this launch's slot (ce_slots.cuh)
    uint32_t tx_extra;                 // 0; > 0 only in the give-up test (a stage never completes)
};

__device__ __forceinline__ bool label_valid(const Args& a, int64_t t) {
    return t != a.ignore_index && t >= 0 && t < a.V;
}

// kSmooth: label smoothing eps > 0; each row's sum of all logits is reduced alongside the pair.
// kGroups: consumer groups (1 or 2), each summing whole rows (see the file comment).
template <typename S, bool kSmooth, int kGroups>
__global__ void __launch_bounds__(kThreads, 1) k_ce_fwd_ring(const __grid_constant__ Args a) {
    constexpr int G = Elt<S>::kGroup;
    constexpr int kGW = kConsumerWarps / kGroups;   // warps of a group
    constexpr int kGT = kGW * 32;                   // threads of a group
    static_assert(kGroups == 1 || kGroups == 2, "consumer groups");
    // Hand-off slots in use.  With groups, a group waits on a stage's fill of ring position p
    // while other groups may still hold earlier positions; the parity wait is only sound once
    // the stage's previous fill (p - kStages) has landed.  A group starts row e after the stats
    // warp read row e - kUse, so every row up to e - kUse has been summed; with kUse * nchunk <=
    // kStages that covers p - kStages for every chunk of row e.  kUse >= kGroups keeps the
    // slot barriers within one phase of their waiters.
    constexpr int kUse = kGroups == 2 ? 3 : kSlots;
    static_assert(kUse <= kSlots && kUse >= kGroups, "slot count");
    extern __shared__ __align__(128) uint8_t smem[];
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem + kStages * kChunk);
    volatile int* abort_flag = &ctl.abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t stride = gridDim.x;
    const int64_t bytes = a.V * (int64_t)sizeof(S);
    const int nchunk = (int)((bytes + kChunk - 1) / kChunk);
    if (kGroups > 1 && nchunk * kUse > kStages) {   // rows too long for groups (the host never asks)
        if (threadIdx.x == 0 && blockIdx.x == 0) *a.status = kErrGroups;   // the slot stays untouched
        return;
    }
    slots::LaunchSlot& slot = slots::g_launch_slots[a.slot];

    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; ++st) {
            tc::mbar_init(&ctl.full[st], 1);
            tc::mbar_init(&ctl.empty[st], kGW);
        }
        for (int p = 0; p < kUse; ++p) {
            tc::mbar_init(&ctl.rbar[p], kGW);
            tc::mbar_init(&ctl.fbar[p], 1);
        }
        tc::mbar_init(&ctl.nbar, kConsumerWarps);
        for (int i = 0; i < kInfoSlots; ++i) ctl.info[i] = RowInfo{-1, -1, 0};
        ctl.abort = 0;
        ctl.err = 0;
        ctl.n_all = 0;
        tc::fence_mbar_init();
    }
    __syncthreads();
    // error codes: the CTA's word, merged into the launch slot at the end
    int32_t* errp = &ctl.err;

    if (warp == kProducerWarp) {
        // ---------------- producer ----------------
        // A CTA's first kPre rows are fixed (blockIdx.x + k gridDim.x, k < kPre): the warp loads
        // their labels at once and lane 0 issues the valid ones back to back, which fills the
        // ring without waiting on anything.  Every later row is claimed one at a time, as
        // kPre gridDim.x + the launch slot's count of earlier claims, so a CTA that streams
        // faster takes more rows and all end within about a row of each other.  The first two
        // claims go out before the fixed rows; after that, the claim of the row after next and
        // the label of the next row are in flight while this row's copies wait for free stages.
        // Rows whose label is not valid are skipped (the stats warp writes their outputs).
        // After the last row, kGroups end markers (row -1) complete the first stage of the next
        // kGroups rows without data.
        uint32_t q = 0, e = 0, q_copies = 0;   // ring positions used; of them, by copies (lane 0)
        bool stop = false;
        auto issue = [&](int64_t row, int64_t t) {   // lane 0: the copies of a valid row
            ctl.info[e % kInfoSlots] = RowInfo{row, (int)t, 0};   // published with the first stage
            const char* src = static_cast<const char*>(a.logits) + row * a.ld * (int64_t)sizeof(S);
            for (int j = 0; j < nchunk; ++j) {
                const int st = (int)(q % kStages);
                if (!tc::mbar_wait(&ctl.empty[st], ((q / kStages) & 1) ^ 1, abort_flag, errp, kErrEmpty, a.wait_ns,
                                   kSuspendNs)) {
                    stop = true;
                    return;
                }
                const uint32_t nb = (uint32_t)std::min<int64_t>(kChunk, bytes - (int64_t)j * kChunk);
                if (!dbg::ok(row < a.T && (int64_t)j * kChunk + nb <= bytes && a.V <= a.ld, dbg::kCols)) {
                    *abort_flag = 1;   // no copy: the other roles stop at their next wait
                    stop = true;
                    return;
                }
                tc::mbar_arrive_expect_tx(&ctl.full[st], nb + a.tx_extra);
                tc::bulk_load(smem + st * kChunk, src + (int64_t)j * kChunk, nb, &ctl.full[st]);
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
        const int64_t t_my = lane < kPre && my < a.T ? a.labels[my] : 0;
        const uint32_t pre = __ballot_sync(0xFFFFFFFFu, lane < kPre && my < a.T && label_valid(a, t_my));
#pragma unroll
        for (int k = 0; k < kPre; ++k) {
            const int64_t t = __shfl_sync(0xFFFFFFFFu, t_my, k);
            if (lane == 0 && ((pre >> k) & 1u) && !stop) issue(blockIdx.x + (int64_t)k * stride, t);
        }
        if (lane == 0) {
            const int64_t base = (int64_t)kPre * stride;
            int64_t r0 = base + c1, r1 = base + c2;
            int64_t t0 = r0 < a.T ? a.labels[r0] : 0;
            while (r0 < a.T && !stop) {
                const int64_t r2 = base + atomicAdd(&slot.rows, 1u);
                const int64_t t1 = r1 < a.T ? a.labels[r1] : 0;
                if (label_valid(a, t0)) issue(r0, t0);
                r0 = r1;
                t0 = t1;
                r1 = r2;
            }
            // Wait for the last claim's reply: every claim on the slot's counter has landed before
            // this CTA counts itself finished, so the last CTA's reset of it comes after them all.
            *reinterpret_cast<volatile int64_t*>(&ctl.last_claim) = r1;
            for (int g = 0; g < kGroups && !stop; ++g) {   // end markers, one per consumer group
                const int st = (int)(q % kStages);
                if (!tc::mbar_wait(&ctl.empty[st], ((q / kStages) & 1) ^ 1, abort_flag, errp, kErrEmpty, a.wait_ns,
                                   kSuspendNs))
                    break;
                ctl.info[e % kInfoSlots] = RowInfo{-1, -1, 0};
                tc::mbar_arrive(&ctl.full[st]);
                q += (uint32_t)nchunk;   // the marker stands for a whole row's positions
                ++e;
            }
            // After an abort, copies still in flight land before the CTA may exit.  Only the last
            // kStages positions can hold one, and only those no later marker refilled (a refill
            // waited for the consumers to release the stage, so its copy had landed).
            if (*abort_flag) {
                int never = 0;
                const uint32_t lo = q > (uint32_t)kStages ? q - kStages : 0;
                for (uint32_t p = q_copies > (uint32_t)kStages ? q_copies - kStages : 0; p < q_copies; ++p)
                    if (p >= lo)
                        tc::mbar_wait(&ctl.full[p % kStages], (p / kStages) & 1, &never, nullptr, 0, a.wait_ns);
            }
        }
        __syncwarp();
    } else if (warp == kStatsWarp) {
        // ---------------- row statistics ----------------
        // Rows whose label is ignore_index or invalid (the logits are not read): one per lane,
        // four labels loaded before any is used.
        for (int64_t base = blockIdx.x + (int64_t)lane * stride; base < a.T; base += 4 * 32 * stride) {
            int64_t tu[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t row = base + (int64_t)u * 32 * stride;
                tu[u] = row < a.T ? a.labels[row] : 0;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t row = base + (int64_t)u * 32 * stride;
                const int64_t t = tu[u];
                if (row >= a.T || label_valid(a, t)) continue;
                a.loss_rows[row] = (t == a.ignore_index) ? 0.f : __int_as_float(0x7FC00000);
                a.row_stats[row] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (t != a.ignore_index) atomicCAS(errp, 0, (int32_t)VCE_ERR_LABEL);
            }
        }
        __syncwarp();
        // folded reduction: the batch's valid labels, counted by the consumer warps (MEAN weight)
        float w_valid = 1.f;
        if (a.fold) {
            tc::mbar_wait(&ctl.nbar, 0, abort_flag, errp, kErrCount, a.wait_ns, kSuspendNs);
            if (lane == 0) {
                long long n = 0;
                for (int w = 0; w < kConsumerWarps; ++w) n += ctl.nwarp[w];
                ctl.n_all = n;
                if (a.red == VCE_RED_MEAN) w_valid = n > 0 ? (float)(1.0 / (double)n) : 0.f;
            }
        }
        for (int e = 0;; ++e) {   // until the end marker
            const int par = e % kUse;
            const bool ok = tc::mbar_wait(&ctl.rbar[par], (e / kUse) & 1, abort_flag, errp, kErrPartials, a.wait_ns,
                                          kSuspendNs);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            const RowInfo ri = ctl.info[e % kInfoSlots];
            if (ri.row < 0) break;
            float m = lane < kGW ? ctl.red_m[par][lane] : -kInf;
            float s = lane < kGW ? ctl.red_s[par][lane] : 0.f;
#pragma unroll
            for (int off = kGW / 2; off > 0; off >>= 1) {
                const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, off);
                const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, off);
                ms_merge(m, s, m2, s2);
            }
            float tot = 0.f;   // the row's sum of logits, warps added in a fixed order
            if (kSmooth && lane == 0)
                for (int w = 0; w < kGW; ++w) tot += ctl.red_z[par][w];
            if (lane == 0) {
                const float zt = ctl.zt[par];
                tc::mbar_arrive(&ctl.fbar[par]);   // the slot may be rewritten
                if (ri.row < a.T) {
                    float loss;
                    float4 st4 = kSmooth ? ce_row_finish_smoothed(m, s, zt, tot, a.V, a.eps, &loss)
                                         : ce_row_finish(m, s, zt, &loss);
                    st4.w = w_valid;   // 1, or 1/N for a folded MEAN (else k_ce_reduce writes it)
                    a.row_stats[ri.row] = st4;
                    a.loss_rows[ri.row] = loss;
                }
            }
            __syncwarp();
        }
    } else {
        // ---------------- consumers ----------------
        const int grp = warp / kGW, gw = warp % kGW;
        const int gtid = threadIdx.x - grp * kGT;   // thread index within the group
        if (a.fold) {   // the batch's valid labels, consumer thread c taking rows c, c + kConsumers, ...
            int n = fold::count_valid_strided(a.labels, a.T, a.V, a.ignore_index, threadIdx.x, kConsumers);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) n += __shfl_xor_sync(0xFFFFFFFFu, n, off);
            if (lane == 0) {
                ctl.nwarp[warp] = n;
                tc::mbar_arrive(&ctl.nbar);
            }
        }
        for (int e = grp;; e += kGroups) {   // until this group's end marker
            const int par = e % kUse;
            const uint32_t q = (uint32_t)e * (uint32_t)nchunk;   // ring chunk of the row's first chunk
            // the slot was read for row e - kUse
            if (e >= kUse) {
                const bool ok = tc::mbar_wait(&ctl.fbar[par], ((e / kUse) & 1) ^ 1, abort_flag, errp, kErrSlots,
                                              a.wait_ns, kSuspendNs);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;
            }
            // the row's first stage, or its end marker
            const bool ok0 = tc::mbar_wait(&ctl.full[q % kStages], (q / kStages) & 1, abort_flag, errp, kErrFull,
                                           a.wait_ns, kSuspendNs);
            if (!__all_sync(0xFFFFFFFFu, ok0)) break;
            const RowInfo ri = ctl.info[e % kInfoSlots];
            if (ri.row < 0) {   // no more rows: the stats warp learns it from the same slot
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&ctl.rbar[par]);
                break;
            }
            const int tl = ri.tl;
            float m = -kInf, s = 0.f, mb = 0.f, sz = 0.f;
            for (int j = 0; j < nchunk; ++j) {
                const uint32_t p = q + j;
                const int st = (int)(p % kStages);
                const bool ok = j == 0 || __all_sync(0xFFFFFFFFu, tc::mbar_wait(&ctl.full[st], (p / kStages) & 1,
                                                                                abort_flag, errp, kErrFull,
                                                                                a.wait_ns, kSuspendNs));
                if (ok) {
                    const uint4* buf = reinterpret_cast<const uint4*>(smem + st * kChunk);
                    const int nvec = (int)(std::min<int64_t>(kChunk, bytes - (int64_t)j * kChunk) / 16);
#pragma unroll
                    for (int b = 0; b < kGroups; ++b) {   // batches of kVecPerThread vectors per thread
                        const int v0 = b * kVecPerThread * kGT;
                        if (v0 >= nvec) break;
                        const int rel0 = tl - (j * (kChunk / (int)sizeof(S)) + (v0 + gtid) * G);
                        stage::fwd_stage_any<S, kGT, kVecPerThread, kSmooth>(buf + v0, nvec - v0, rel0, gtid, m, s,
                                                                             mb, &ctl.zt[par], &sz);
                    }
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&ctl.empty[st]);
            }
            ms_warp_reduce(m, s);
            if (kSmooth) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sz += __shfl_xor_sync(0xFFFFFFFFu, sz, off);
            }
            if (lane == 0) {
                ctl.red_m[par][gw] = m;
                ctl.red_s[par][gw] = s;
                if (kSmooth) ctl.red_z[par][gw] = sz;
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ctl.rbar[par]);
        }
    }

    // ---------------- the launch's end: status word, folded reduction ----------------
    fold::finish_slot<kThreads>(slot, a.status, &ctl.err, a.fold != 0, a.loss_rows, a.T, ctl.n_all, a.red,
                                a.loss_out, ctl.red_sum, ctl.red_comp, &ctl.last);
}

template <typename S, int kGroups>
cudaError_t launch_groups(const Args& args, int sms, cudaStream_t s) {
    auto kern = args.eps > 0.f ? k_ce_fwd_ring<S, true, kGroups> : k_ce_fwd_ring<S, false, kGroups>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(sms, args.T);
    kern<<<grid, kThreads, kSmemBytes, s>>>(args);
    return cudaGetLastError();
}

template <typename S>
cudaError_t launch(const Args& args, int sms, cudaStream_t s) {
    const int64_t nchunk = (args.V * (int64_t)sizeof(S) + kChunk - 1) / kChunk;
    if (nchunk == 2) return launch_groups<S, 2>(args, sms, s);
    return launch_groups<S, 1>(args, sms, s);
}

}  // namespace fring

VCE_DEBUG_READER(debug_word_ce_fwd_ring)

cudaError_t launch_fwd_ring(vce_dtype dt, const void* logits, int64_t T, int64_t V, int64_t ld, const int64_t* labels,
                            int64_t ignore_index, float eps, int red, float* loss_rows, float* loss_out,
                            float* row_stats, int32_t* status, cudaStream_t s, bool* launched, bool* reduced,
                            uint64_t wait_ns, uint32_t tx_extra) {
    using namespace fring;
    *launched = false;
    *reduced = false;
    // 16-byte rows: every row starts on a 16-byte boundary and is whole 16-byte vectors.
    if (T < 1 || V % 8 || ld % 8 || !aligned(logits, 16) || V > (int64_t)1 << 30) return cudaSuccess;
    const bool in_kernel = red != VCE_RED_NONE && T <= fold::kMaxRows;
    Args args{logits,    T,   V,          ld,          labels,          ignore_index, loss_rows,
              reinterpret_cast<float4*>(row_stats), status, eps, wait_ns, in_kernel ? 1 : 0, red, loss_out,
              slots::next_slot(), tx_extra};
    const int sms = device_sm_count();
    const cudaError_t e = dt == VCE_BF16 ? launch<uint16_t>(args, sms, s) : launch<float>(args, sms, s);
    if (e == cudaSuccess) {
        *launched = true;
        *reduced = in_kernel;
    }
    return e;
}

}  // namespace vce

using namespace vce;

extern "C" int vce_test_ce_fwd_stall(const void* logits, int64_t T, int64_t V, const int64_t* labels, float* loss_rows,
                                     float* row_stats, float* loss_out, uint64_t wait_ns, int32_t* status,
                                     vce_stream_t s) {
    if (!logits || !labels || !loss_rows || !row_stats || !loss_out || !status) return VCE_ERR_NULL;
    if (T < 1 || T > fold::kMaxRows || V < 1) return VCE_ERR_SHAPE;
    if (wait_ns < 1000000ull || wait_ns > tc::kWaitNs) return VCE_ERR_ARG;
    if (V * 2 <= 32768) return VCE_ERR_ARG;   // rows of at most 32 KB take the warp kernel
    if (!aligned(row_stats, 16) || !aligned(labels, 8) || !aligned(loss_rows, 4) || !aligned(loss_out, 4))
        return VCE_ERR_ALIGN;
    int rc = require_sm100();
    if (rc) return rc;
    bool launched = false, reduced = false;
    // 16 bytes announced beyond each copy: no stage ever completes
    if (launch_fwd_ring(VCE_BF16, logits, T, V, V, labels, -100, 0.f, VCE_RED_SUM, loss_rows, loss_out, row_stats,
                        status, s, &launched, &reduced, wait_ns, 16) != cudaSuccess)
        return VCE_ERR_CUDA;
    return launched ? VCE_OK : VCE_ERR_ARG;
}
