// One-pass cross-entropy forward and backward with every row held on chip between its two
// passes, so HBM moves exactly one read of the logits and one write of the gradient.
//
// Method: torchtitan PR #5723 "[loss] fix softmax collapse with improved ce perf" — the same
// numerics as ce_forward / ce_backward (Numerics: target-excluded log-sum-exp, softplus NLL,
// the p_t = 1/4 branch; Memory/perf: "forward also prepares the backward").  The vocabulary
// split across a thread-block cluster is the single-GPU form of the Megatron-core
// vocab-parallel cross-entropy (Cross Entropy Loss / VocabParallelCrossEntropy: each part
// reduces its own columns, the parts exchange (max, sum-exp, target logit), every part
// writes its own gradient columns).
//
// A row of a 128256-entry vocabulary in bf16 (250.5 KB) does not fit one SM's shared memory,
// so a cluster of C CTAs on C SMs takes it, each CTA a column slice of at most 128 KB of its
// stage ring (224 KB: seven 32 KB stages, or fourteen 16 KB stages for bf16 rows in a cluster).
// A cluster walks the rows cid, cid + ncl, ... (cid: the cluster's index, ncl: the clusters);
// a single CTA, for rows of at most 128 KB, takes four such rows and then claims rows one at a
// time from its launch slot (ce_slots.cuh), so the CTAs end within about a row of each other.
// Each CTA (one per SM) skips the rows whose label is not valid and has three roles:
//   producer warp   one lane streams each row's slice into the shared-memory stage ring
//                   with bulk asynchronous copies (cp.async.bulk; completion counted
//                   on a per-stage mbarrier), running ahead into later rows as stages free up;
//                   after the last row, an end marker that the other roles stop at
//   consumer warps  forward of a row over its held stages (per-thread (max, sum-exp) pairs,
//                   the target masked out by its column), each warp's pair published to shared
//                   memory; then, while the row's statistics are being finished, the forward
//                   of the next row over the stages already loaded beside it; then the
//                   row's gradient from its held stages, releasing each stage to the producer;
//                   then the rest of the next row's forward
//   stats warp      per row: merges the consumer warps' pairs, exchanges the slice pair with
//                   the cluster's other CTAs through distributed shared memory (each CTA stores
//                   its pair into every peer and arrives on the peer's mbarrier), merges the C
//                   pairs in rank order (identically in every CTA), finishes the row, and
//                   publishes the gradient coefficients
// so the exchange and the row finish run while the consumers stream the next row.  Row
// hand-offs go through mbarriers only, double-buffered by the parity of the row's index in
// the CTA's sequence: a slot of one parity is rewritten two rows later, after every reader of
// it has arrived on a barrier the writer waits for.
//
// The CTA that finishes last writes the status word (the launch's first error code, or 0) and
// puts the launch slot back to zero, so the caller's status word needs no clearing first.  The
// loss reduction folded in (Args::fold, for SUM / MEAN over at most fold::kMaxRows rows;
// ce_fold.cuh): the consumer warps count the batch's valid labels before their first row, so the
// stats warp has 1/N for the row weights and gradient coefficients without a counting kernel
// before this one, and the last CTA also sums the rows' losses; no reduction kernel after it
// either.
//
// Every wait is bounded (2 s).  A wait that gives up records its code (105 free stage, 106
// loaded stage, 107 cluster exchange, 108 warp partials, 109 row coefficients) and sets the
// CTA's abort flag; its roles then stop at their next wait (a peer waiting on this CTA's
// exchange gives up in turn, bounded), and the producer waits, again bounded, for its copies
// in flight before the CTA reaches the closing cluster barrier.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "ce_segments.h"
#include "vce.h"
#include "ce_fold.cuh"
#include "ce_stage.cuh"
#include "vce_async.cuh"
#include "vce_device.cuh"
#include "vce_check.cuh"
#include "vce_host.h"

namespace vce {
namespace ring {

constexpr int kRingBytes = 229376;     // the stage ring: 224 KB of shared memory
constexpr int kSliceBytes = 131072;    // a CTA's slice of a row occupies at most this much of it
constexpr int kMaxStages = 14;
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps, kStatsWarp = kConsumerWarps + 1;
constexpr int kThreads = kConsumers + 64;
constexpr int kMaxCluster = 8;
constexpr int kMaxDevices = 64;
// Stage geometry: a single CTA streams seven 32 KB stages; a cluster's CTAs on bf16 rows stream
// fourteen 16 KB stages, so a held slice (up to eight of them) frees its stages in smaller steps
// and the next row's loads start sooner.  Measured against 32 KB stages (ms per call): pages'
// shape (2-CTA clusters) 1.329 against 1.342, 16384 x 70000 0.978 against 1.048, 2048 x 400000
// (8-CTA clusters) 0.832 against 0.870.  Single CTAs ran 9-11% slower on 16 KB stages (4096 and
// 16384 rows of 32000) and fp32 rows 2% slower (4096 x 128256, 4-CTA clusters): a thread's
// share of a 16 KB stage is only 8 fp32 values for the same per-stage work.
template <typename S, int C>
struct Geom {
    static constexpr int kChunk = (C > 1 && sizeof(S) == 2) ? 16384 : 32768;   // bytes per stage (one bulk copy)
    static constexpr int kStages = kRingBytes / kChunk;
    static constexpr int kVecPerThread = kChunk / 16 / kConsumers;   // 16-B vectors per consumer per stage
    static_assert(kStages <= kMaxStages && kStages * kChunk == kRingBytes, "stage ring");
    static_assert(kSliceBytes % kChunk == 0 && kSliceBytes / kChunk < kStages, "a held slice leaves stages free");
};
// Longest sleep of one poll of an incomplete mbarrier phase: the waiting warps (the producer on a
// free stage, the stats warp on the partials, consumers on data) leave the issue slots to the
// working ones and wake when the phase completes.
constexpr uint32_t kSuspendRole = 10000, kSuspendConsumer = 10000;
static_assert((kConsumerWarps & (kConsumerWarps - 1)) == 0 && kConsumerWarps <= 32, "warp partials merge in one warp");
enum { kErrEmpty = 105, kErrFull = 106, kErrExchange = 107, kErrPartials = 108, kErrCoefs = 109 };

// A valid row of the CTA's sequence: its index and its target's column local to the slice.
struct RowInfo {
    int64_t row;
    int tl;
    int pad;
};
constexpr int kInfoSlots = 16;         // > the rows the producer can run ahead (kStages at one chunk a row; a
                                       // cluster's slices are more than four 16 KB stages)
constexpr int kPre = 4;                // a single CTA's fixed rows before the claimed ones

struct alignas(16) Ctl {
    RowInfo info[kInfoSlots];          // by the row's index in the sequence, mod kInfoSlots
    float4 slot[2][kMaxCluster];       // (m, s, z_t, owner) of each CTA of the cluster
    float slot_z[2][kMaxCluster];      // label smoothing: each CTA's sum of its slice's logits
    float4 coefs[2];                   // (coef, bias, target gradient, non-target shift) of the row
    float red_m[2][kConsumerWarps], red_s[2][kConsumerWarps], red_z[2][kConsumerWarps];
    float zt[2];
    uint64_t full[kMaxStages];         // stage loaded (producer's expect-tx + the copy's bytes)
    uint64_t empty[kMaxStages];        // stage released (one arrival per consumer warp)
    uint64_t xbar[2];                  // cluster pairs stored (one arrival per CTA)
    uint64_t rbar[2];                  // warp pairs published (one arrival per consumer warp)
    uint64_t cbar[2];                  // coefficients published (the stats warp)
    uint64_t nbar;                     // the consumer warps' label counts published (folded reduction)
    int nwarp[kConsumerWarps];         // each consumer warp's count of the batch's valid labels
    long long n_all;                   // the batch's valid labels (stats warp)
    float red_sum[kThreads / 32], red_comp[kThreads / 32];   // the last CTA's loss sum, per warp
    int err;                           // first error code of the CTA
    int last;                          // this CTA finished last
    int abort;
    int64_t last_claim;                // a single CTA's last claim, stored once its reply is in
};
constexpr int kSmemBytes = kRingBytes + (int)sizeof(Ctl);

struct Args {
    const void* logits;
    int64_t T, V, ld;
    const int64_t* labels;
    int64_t ignore_index;
    int red;
    const float* grad_output;
    const float* inv_n;
    float* loss_rows;
    float4* row_stats;
    void* grad;
    int64_t ld_g;
    int32_t* status;
    int64_t slice;                     // columns per CTA (a multiple of 8)
    uint64_t wait_ns;                  // bound of every wait
    uint32_t tx_extra;                 // 0; > 0 only in the give-up test (a stage never completes)
    float eps;                         // label smoothing (k_ce_fused_ring<S, O, C, true> only)
    int fold;                          // reduce the losses in this kernel (SUM / MEAN; inv_n unused)
    float* loss_out;                   // the reduced loss (fold)
    int slot;                          // this launch's slot (ce_slots.cuh)
};

// ---- cluster and bulk-copy primitives (inline PTX) -----------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(tc::smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_peer1(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_peer(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ void arrive_peer(uint32_t bar_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_addr) : "memory");
}
__device__ __forceinline__ bool try_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t suspend_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(tc::smem_u32(bar)), "r"(parity), "r"(suspend_ns)
        : "memory");
    return ok != 0;
}
// Bounded wait on a phase of an mbarrier written by peers of the cluster.
__device__ __forceinline__ bool wait_exchange(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int32_t* err, uint64_t wait_ns) {
    if (*abort_flag) return false;
    const uint64_t t0 = tc::globaltimer();
    while (!try_wait_cluster(bar, parity, kSuspendRole)) {
        if (*abort_flag) return false;
        if (tc::globaltimer() - t0 > wait_ns) {
            *abort_flag = 1;
            if (err) atomicCAS(err, 0, (int32_t)kErrExchange);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ bool label_valid(const Args& a, int64_t t) {
    return t != a.ignore_index && t >= 0 && t < a.V;
}
// The first row with a valid label among row, row + stride, ...; T if none.
__device__ __forceinline__ int64_t next_valid(const Args& a, int64_t row, int64_t stride) {
    for (; row < a.T; row += stride)
        if (label_valid(a, a.labels[row])) return row;
    return a.T;
}

// ---- the kernel -----------------------------------------------------------------------------

// kSmooth: label smoothing eps > 0.  Each row's sum of all logits is reduced beside the pair
// and exchanged with it; the non-target gradient entries lose c eps / V.
template <typename S, typename O, int C, bool kSmooth>
__global__ void __launch_bounds__(kThreads, 1) k_ce_fused_ring(const __grid_constant__ Args a) {
    constexpr int G = Elt<S>::kGroup;
    using Ring = Geom<S, C>;
    constexpr int kChunk = Ring::kChunk, kStages = Ring::kStages, kVecPerThread = Ring::kVecPerThread;
    constexpr int kFullVec = kChunk / 16;
    extern __shared__ __align__(128) uint8_t smem[];
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem + kStages * kChunk);
    volatile int* abort_flag = &ctl.abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = C > 1 ? cluster_rank() : 0;
    const int64_t cid = blockIdx.x / C, ncl = gridDim.x / C;
    const int64_t c0 = std::min<int64_t>(a.V, (int64_t)rank * a.slice);
    const int w = (int)(std::min<int64_t>(a.V, c0 + a.slice) - c0);   // this CTA's columns [c0, c0 + w)
    const int bytes = w * (int)sizeof(S);
    const int nchunk = (bytes + kChunk - 1) / kChunk;
    // chunks of the next row that fit beside a held row (all of them for short slices)
    const int pre = std::min(nchunk, kStages - nchunk);

    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; ++st) {
            tc::mbar_init(&ctl.full[st], 1);
            tc::mbar_init(&ctl.empty[st], kConsumerWarps);
        }
        for (int p = 0; p < 2; ++p) {
            tc::mbar_init(&ctl.xbar[p], C);
            tc::mbar_init(&ctl.rbar[p], kConsumerWarps);
            tc::mbar_init(&ctl.cbar[p], 1);
        }
        tc::mbar_init(&ctl.nbar, kConsumerWarps);
        for (int i = 0; i < kInfoSlots; ++i) ctl.info[i] = RowInfo{-1, -1, 0};
        ctl.abort = 0;
        ctl.err = 0;
        ctl.n_all = 0;
        tc::fence_mbar_init();
    }
    if (C > 1) cluster_sync();   // peers arrive on these barriers from now on
    else __syncthreads();
    // error codes: the CTA's word, merged into the launch slot at the end
    int32_t* errp = &ctl.err;
    slots::LaunchSlot& slot = slots::g_launch_slots[a.slot];

    if (warp == kProducerWarp) {
        // ---------------- producer ----------------
        // A single CTA takes its first kPre rows fixed (blockIdx.x + k gridDim.x, k < kPre) and
        // then claims rows one at a time from the launch slot's counter (kPre gridDim.x + the
        // count of earlier claims), so a CTA that streams faster takes more rows.  The claims of
        // the next three rows and the label of the next row are in flight while this row's
        // copies wait for free stages.  A cluster walks the fixed rows cid, cid + ncl, ...: a
        // claim would have to reach every CTA of the cluster, and handing each one on through
        // the peers' shared memory cost more (pages' shape, 2-CTA clusters: 1.37-1.46 ms against
        // 1.33-1.34 ms) than the balance gained.  Rows whose label is not valid are skipped (the
        // consumer warps zero-fill their gradients).  After the last row, an end marker (row -1)
        // completes the next row's first stage without data.
        if (lane == 0) {
            uint32_t q = 0, e = 0, q_copies = 0;   // ring positions used; of them, by copies
            bool stop = false;
            auto issue = [&](int64_t row, int64_t t) {   // the copies of a valid row
                // the row's index and target column, for the other roles (published by the first
                // chunk's barrier arrival)
                ctl.info[e % kInfoSlots] = RowInfo{row, (int)(t - c0), 0};
                const char* src = static_cast<const char*>(a.logits) + (row * a.ld + c0) * (int64_t)sizeof(S);
                for (int j = 0; j < nchunk; ++j) {
                    const int st = (int)(q % kStages);
                    if (!tc::mbar_wait(&ctl.empty[st], ((q / kStages) & 1) ^ 1, abort_flag, errp, kErrEmpty,
                                       a.wait_ns, kSuspendRole)) {
                        stop = true;
                        return;
                    }
                    const uint32_t nb = (uint32_t)min(kChunk, bytes - j * kChunk);
                    if (!dbg::ok(row < a.T && c0 + w <= a.V && a.V <= a.ld && j * kChunk + (int)nb <= bytes,
                                 dbg::kCols)) {
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
            const int64_t base = (int64_t)kPre * ncl;
            unsigned int c1 = 0, c2 = 0, c3 = 0;
            if (C == 1) {   // the first three claims go out before the fixed rows
                c1 = atomicAdd(&slot.rows, 1u);
                c2 = atomicAdd(&slot.rows, 1u);
                c3 = atomicAdd(&slot.rows, 1u);
            }
            int64_t tp[kPre];
#pragma unroll
            for (int k = 0; k < kPre; ++k) {
                const int64_t row = cid + (int64_t)k * ncl;
                tp[k] = row < a.T ? a.labels[row] : 0;
            }
#pragma unroll
            for (int k = 0; k < kPre; ++k) {
                const int64_t row = cid + (int64_t)k * ncl;
                if (row < a.T && label_valid(a, tp[k]) && !stop) issue(row, tp[k]);
            }
            // Rows r0, r1, r2: the next three of the sequence (the claims' replies are taken even
            // after an abort: see below).
            auto fixed = [&](uint32_t k) { return base + (int64_t)k * ncl + cid; };
            int64_t r0 = C == 1 ? base + c1 : fixed(0);
            int64_t r1 = C == 1 ? base + c2 : fixed(1);
            int64_t r2 = C == 1 ? base + c3 : fixed(2);
            uint32_t k_next = 3;
            int64_t t0 = r0 < a.T ? a.labels[r0] : 0;
            while (r0 < a.T && !stop) {
                const int64_t r3 = C == 1 ? base + atomicAdd(&slot.rows, 1u) : fixed(k_next);
                const int64_t t1 = r1 < a.T ? a.labels[r1] : 0;
                if (label_valid(a, t0)) issue(r0, t0);
                ++k_next;
                r0 = r1;
                t0 = t1;
                r1 = r2;
                r2 = r3;
            }
            // Every claim's reply is in before this CTA counts itself finished (r0, r1 and r2 hold
            // the last ones), so the last CTA's reset of the counter comes after them all.
            *reinterpret_cast<volatile int64_t*>(&ctl.last_claim) = r0 + r1 + r2;
            if (!stop) {   // the end marker: the next row's first stage completes without data
                const int st = (int)(q % kStages);
                if (tc::mbar_wait(&ctl.empty[st], ((q / kStages) & 1) ^ 1, abort_flag, errp, kErrEmpty, a.wait_ns,
                                  kSuspendRole)) {
                    ctl.info[e % kInfoSlots] = RowInfo{-1, -1, 0};
                    tc::mbar_arrive(&ctl.full[st]);
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
    } else if (warp == kStatsWarp) {
        // ---------------- row statistics ----------------
        float w_valid = 1.f;   // the row weight: 1/N for MEAN
        if (a.fold) {   // N from the consumer warps' counts
            tc::mbar_wait(&ctl.nbar, 0, abort_flag, errp, kErrPartials, a.wait_ns, kSuspendRole);
            long long n = 0;
            for (int k = 0; k < kConsumerWarps; ++k) n += ctl.nwarp[k];
            if (lane == 0) ctl.n_all = n;
            if (a.red == VCE_RED_MEAN) w_valid = n > 0 ? (float)(1.0 / (double)n) : 0.f;   // as k_ce_reduce
        } else if (a.red == VCE_RED_MEAN) {
            w_valid = *a.inv_n;
        }
        for (int e = 0;; ++e) {   // until the end marker
            const int par = e & 1;
            const uint32_t ph = (e >> 1) & 1;
            const bool ok = tc::mbar_wait(&ctl.rbar[par], ph, abort_flag, errp, kErrPartials, a.wait_ns, kSuspendRole);
            // (after an abort the consumers may have ended early: their slot is then not a row's)
            if (!__all_sync(0xFFFFFFFFu, ok) || __any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
            const RowInfo ri = ctl.info[e % kInfoSlots];
            if (ri.row < 0) break;
            float m = lane < kConsumerWarps ? ctl.red_m[par][lane] : -kInf;
            float s = lane < kConsumerWarps ? ctl.red_s[par][lane] : 0.f;
#pragma unroll
            for (int off = kConsumerWarps / 2; off > 0; off >>= 1) {   // lanes 0..kConsumerWarps-1 into lane 0
                const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, off);
                const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, off);
                ms_merge(m, s, m2, s2);
            }
            if (lane == 0) {
                const bool own = (uint32_t)ri.tl < (uint32_t)w;
                float sz = 0.f;   // the slice's sum of logits, warps added in a fixed order
                if (kSmooth)
                    for (int k = 0; k < kConsumerWarps; ++k) sz += ctl.red_z[par][k];
                float M = m, Ssum = s, zt = own ? ctl.zt[par] : 0.f, tot = sz;
                if (C > 1) {
                    const float4 mine = make_float4(m, s, zt, own ? 1.f : 0.f);
                    for (uint32_t r = 0; r < (uint32_t)C; ++r) {
                        st_peer(peer_addr(&ctl.slot[par][rank], r), mine);
                        if (kSmooth) st_peer1(peer_addr(&ctl.slot_z[par][rank], r), sz);
                    }
                    for (uint32_t r = 0; r < (uint32_t)C; ++r) arrive_peer(peer_addr(&ctl.xbar[par], r));
                    wait_exchange(&ctl.xbar[par], ph, abort_flag, errp, a.wait_ns);
                    M = -kInf;
                    Ssum = 0.f;
                    tot = 0.f;
                    for (int r = 0; r < C; ++r) {   // the same order in every CTA
                        const float4 o = ctl.slot[par][r];
                        ms_merge(M, Ssum, o.x, o.y);
                        if (o.w != 0.f) zt = o.z;
                        if (kSmooth) tot += ctl.slot_z[par][r];
                    }
                }
                const bool in_range = ri.row < a.T;   // false only after an abort
                float loss;
                float4 st4 = kSmooth ? ce_row_finish_smoothed(M, Ssum, zt, tot, a.V, a.eps, &loss)
                                     : ce_row_finish(M, Ssum, zt, &loss);
                st4.w = w_valid;
                const float c = in_range ? a.grad_output[a.red == VCE_RED_NONE ? ri.row : 0] * w_valid : 0.f;
                ctl.coefs[par] = make_float4(c * st4.y, (st4.x == -kInf) ? 0.f : st4.x * kLog2e, c * st4.z,
                                             kSmooth ? c * (a.eps / (float)a.V) : 0.f);
                tc::mbar_arrive(&ctl.cbar[par]);
                if (rank == 0 && in_range) {
                    a.row_stats[ri.row] = st4;
                    a.loss_rows[ri.row] = loss;
                }
            }
            __syncwarp();
        }
    } else {
        // ---------------- consumers ----------------
        const int tid = threadIdx.x;
        if (a.fold) {   // the batch's valid labels, consumer thread c taking rows c, c + kConsumers, ...
            int n = fold::count_valid_strided(a.labels, a.T, a.V, a.ignore_index, tid, kConsumers);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) n += __shfl_xor_sync(0xFFFFFFFFu, n, off);
            if (lane == 0) {
                ctl.nwarp[warp] = n;
                tc::mbar_arrive(&ctl.nbar);
            }
        }

        // Rows whose label is ignore_index or invalid: gradient +0.0 by selection, logits unread.
        // Each warp reads the labels of 32 of the cluster's rows at once and zero-fills the
        // invalid ones' slices.
        for (int64_t base = cid + (int64_t)warp * 32 * ncl; base < a.T; base += (int64_t)kConsumerWarps * 32 * ncl) {
            const int64_t my = base + (int64_t)lane * ncl;
            const int64_t t_my = my < a.T ? a.labels[my] : 0;
            uint32_t bad = __ballot_sync(0xFFFFFFFFu, my < a.T && !label_valid(a, t_my));
            while (bad) {
                const int b = __ffs(bad) - 1;
                bad &= bad - 1;
                const int64_t row = base + (int64_t)b * ncl;
                const int64_t t = __shfl_sync(0xFFFFFFFFu, t_my, b);
                if (rank == 0 && lane == 0) {
                    a.loss_rows[row] = (t == a.ignore_index) ? 0.f : __int_as_float(0x7FC00000);
                    a.row_stats[row] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (t != a.ignore_index) atomicCAS(errp, 0, (int32_t)VCE_ERR_LABEL);
                }
                if (!dbg::ok(c0 + w <= a.ld_g, dbg::kCols)) continue;
                O* grow = static_cast<O*>(a.grad) + row * a.ld_g + c0;
                const float zero[G] = {};
                for (int vi = lane; vi < w / G; vi += 32) GroupStore<O, G>::run(grow + vi * G, zero);
            }
        }

        // Forward over chunks [j0, j1) of valid row e, whose first chunk is ring chunk q0.  The
        // row's index and target column are read once its first chunk has landed; false if that
        // was the end marker (or the wait gave up).
        auto forward = [&](uint32_t q0, int j0, int j1, int e, RowInfo& ri, float& m, float& s, float& mb,
                           float& sz) {
            for (int j = j0; j < j1; ++j) {
                const uint32_t p = q0 + j;
                const int st = (int)(p % kStages);
                bool ok = tc::mbar_wait(&ctl.full[st], (p / kStages) & 1, abort_flag, errp, kErrFull, a.wait_ns,
                                        kSuspendConsumer);
                if (j == 0) {
                    if (!__all_sync(0xFFFFFFFFu, ok)) return false;
                    ri = ctl.info[e % kInfoSlots];
                    if (ri.row < 0) return false;
                }
                if (!ok) continue;
                const uint4* buf = reinterpret_cast<const uint4*>(smem + st * kChunk);
                const int nvec = min(kChunk, bytes - j * kChunk) / 16;
                const int rel0 = ri.tl - (j * (kChunk / (int)sizeof(S)) + tid * G);
                stage::fwd_stage_any<S, kConsumers, kVecPerThread, kSmooth>(buf, nvec, rel0, tid, m, s, mb,
                                                                            &ctl.zt[e & 1], &sz);
            }
            return true;
        };
        // This warp's pair of the row, for the stats warp.
        auto publish = [&](int par, float m, float s, float sz) {
            ms_warp_reduce(m, s);
            if (kSmooth) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sz += __shfl_xor_sync(0xFFFFFFFFu, sz, off);
            }
            if (lane == 0) {
                ctl.red_m[par][warp] = m;
                ctl.red_s[par][warp] = s;
                if (kSmooth) ctl.red_z[par][warp] = sz;
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ctl.rbar[par]);
        };

        // The stats warp learns of the end from the end marker's slot: the warps arrive on its
        // partials barrier without partials.
        auto publish_end = [&](int par) {
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ctl.rbar[par]);
        };
        uint32_t q = 0;   // ring chunk of the current row's first chunk
        RowInfo ri{-1, -1, 0};
        bool have;
        {
            float m = -kInf, s = 0.f, mb = 0.f, sz = 0.f;
            have = forward(q, 0, nchunk, 0, ri, m, s, mb, sz);
            if (have) publish(0, m, s, sz);
            else publish_end(0);
        }
        for (int e = 0; have; ++e) {
            const int par = e & 1;
            RowInfo ri2{-1, -1, 0};
            float m2 = -kInf, s2 = 0.f, mb2 = 0.f, sz2 = 0.f;
            const bool more = forward(q + nchunk, 0, pre, e + 1, ri2, m2, s2, mb2, sz2);

            // the row's gradient, each stage released once this warp is done with it
            tc::mbar_wait(&ctl.cbar[par], (e >> 1) & 1, abort_flag, errp, kErrCoefs, a.wait_ns, kSuspendConsumer);
            const float4 cf = ctl.coefs[par];
            const bool in_range = ri.row >= 0 && ri.row < a.T;   // false only after an abort
            O* grow = static_cast<O*>(a.grad) + (in_range ? ri.row : 0) * a.ld_g + c0;
            for (int j = 0; j < nchunk; ++j) {
                const int st = (int)((q + j) % kStages);
                if (in_range && !*abort_flag) {
                    const uint4* buf = reinterpret_cast<const uint4*>(smem + st * kChunk);
                    const int nvec = min(kChunk, bytes - j * kChunk) / 16;
                    const int col0 = j * (kChunk / (int)sizeof(S));
                    const int rel0 = ri.tl - (col0 + tid * G);
                    if (!dbg::ok(col0 + nvec * G <= w && c0 + w <= a.ld_g, dbg::kCols))
                        ;   // the stage's columns would leave the CTA's slice: no store
                    else if (nvec == kFullVec)
                        stage::bwd_stage<S, O, kConsumers, kVecPerThread, true, kSmooth, true>(
                            buf, nvec, grow + col0, rel0, tid, cf.x, cf.y, cf.z, cf.w);
                    else
                        stage::bwd_stage<S, O, kConsumers, kVecPerThread, false, kSmooth, true>(
                            buf, nvec, grow + col0, rel0, tid, cf.x, cf.y, cf.z, cf.w);
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&ctl.empty[st]);
            }
            q += nchunk;

            if (more) {
                forward(q, pre, nchunk, e + 1, ri2, m2, s2, mb2, sz2);
                publish(par ^ 1, m2, s2, sz2);
            } else {
                publish_end(par ^ 1);
            }
            ri = ri2;
            have = more;
        }
    }
    if (C > 1) cluster_sync();   // no CTA leaves while a peer may still write into its shared memory
    fold::finish_slot<kThreads>(slot, a.status, &ctl.err, a.fold != 0, a.loss_rows, a.T, ctl.n_all, a.red,
                                a.loss_out, ctl.red_sum, ctl.red_comp, &ctl.last);
}

template <typename S, typename O, int C, bool kSmooth>
cudaError_t launch(const Args& args, int sms, cudaStream_t s, bool* launched) {
    auto kern = k_ce_fused_ring<S, O, C, kSmooth>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = sms;
    if (C > 1) {   // clusters that fit at once, queried once per device
        static std::atomic<int> fit[kMaxDevices];
        int dev = 0;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDevices) return cudaSuccess;
        clusters = fit[dev].load() - 1;
        if (clusters < 0) {
            cfg.gridDim = dim3(C * (sms / C));
            e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
            if (e != cudaSuccess) return e;
            fit[dev].store(clusters + 1);
        }
        if (clusters < 1) return cudaSuccess;   // no room for one cluster: not launched
    }
    clusters = (int)std::min<int64_t>(clusters, args.T);
    cfg.gridDim = dim3(C * clusters);
    e = cudaLaunchKernelEx(&cfg, kern, args);
    if (e == cudaSuccess) *launched = true;
    return e;
}

template <typename S, typename O, bool kSmooth>
cudaError_t launch_c(int C, const Args& args, int sms, cudaStream_t s, bool* launched) {
    switch (C) {
        case 1: return launch<S, O, 1, kSmooth>(args, sms, s, launched);
        case 2: return launch<S, O, 2, kSmooth>(args, sms, s, launched);
        case 4: return launch<S, O, 4, kSmooth>(args, sms, s, launched);
        default: return launch<S, O, 8, kSmooth>(args, sms, s, launched);
    }
}

template <typename S, typename O>
cudaError_t launch_cs(int C, const Args& args, int sms, cudaStream_t s, bool* launched) {
    return args.eps > 0.f ? launch_c<S, O, true>(C, args, sms, s, launched)
                          : launch_c<S, O, false>(C, args, sms, s, launched);
}

}  // namespace ring

VCE_DEBUG_READER(debug_word_ce_ring)

namespace {
// The cluster size and slice (columns per CTA, a multiple of 8) for rows of V entries of es
// bytes: the smallest cluster whose slices fit kSliceBytes; C > kMaxCluster if none.
void cluster_shape(int64_t V, int64_t es, int* C_out, int64_t* slice_out) {
    using namespace ring;
    int C = 1;
    int64_t slice = V;
    for (; C <= kMaxCluster; C *= 2) {
        slice = ((V + C - 1) / C + 7) / 8 * 8;
        if (slice * es <= (int64_t)kSliceBytes) break;
    }
    *C_out = C;
    *slice_out = slice;
}
}  // namespace

bool fused_ring_layout_ok(vce_dtype dt, int64_t T, int64_t V, int64_t ld, int64_t ld_g, const void* logits,
                          const void* grad) {
    // 16-byte rows and slices: every row and slice starts on a 16-byte boundary, and each slice
    // is whole 16-byte vectors of input and output.
    if (T < 1 || V % 8 || ld % 8 || ld_g % 8 || !aligned(logits, 16) || !aligned(grad, 16)) return false;
    int C;
    int64_t slice;
    cluster_shape(V, dt == VCE_BF16 ? 2 : 4, &C, &slice);
    return C <= ring::kMaxCluster;
}

bool fused_ring_reduces(int red, int64_t T) { return red != VCE_RED_NONE && T >= 1 && T <= fold::kMaxRows; }

cudaError_t launch_fused_ring(vce_dtype dt, vce_dtype gdt, const void* logits, int64_t T, int64_t V, int64_t ld,
                              const int64_t* labels, int64_t ignore_index, int red, const float* grad_output,
                              const float* inv_n, float* loss_rows, float* row_stats, void* grad, int64_t ld_g,
                              int32_t* status, cudaStream_t s, bool* launched, float eps, uint64_t wait_ns,
                              uint32_t tx_extra, bool* reduced, float* loss_out) {
    using namespace ring;
    *launched = false;
    if (reduced) *reduced = false;
    if (!fused_ring_layout_ok(dt, T, V, ld, ld_g, logits, grad)) return cudaSuccess;
    int C;
    int64_t slice;
    cluster_shape(V, dt == VCE_BF16 ? 2 : 4, &C, &slice);
    const bool in_kernel = reduced && loss_out && fused_ring_reduces(red, T);
    Args args{logits, T,   V,    ld,   labels, ignore_index, red,   grad_output, inv_n,
              loss_rows, reinterpret_cast<float4*>(row_stats), grad, ld_g, status, slice, wait_ns, tx_extra, eps,
              in_kernel ? 1 : 0, loss_out, slots::next_slot()};
    const int sms = device_sm_count();
    cudaError_t e;
    if (dt == VCE_BF16 && gdt == VCE_BF16) e = launch_cs<uint16_t, uint16_t>(C, args, sms, s, launched);
    else if (dt == VCE_BF16) e = launch_cs<uint16_t, float>(C, args, sms, s, launched);
    else if (gdt == VCE_BF16) e = launch_cs<float, uint16_t>(C, args, sms, s, launched);
    else e = launch_cs<float, float>(C, args, sms, s, launched);
    if (e == cudaSuccess && *launched && reduced) *reduced = in_kernel;
    return e;
}

}  // namespace vce

using namespace vce;

extern "C" int vce_test_ce_fused_stall(const void* logits, int64_t T, int64_t V, const int64_t* labels,
                                       const float* grad_output, float* loss_rows, float* row_stats,
                                       void* grad_logits, uint64_t wait_ns, int32_t* status, vce_stream_t s) {
    if (!logits || !labels || !grad_output || !loss_rows || !row_stats || !grad_logits || !status) return VCE_ERR_NULL;
    if (T < 1 || V < 1) return VCE_ERR_SHAPE;
    if (wait_ns < 1000000ull || wait_ns > tc::kWaitNs) return VCE_ERR_ARG;
    if (!aligned(row_stats, 16) || !aligned(labels, 8)) return VCE_ERR_ALIGN;
    int rc = require_sm100();
    if (rc) return rc;
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return VCE_ERR_CUDA;
    bool launched = false;
    // 16 bytes announced beyond each copy: no stage ever completes
    if (launch_fused_ring(VCE_BF16, VCE_BF16, logits, T, V, V, labels, -100, VCE_RED_SUM, grad_output, nullptr,
                          loss_rows, row_stats, grad_logits, V, status, s, &launched, 0.f, wait_ns, 16) != cudaSuccess)
        return VCE_ERR_CUDA;
    return launched ? VCE_OK : VCE_ERR_ARG;
}
