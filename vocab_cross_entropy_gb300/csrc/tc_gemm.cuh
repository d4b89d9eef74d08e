// A persistent, warp-specialised bf16 GEMM on the sm_100-family tensor cores:
//     acc[m, n] = sum_k A[m, k] * B[n, k]      (fp32 accumulators)
// Each operand is K-major (global rows run along K) or MN-major (global rows run along M,
// resp. N), chosen at compile time.
// with a caller-supplied epilogue that consumes each 128 x 256 accumulator tile from
// tensor memory.  Hand-written PTX for the TMA loads (cp.async.bulk.tensor), the
// mbarrier pipeline and the tcgen05 MMA / TMEM instructions.
//
//   warp 0 (one lane)  TMA producer: A tile 128 x 64 and B tile 256 x 64 per stage (K-major:
//                      one box of 64 K x rows; MN-major: boxes of 64 MN x 64 K)
//   warp 1 (one lane)  MMA issuer:   4 x tcgen05.mma (M=128, N=256, K=16) per stage
//   warp 2             TMEM allocation / release (512 columns = two accumulators)
//   warps 4..7         epilogue: tcgen05.ld 32 lanes x 32 columns at a time, one
//                      accumulator row per thread
// The accumulator is double buffered so the epilogue of tile i overlaps the MMAs of
// tile i+1.  Shared-memory tiles use the 128-byte swizzle that TMA writes and the MMA
// descriptors read.  Every wait is bounded: a wait that exceeds kWaitNs sets an error
// code, every role stops, in-flight copies are drained (bounded) and TMEM is released.
// Two options: a launch as 2-CTA clusters whose CTAs share each B tile through TMA multicast
// (kPair), and K-block skipping from a per-tile bit table (GemmArgs::skip, gradient
// filtering), which visits only the K blocks whose bits are set.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "vce_async.cuh"

namespace vce {
namespace tc {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_BYTES = BN * BK * 2;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;      // two fp32 accumulators of 128 lanes x 256 columns
constexpr int kThreads = 256;
constexpr int EPI_WARP_BYTES = 5120;   // per epilogue warp: staging space an epilogue may use
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 4 * EPI_WARP_BYTES + 1024 /*align*/ + 256 /*barriers*/;

// error codes written to the kernel's error word when a wait gives up
enum { kErrWaitEmpty = 101, kErrWaitFull = 102, kErrWaitAccFree = 103, kErrWaitAccFull = 104 };

// ---- tcgen05 ------------------------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate, one thread issues.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// As mma_commit, arriving on the mbarrier at the same shared-memory offset in every CTA of the
// cluster that `mask` names.
__device__ __forceinline__ void mma_commit_mc(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}

// TMA tile load into the same shared-memory offset of every CTA of the cluster that `mask`
// names, each completing bytes on its own mbarrier at `bar`'s offset.
__device__ __forceinline__ void tma_load_2d_mc(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                               uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "h"(mask)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (lane = 32 * (warp % 4) + lane id).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// Wait until this thread's tcgen05.ld have landed.  r, the destination of the last load, is
// tied to the wait, so no use of it can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Shared-memory matrix descriptor: K-major operand, rows of 64 bf16 (128 B) written by TMA
// with the 128-byte swizzle; 8-row groups 1024 B apart (stride byte offset).  The leading
// byte offset is unused for this layout.  Bits 46-47 hold the descriptor version (1).
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Shared-memory matrix descriptor: MN-major operand written by TMA as boxes of 64 K-rows x
// 128 B (64 MN elements) with the 128-byte swizzle.  Swizzle atoms are 8 K-rows x 64 MN:
// atoms along K are 1024 B apart (stride byte offset), atoms along MN one box (8 KB) apart
// (leading byte offset).
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(8192 >> 4) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, M x N; a_mn / b_mn
// select MN-major ("transposed") A / B.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn = false, bool b_mn = false) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---- the kernel ---------------------------------------------------------------------------

struct GemmArgs {
    int tiles_m, tiles_n;   // output tiles (BM x BN)
    int nk;                 // K blocks (of BK) per tile
    int nk_a0;              // the first nk_a0 blocks read A0, the rest A1 (K restarts at 0 for A1)
    int b_x0;               // B's K coordinate of block kb is b_x0 + (kb mod nk_a0) * BK
    int a_y0, b_y0;         // row offsets of the A and B tiles
    int n_fastest;          // tile order: 0 = m fastest (blocks in flight share B tiles),
                            //             1 = n fastest (blocks in flight share A tiles)
    int32_t* err;           // error word (wait timeouts)
    uint32_t tx_extra;      // bytes announced per stage beyond the copies (0; > 0 only to test the
                            // give-up path: the stage never completes and the waits must time out)
    uint64_t wait_ns;       // limit of every wait (0: kWaitNs)
    // Optional K-block skipping (gradient filtering): row tm of skip holds one bit per 128
    // K columns (two K blocks) of M tile tm, skip_ld 32-bit words per row; a clear bit means
    // A is all zero there for this tile.  Applies to both halves (A0 and A1) alike.  Null:
    // every K block runs.
    const uint32_t* skip;
    int skip_ld;
};

// Calls f(kb, ka, mine) for the K blocks of M tile tm in order -- kb the block index (A0
// blocks, then A1 blocks), ka its index within its half -- and stops when f returns false.
// Without skip bits that is every K block (mine = true).  With them (gradient filtering) it is
// the K blocks of the 128-column blocks whose bit is set for this tile or, for a CTA pair, for
// its partner (both CTAs then load the same stages; mine says whether this tile multiplies).
// The bits are scanned 32 blocks at a time with find-first-set, the next word loaded while the
// current one is walked, so skipped blocks cost nothing.  nk is nk_a0 or 2 nk_a0.
template <class F>
__device__ __forceinline__ void for_each_kblock(const GemmArgs& g, int tm, bool pair, F&& f) {
    if (!g.skip) {
        for (int kb = 0; kb < g.nk; ++kb)
            if (!f(kb, kb >= g.nk_a0 ? kb - g.nk_a0 : kb, true)) return;
        return;
    }
    const uint32_t* own = g.skip + (size_t)tm * g.skip_ld;
    const uint32_t* peer = pair ? g.skip + (size_t)(tm ^ 1) * g.skip_ld : own;
    for (int half = 0; half * g.nk_a0 < g.nk; ++half) {
        uint32_t on = own[0], pn = peer[0];
        for (int w = 0; w < g.skip_ld; ++w) {
            const uint32_t o = on;
            uint32_t m = on | pn;
            if (w + 1 < g.skip_ld) {
                on = own[w + 1];
                pn = peer[w + 1];
            }
            while (m) {
                const int bit = __ffs(m) - 1;
                m &= m - 1u;
                const bool mine = (o >> bit) & 1u;
                const int ka0 = 2 * (w * 32 + bit);   // 128 columns = two K blocks
                for (int ka = ka0; ka < ka0 + 2 && ka < g.nk_a0; ++ka)
                    if (!f(half * g.nk_a0 + ka, ka, mine)) return;
            }
        }
    }
}

// Whether M tile tm reads any kept K block.
__device__ __forceinline__ bool tile_has_blocks(const GemmArgs& g, int tm) {
    if (!g.skip) return true;
    uint32_t m = 0;
    for (int w = 0; w < g.skip_ld; ++w) m |= g.skip[(size_t)tm * g.skip_ld + w];
    return m != 0u;
}

// kPair: the grid runs as clusters of two CTAs (blockIdx 2c and 2c + 1) that take tiles 2q and
// 2q + 1, which are (2p, n) and (2p + 1, n): the two share their B tile.  tiles_m is even.
template <bool kPair>
__device__ __forceinline__ void tile_coords(const GemmArgs& g, int tile, int& tm, int& tn) {
    if (kPair && g.n_fastest) {
        const int q = tile >> 1;
        tn = q % g.tiles_n;
        tm = 2 * (q / g.tiles_n) + (tile & 1);
    } else if (g.n_fastest) {
        tn = tile % g.tiles_n;
        tm = tile / g.tiles_n;
    } else {
        tm = tile % g.tiles_m;
        tn = tile / g.tiles_m;
    }
}

// kAmn / kBmn: the operand is MN-major; its tensor map then has 64 x 64 boxes over a global
// [K, M] (resp. [K, N]) matrix, and the tile is loaded as BM/64 (resp. BN/64) boxes.
// kPair: launched as clusters of two CTAs that compute the two M-neighbours of one B tile
// (tile_coords).  Each CTA loads its own A tile and one half of the shared B tile, multicast
// into the same stage of both CTAs (a K-major B map then has boxes of BN/2 rows), so B crosses
// from L2 once per pair.  A stage is free again once both CTAs' MMAs have read it: every MMA
// commit arrives on the stage's empty barrier in both CTAs, and empty counts two arrivals.
template <class Epi, bool kAmn = false, bool kBmn = false, bool kPair = false>
__global__ void __launch_bounds__(kThreads, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap mapA0, const __grid_constant__ CUtensorMap mapA1,
              const __grid_constant__ CUtensorMap mapB, const GemmArgs g, const typename Epi::Params ep) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* smA = smem;
    uint8_t* smB = smem + STAGES * A_BYTES;
    uint8_t* epi_smem = smem + STAGES * STAGE_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(epi_smem + 4 * EPI_WARP_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;
    uint64_t* acc_free = acc_full + 2;
    uint64_t* drain = acc_free + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kPair ? 2 : 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_free[a], 4 * 32);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_map(&mapA0);
        prefetch_map(&mapA1);
        prefetch_map(&mapB);
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    if (kPair)
        cluster_sync_all();   // the peer's copies and commits reach these barriers only once they exist
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;
    const int ntiles = g.tiles_m * g.tiles_n;
    const uint64_t wns = g.wait_ns ? g.wait_ns : kWaitNs;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;   // stages whose copies were issued and not yet known complete
        for (int tile = blockIdx.x; tile < ntiles && !*abort_flag; tile += gridDim.x) {
            int tm, tn;
            tile_coords<kPair>(g, tile, tm, tn);
            for_each_kblock(g, tm, kPair, [&](int kb, int ka, bool) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, g.err, kErrWaitEmpty, wns)) return false;
                mbar_arrive_expect_tx(&full[stage], STAGE_BYTES + g.tx_extra);
                const bool second = kb >= g.nk_a0;
                const CUtensorMap* ma = second ? &mapA1 : &mapA0;
                if (kAmn) {
#pragma unroll
                    for (int h = 0; h < BM / 64; ++h)
                        tma_load_2d(smA + stage * A_BYTES + h * (64 * BK * 2), ma, &full[stage],
                                    g.a_y0 + tm * BM + h * 64, ka * BK);
                } else {
                    tma_load_2d(smA + stage * A_BYTES, ma, &full[stage], ka * BK, g.a_y0 + tm * BM);
                }
                if (kPair && kBmn) {
#pragma unroll
                    for (int i = 0; i < BN / 128; ++i) {
                        const int h = (int)rank * (BN / 128) + i;
                        tma_load_2d_mc(smB + stage * B_BYTES + h * (64 * BK * 2), &mapB, &full[stage],
                                       g.b_y0 + tn * BN + h * 64, g.b_x0 + ka * BK, 0x3);
                    }
                } else if (kPair) {
                    tma_load_2d_mc(smB + stage * B_BYTES + rank * (B_BYTES / 2), &mapB, &full[stage],
                                   g.b_x0 + ka * BK, g.b_y0 + tn * BN + (int)rank * (BN / 2), 0x3);
                } else if (kBmn) {
#pragma unroll
                    for (int h = 0; h < BN / 64; ++h)
                        tma_load_2d(smB + stage * B_BYTES + h * (64 * BK * 2), &mapB, &full[stage],
                                    g.b_y0 + tn * BN + h * 64, g.b_x0 + ka * BK);
                } else {
                    tma_load_2d(smB + stage * B_BYTES, &mapB, &full[stage], g.b_x0 + ka * BK, g.b_y0 + tn * BN);
                }
                issued = issued < STAGES ? issued + 1 : STAGES;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                return true;
            });
        }
        if (kPair && !*abort_flag) {
            // the peer's MMA commits land on these empty barriers: wait (bounded) for the last
            // STAGES of them so none arrives after this CTA has exited
            for (int i = 0; i < STAGES; ++i) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, g.err, kErrWaitEmpty, wns)) break;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (*abort_flag) {
            // drain: wait (bounded) for the copies of the last `issued` stages so no TMA write
            // lands in shared memory after the block has exited
            for (int i = 0; i < issued; ++i) {
                if (--stage < 0) { stage = STAGES - 1; phase ^= 1u; }
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(&full[stage], phase) && globaltimer() - t0 < wns) {
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, kAmn, kBmn);
        // one MMA consumes K = 16: 32 B along a K-major row, or 16 K-rows (2 KB) of an MN-major tile
        constexpr uint32_t kStepA = kAmn ? (2048 >> 4) : (32 >> 4);
        constexpr uint32_t kStepB = kBmn ? (2048 >> 4) : (32 >> 4);
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        const uint32_t a0 = smem_u32(smA), b0 = smem_u32(smB);
        for (int tile = blockIdx.x; tile < ntiles && !*abort_flag; tile += gridDim.x) {
            if (!mbar_wait(&acc_free[acc], acc_phase ^ 1u, abort_flag, g.err, kErrWaitAccFree, wns)) break;
            tc_fence_after();
            const uint32_t d = tmem_base + (uint32_t)(acc * BN);
            int tm, tn;
            tile_coords<kPair>(g, tile, tm, tn);
            bool ok = true, issued = false;
            for_each_kblock(g, tm, kPair, [&](int, int, bool mine) {
                if (!mbar_wait(&full[stage], phase, abort_flag, g.err, kErrWaitFull, wns)) {
                    ok = false;
                    return false;
                }
                tc_fence_after();
                const uint64_t ad = kAmn ? desc_mnmajor_sw128(a0 + stage * A_BYTES) : desc_kmajor_sw128(a0 + stage * A_BYTES);
                const uint64_t bd = kBmn ? desc_mnmajor_sw128(b0 + stage * B_BYTES) : desc_kmajor_sw128(b0 + stage * B_BYTES);
                if (mine) {   // else loaded for the partner only: released without MMAs
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)   // advance the start address by one K = 16 step
                        mma_bf16(d, ad + kStepA * k, bd + kStepB * k, idesc, (issued || k != 0) ? 1u : 0u);
                    issued = true;
                }
                if (kPair)
                    mma_commit_mc(&empty[stage], 0x3);
                else
                    mma_commit(&empty[stage]);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                return true;
            });
            if (!ok) break;
            mma_commit(&acc_full[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        // every MMA this thread issued has finished before TMEM can be released
        mma_commit(drain);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < wns) {
        }
    } else if (warp >= 4) {
        // ---------------- epilogue: thread = accumulator row
        const int sub = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            if (!mbar_wait(&acc_full[acc], acc_phase, abort_flag, g.err, kErrWaitAccFull, wns)) break;
            tc_fence_after();
            int tm, tn;
            tile_coords<kPair>(g, tile, tm, tn);
            const int row = tm * BM + sub * 32 + lane;
            const uint32_t t0 = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(sub * 32) << 16);
            uint8_t* stage = epi_smem + sub * EPI_WARP_BYTES;
            // Two register buffers: the next 32 columns load from TMEM while these are consumed.
            static_assert((BN / 32) % 2 == 0, "column pieces go in pairs");
            uint32_t ra[32], rb[32];
            typename Epi::Row st;
            if (!tile_has_blocks(g, tm)) {   // every K block skipped: no MMA wrote the accumulator
#pragma unroll
                for (int k = 0; k < 32; ++k) ra[k] = 0u;
                Epi::begin(ep, st, row, tn);
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) Epi::consume(ep, st, row, tn * BN + c * 32, ra, stage);
            } else {
                tmem_ld32(t0, ra);
                Epi::begin(ep, st, row, tn);   // its global loads overlap the first TMEM load
#pragma unroll 1
                for (int c = 0; c < BN / 32; c += 2) {
                    tmem_wait_ld(ra);
                    tmem_ld32(t0 + (uint32_t)((c + 1) * 32), rb);
                    Epi::consume(ep, st, row, tn * BN + c * 32, ra, stage);
                    tmem_wait_ld(rb);
                    if (c + 2 < BN / 32) tmem_ld32(t0 + (uint32_t)((c + 2) * 32), ra);
                    Epi::consume(ep, st, row, tn * BN + (c + 1) * 32, rb, stage);
                }
            }
            Epi::end(ep, st, row, tn);
            tc_fence_before();
            mbar_arrive(&acc_free[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (kPair) cluster_sync_all();   // neither CTA leaves while the other may still write to it
}

}  // namespace tc
}  // namespace vce
