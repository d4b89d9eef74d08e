// A persistent, warp-specialised bf16 GEMM on the sm_100-family tensor cores:
//     acc[m, n] = sum_k A[m, k] * B[n, k]      (fp32 accumulators in tensor memory)
// Each operand is K-major (global rows run along K) or MN-major (global rows run along M,
// resp. N), chosen at compile time, with a caller-supplied epilogue that consumes each
// accumulator tile from tensor memory.  Hand-written PTX for the TMA loads
// (cp.async.bulk.tensor), the mbarrier pipeline and the tcgen05 MMA / TMEM instructions.
//
//   warp 0 (one lane)  TMA producer: this CTA's A tile (128 x 64) and B rows (x 64) per stage
//   warp 1 (one lane)  MMA issuer:   4 x tcgen05.mma (K = 16) per stage, 8 with dual A operands
//                                    or two K blocks per stage
//   warp 2             TMEM allocation / release (all 512 columns)
//   warps 4..7         epilogue: tcgen05.ld 32 lanes x 32 columns at a time, one
//                      accumulator row per thread
// The accumulator is double buffered so the epilogue of tile i overlaps the MMAs of tile
// i+1.  Shared-memory tiles use the 128-byte swizzle that TMA writes and the MMA descriptors
// read.  Every wait is bounded: a wait that exceeds its limit sets an error code, every role
// stops, in-flight copies are drained (bounded) and TMEM is released.
//
// Two launch forms (template kCta2):
//   single CTAs      tile 128 x 256; the CTA loads A (128 rows) and all 256 rows of B.
//   CTA pairs        a 2-CTA cluster computes a 256 x 256 tile with tcgen05.mma.cta_group::2:
//                    each CTA loads its own 128 rows of A and its own 128 rows of B into its
//                    own shared memory (plain TMA loads, no multicast), the even CTA issues the
//                    MMAs, which read both CTAs' operands and write each CTA's 128 accumulator
//                    rows into that CTA's tensor memory.  Both CTAs' copies complete on the even
//                    CTA's stage barrier; the MMA commits arrive on both CTAs' barriers.  Per
//                    CTA a stage holds A plus half of B, so B crosses from L2 once per pair,
//                    shared memory reads per MMA fall by a third and seven stages fit.
// Options: K-block skipping from a per-tile bit table (GemmArgs::skip, gradient filtering,
// single CTAs only); a K offset (GemmArgs::ka0) so that one product can be split along K into
// launches whose partial sums the caller merges; dual A operands (template kDualA):
// acc = (A0 + A1) B^T with A0's and A1's tiles of one K block held in the same stage beside a
// single B tile, so B is loaded once for both (the linear-CE's G_hi and G_lo); and two K blocks
// per stage (template kK2: A's and B's tiles of blocks k and k + 1 in one stage, eight MMAs per
// stage, the same accumulation order; one A operand, no skip bits, an even number of blocks).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "vce_async.cuh"
#include "vce_check.cuh"

namespace vce {
namespace tc {

constexpr int BM = 128, BN = 256, BK = 64;   // A rows per CTA, tile columns, K per stage
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int kThreads = 256;
constexpr int TMEM_COLS = 2 * BN;             // two fp32 accumulators of 128 lanes x 256 columns
constexpr int kMaxSmem = 232448;              // opt-in dynamic shared memory per block (227 KB)

// kK2: a stage holds two consecutive K blocks of A and of B (eight MMAs per stage).
// kScratch: shared memory the epilogue asks for beside the stage ring (Epi::kScratch bytes,
// a quarter per epilogue warp), placed after the barriers.
template <bool kCta2, bool kDualA = false, bool kK2 = false, int kScratch = 0>
struct Cfg {
    static_assert(!(kDualA && kK2), "dual A operands take one K block per stage");
    static constexpr int kKPer = kK2 ? 2 : 1;              // K blocks per stage
    static constexpr int kBRows = kCta2 ? BN / 2 : BN;   // rows of the B tile this CTA loads
    static constexpr int kBBlock = kBRows * BK * 2;       // B bytes of one K block
    static constexpr int kBBytes = kKPer * kBBlock;
    static constexpr int kABytes = (kDualA ? 2 : kKPer) * A_BYTES;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kReserve = 1024 /*alignment*/ + 256 /*barriers*/ + kScratch;
    // single: 4 stages (3 with dual A, 2 with two K blocks); pair: 7 stages (4 with dual A, 3
    // with two K blocks)
    static constexpr int kStages = (kMaxSmem - kReserve) / kStageBytes;
    static constexpr int kSmem = kStages * kStageBytes + kReserve;
};

// error codes written to the kernel's error word when a wait gives up (100: the two CTAs of a
// pair were given different tensor-memory columns)
enum { kErrTmemPair = 100, kErrWaitEmpty = 101, kErrWaitFull = 102, kErrWaitAccFree = 103, kErrWaitAccFull = 104 };

// ---- cluster helpers ----------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// The shared::cluster address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
// Arrive on an mbarrier given by its shared::cluster address (this CTA's or a peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait (as mbar_wait); kCluster: with cluster-scope acquire, for barriers that the
// other CTA of a pair arrives on.
template <bool kCluster>
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                         int code, uint64_t wait_ns) {
    if (!kCluster) return mbar_wait(bar, parity, abort_flag, err, code, wait_ns);
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > wait_ns) {
            *abort_flag = 1;
            if (err) atomicCAS(err, 0, code);
            return false;
        }
    }
}

// TMA tile load into this CTA's shared memory, completing its bytes on the mbarrier at the
// shared::cluster address `bar` -- this CTA's or, for a CTA pair, the even CTA's.
template <bool kCta2>
__device__ __forceinline__ void tma_load(void* dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
    if constexpr (kCta2) {
        asm volatile(
            "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
            "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
            "l"(map), "r"(x), "r"(y), "r"(bar)
            : "memory");
    } else {
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
            "[%4];" ::"r"(smem_u32(dst)),
            "l"(map), "r"(x), "r"(y), "r"(bar)
            : "memory");
    }
}

// ---- tcgen05 ------------------------------------------------------------------------------

template <bool kCta2>
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    if constexpr (kCta2)
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                     "r"(ncols)
                     : "memory");
}
template <bool kCta2>
__device__ __forceinline__ void tmem_relinquish() {
    if constexpr (kCta2)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
template <bool kCta2>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    if constexpr (kCta2)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate, one thread issues (for a
// pair: a thread of the even CTA, and A, B, D span both CTAs).
template <bool kCta2>
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    if constexpr (kCta2)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Arrive on the mbarrier at shared::cluster address `bar` once every tcgen05.mma issued so far
// by this thread has completed.
template <bool kCta2>
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    if constexpr (kCta2)
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
    else
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
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
    int tiles_m, tiles_n;   // output tiles of 128 rows x 256 columns (tiles_m even for CTA pairs)
    int nk;                 // K blocks (of BK) per tile
    int nk_a0;              // the first nk_a0 blocks read A0, the rest A1 (K restarts at 0 for A1);
                            // with dual A operands each of the nk_a0 blocks reads both
    int b_x0;               // B's K coordinate of block kb is b_x0 + (ka0 + kb mod nk_a0) * BK
    int a_y0, b_y0;         // row offsets of the A and B tiles
    int n_fastest;          // tile order: 0 = m fastest (blocks in flight share B tiles),
                            //             1 = n fastest (blocks in flight share A tiles)
    int32_t* err;           // error word (wait timeouts)
    uint32_t tx_extra;      // bytes announced per stage beyond the copies (0; > 0 only to test the
                            // give-up path: the stage never completes and the waits must time out)
    uint64_t wait_ns;       // limit of every wait (0: kWaitNs)
    // Optional K-block skipping (gradient filtering, single CTAs): row tm of skip holds one bit
    // per 128 K columns (two K blocks) of M tile tm, skip_ld 32-bit words per row; a clear bit
    // means A is all zero there for this tile.  Applies to both halves (A0 and A1) alike.
    // Null: every K block runs.
    const uint32_t* skip;
    int skip_ld;
    // K offset: block ka of a half reads K block ka0 + ka of A (and of B, after b_x0), so a
    // product split along K runs as launches over [ka0, ka0 + nk_a0).
    int ka0;
};

// Calls f(kb, ka) for the K blocks of M tile tm in order -- kb the block index (A0 blocks,
// then A1 blocks), ka its index within its half -- and stops when f returns false.  Without
// skip bits that is every K block.  With them (gradient filtering) it is the K blocks of the
// 128-column blocks whose bit is set for this tile.  The bits are scanned 32 blocks at a time
// with find-first-set, the next word loaded while the current one is walked, so skipped
// blocks cost nothing.  nk is nk_a0 or 2 nk_a0.
template <class F>
__device__ __forceinline__ void for_each_kblock(const GemmArgs& g, int tm, F&& f) {
    if (!g.skip) {
        for (int kb = 0; kb < g.nk; ++kb)
            if (!f(kb, kb >= g.nk_a0 ? kb - g.nk_a0 : kb)) return;
        return;
    }
    const uint32_t* own = g.skip + (size_t)tm * g.skip_ld;
    for (int half = 0; half * g.nk_a0 < g.nk; ++half) {
        uint32_t on = own[0];
        for (int w = 0; w < g.skip_ld; ++w) {
            uint32_t m = on;
            if (w + 1 < g.skip_ld) on = own[w + 1];
            while (m) {
                const int bit = __ffs(m) - 1;
                m &= m - 1u;
                const int ka0 = 2 * (w * 32 + bit);   // 128 columns = two K blocks
                for (int ka = ka0; ka < ka0 + 2 && ka < g.nk_a0; ++ka)
                    if (!f(half * g.nk_a0 + ka, ka)) return;
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

// Tile `tile` of the launch: M tile tm (128 rows) and N tile tn.  A CTA pair walks tiles of
// 256 rows; CTA `rank` of the pair takes the M tile 2 mm + rank.
template <bool kCta2>
__device__ __forceinline__ void tile_coords(const GemmArgs& g, int tile, uint32_t rank, int& tm, int& tn) {
    const int tiles_mm = kCta2 ? g.tiles_m / 2 : g.tiles_m;
    int mm;
    if (g.n_fastest) {
        tn = tile % g.tiles_n;
        mm = tile / g.tiles_n;
    } else {
        mm = tile % tiles_mm;
        tn = tile / tiles_mm;
    }
    tm = kCta2 ? 2 * mm + (int)rank : mm;
}

// The epilogue interface (Epi):
//   struct Params; struct Row;
//   begin(p, row_state, row, tn)                        before a tile's columns
//   consume(p, row_state, row, col0, acc[32])           32 accumulator columns, in order
//   end(p, row_state, row, tn)                          after them (all lanes of the warp)
// kAmn / kBmn: the operand is MN-major; its tensor map then has 64 x 64 boxes over a global
// [K, M] (resp. [K, N]) matrix, and the tile is loaded as 2 (resp. kBRows / 64) boxes.  A
// K-major B map has boxes of kBRows rows.
template <class Epi, bool kAmn, bool kBmn, bool kCta2, bool kDualA = false, bool kK2 = false>
__global__ void __launch_bounds__(kThreads, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap mapA0, const __grid_constant__ CUtensorMap mapA1,
              const __grid_constant__ CUtensorMap mapB, const GemmArgs g, const typename Epi::Params ep) {
    using C = Cfg<kCta2, kDualA, kK2, Epi::kScratch>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* smA = smem;   // per stage: A0 (and A1) tiles
    uint8_t* smB = smem + S * C::kABytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * C::kStageBytes);
    uint64_t* empty = full + S;
    uint64_t* acc_full = empty + S;
    uint64_t* acc_free = acc_full + 2;
    uint64_t* drain = acc_free + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = kCta2 ? cluster_ctarank() : 0u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_free[a], kCta2 ? 8 : 4);   // one arrival per epilogue warp (of both CTAs)
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_map(&mapA0);
        prefetch_map(&mapA1);
        prefetch_map(&mapB);
    }
    if (warp == 2) {
        tmem_alloc<kCta2>(tmem_slot, TMEM_COLS);
        tmem_relinquish<kCta2>();
    }
    tc_fence_before();
    if (kCta2)
        cluster_sync_all();   // the peer's copies, commits and arrivals reach these barriers only once they exist
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (kCta2 && threadIdx.x == 0 && rank == 1 && ld_cluster_u32(cluster_addr(tmem_slot, 0)) != tmem_base) {
        *abort_flag = 1;   // the pair's MMAs address both CTAs' tensor memory at the even CTA's columns
        if (g.err) atomicCAS(g.err, 0, (int)kErrTmemPair);
    }
    if (kCta2) __syncthreads();   // the check above before any role of this CTA starts
    const int ntiles = (kCta2 ? g.tiles_m / 2 : g.tiles_m) * g.tiles_n;
    const int tile0 = kCta2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int tstep = kCta2 ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const uint64_t wns = g.wait_ns ? g.wait_ns : kWaitNs;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;   // stages whose copies were issued and not yet known complete
        for (int tile = tile0; tile < ntiles && !*abort_flag; tile += tstep) {
            int tm, tn;
            tile_coords<kCta2>(g, tile, rank, tm, tn);
            auto each = [&](auto&& f) {   // the stages of this tile: K blocks, (A0, A1) block pairs
                if (kDualA) {             // or pairs of consecutive K blocks
                    for (int ka = 0; ka < g.nk_a0; ++ka)
                        if (!f(0, ka)) return;
                } else if (kK2) {
                    for (int ka = 0; ka < g.nk; ka += 2)
                        if (!f(ka, ka)) return;
                } else {
                    for_each_kblock(g, tm, f);
                }
            };
            each([&](int kb, int ka) {
                if (!wait_bar<kCta2>(&empty[stage], phase ^ 1u, abort_flag, g.err, kErrWaitEmpty, wns)) return false;
                // the barrier that counts this stage's bytes: the even CTA's for a pair
                const uint32_t fb = kCta2 ? cluster_addr(&full[stage], 0) : smem_u32(&full[stage]);
                if (!kCta2 || rank == 0)
                    mbar_arrive_expect_tx(&full[stage], (kCta2 ? 2 : 1) * C::kStageBytes + g.tx_extra);
                uint8_t* sa = smA + stage * C::kABytes;
                uint8_t* sb = smB + stage * C::kBBytes;
                auto load_a = [&](const CUtensorMap* ma, uint8_t* dst, int k) {
                    if (kAmn) {
#pragma unroll
                        for (int h = 0; h < BM / 64; ++h)
                            tma_load<kCta2>(dst + h * (64 * BK * 2), ma, fb, g.a_y0 + tm * BM + h * 64, k);
                    } else {
                        tma_load<kCta2>(dst, ma, fb, k, g.a_y0 + tm * BM);
                    }
                };
                const int n0 = g.b_y0 + tn * BN + (int)rank * C::kBRows;
                auto load_b = [&](uint8_t* dst, int k) {
                    if (kBmn) {
#pragma unroll
                        for (int h = 0; h < C::kBRows / 64; ++h)
                            tma_load<kCta2>(dst + h * (64 * BK * 2), &mapB, fb, n0 + h * 64, g.b_x0 + k);
                    } else {
                        tma_load<kCta2>(dst, &mapB, fb, g.b_x0 + k, n0);
                    }
                };
                if (kDualA) {
                    const int k = (g.ka0 + ka) * BK;
                    load_a(&mapA0, sa, k);
                    load_a(&mapA1, sa + A_BYTES, k);
                    load_b(sb, k);
                } else {
#pragma unroll
                    for (int h = 0; h < C::kKPer; ++h) {   // K blocks kb (and kb + 1) of the stage
                        const int k = (g.ka0 + ka + h) * BK;
                        load_a(kb + h >= g.nk_a0 ? &mapA1 : &mapA0, sa + h * A_BYTES, k);
                        load_b(sb + h * C::kBBlock, k);
                    }
                }
                issued = issued < S ? issued + 1 : S;
                if (++stage == S) { stage = 0; phase ^= 1u; }
                return true;
            });
        }
        if (*abort_flag) {
            if (!kCta2 || rank == 0) {
                // drain: wait (bounded) for the copies of the last `issued` stages (a pair's
                // stage completes once both CTAs' copies landed) so no TMA write lands in
                // shared memory after the block has exited
                for (int i = 0; i < issued; ++i) {
                    if (--stage < 0) { stage = S - 1; phase ^= 1u; }
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(&full[stage], phase) && globaltimer() - t0 < wns) {
                    }
                }
            } else {
                // the odd CTA's copies complete on the even CTA's barriers: give them time to land
                const uint64_t t0 = globaltimer();
                while (globaltimer() - t0 < 1000000ull) {
                }
            }
        }
    } else if (warp == 1 && lane == 0 && (!kCta2 || rank == 0)) {
        // ---------------- MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(kCta2 ? 2 * BM : BM, BN, kAmn, kBmn);
        // one MMA consumes K = 16: 32 B along a K-major row, or 16 K-rows (2 KB) of an MN-major tile
        constexpr uint32_t kStepA = kAmn ? (2048 >> 4) : (32 >> 4);
        constexpr uint32_t kStepB = kBmn ? (2048 >> 4) : (32 >> 4);
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        const uint32_t a0 = smem_u32(smA), b0 = smem_u32(smB);
        // commits arrive on this CTA's barrier and, for a pair, on the odd CTA's too
        auto commit = [&](uint64_t* bar) {
            mma_commit<kCta2>(smem_u32(bar));
            if (kCta2) mma_commit<kCta2>(cluster_addr(bar, 1));
        };
        for (int tile = tile0; tile < ntiles && !*abort_flag; tile += tstep) {
            if (!wait_bar<kCta2>(&acc_free[acc], acc_phase ^ 1u, abort_flag, g.err, kErrWaitAccFree, wns)) break;
            tc_fence_after();
            const uint32_t d = tmem_base + (uint32_t)(acc * BN);
            int tm, tn;
            tile_coords<kCta2>(g, tile, rank, tm, tn);
            bool ok = true, issued = false;
            auto stage_mmas = [&](int, int) {
                if (!wait_bar<false>(&full[stage], phase, abort_flag, g.err, kErrWaitFull, wns)) {
                    ok = false;
                    return false;
                }
                tc_fence_after();
                const uint32_t sa = a0 + stage * C::kABytes;
#pragma unroll
                for (int h = 0; h < (kDualA ? 2 : C::kKPer); ++h) {   // A0, then A1 against the same B
                    const uint32_t at = sa + h * A_BYTES;             // tile; or K blocks kb, kb + 1
                    const uint32_t bt = b0 + stage * C::kBBytes + (kK2 ? h * C::kBBlock : 0);
                    const uint64_t ad = kAmn ? desc_mnmajor_sw128(at) : desc_kmajor_sw128(at);
                    const uint64_t bd = kBmn ? desc_mnmajor_sw128(bt) : desc_kmajor_sw128(bt);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)   // advance the start address by one K = 16 step
                        mma_bf16<kCta2>(d, ad + kStepA * k, bd + kStepB * k, idesc,
                                        (issued || h != 0 || k != 0) ? 1u : 0u);
                }
                issued = true;
                commit(&empty[stage]);
                if (++stage == S) { stage = 0; phase ^= 1u; }
                return true;
            };
            if (kDualA) {
                for (int ka = 0; ka < g.nk_a0; ++ka)
                    if (!stage_mmas(0, ka)) break;
            } else if (kK2) {
                for (int ka = 0; ka < g.nk; ka += 2)
                    if (!stage_mmas(ka, ka)) break;
            } else {
                for_each_kblock(g, tm, stage_mmas);
            }
            if (!ok) break;
            commit(&acc_full[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        // every MMA this thread issued has finished before TMEM can be released
        mma_commit<kCta2>(smem_u32(drain));
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < wns) {
        }
    } else if (warp >= 4) {
        // ---------------- epilogue: thread = accumulator row
        const int sub = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
        auto release = [&]() {   // this warp is done with accumulator `acc`
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (kCta2)
                    mbar_arrive_cluster(cluster_addr(&acc_free[acc], 0));
                else
                    mbar_arrive(&acc_free[acc]);
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        };
        for (int tile = tile0; tile < ntiles; tile += tstep) {
            // the warp decides together: tcgen05.ld is a warp-wide instruction
            const bool ok = wait_bar<kCta2>(&acc_full[acc], acc_phase, abort_flag, g.err, kErrWaitAccFull, wns);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            int tm, tn;
            tile_coords<kCta2>(g, tile, rank, tm, tn);
            const int row = tm * BM + sub * 32 + lane;
            const uint32_t t0 = tmem_base + (uint32_t)(acc * BN) + lane_off;
            typename Epi::Row st;
            if constexpr (Epi::kScratch > 0)   // this warp's quarter of the scratch after the barriers
                st.scratch = smem + S * C::kStageBytes + 256 + sub * (Epi::kScratch / 4);
            // Two register buffers: the next 32 columns load from TMEM while these are consumed.
            static_assert((BN / 32) % 2 == 0, "column pieces go in pairs");
            uint32_t ra[32], rb[32];
            if (!dbg::ok(tm >= 0 && tm < g.tiles_m && tn >= 0 && tn < g.tiles_n, dbg::kTile)) {
                // warp-uniform: a tile outside the output is not written (its accumulator is released)
            } else if (!tile_has_blocks(g, tm)) {   // every K block skipped: no MMA wrote the accumulator
#pragma unroll
                for (int k = 0; k < 32; ++k) ra[k] = 0u;
                Epi::begin(ep, st, row, tn);
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) Epi::consume(ep, st, row, tn * BN + c * 32, ra);
                Epi::end(ep, st, row, tn);
            } else {
                tmem_ld32(t0, ra);
                Epi::begin(ep, st, row, tn);   // its global loads overlap the first TMEM load
#pragma unroll 1
                for (int c = 0; c < BN / 32; c += 2) {
                    tmem_wait_ld(ra);
                    tmem_ld32(t0 + (uint32_t)((c + 1) * 32), rb);
                    Epi::consume(ep, st, row, tn * BN + c * 32, ra);
                    tmem_wait_ld(rb);
                    if (c + 2 < BN / 32) tmem_ld32(t0 + (uint32_t)((c + 2) * 32), ra);
                    Epi::consume(ep, st, row, tn * BN + (c + 1) * 32, rb);
                }
                Epi::end(ep, st, row, tn);
            }
            release();
        }
    }
    tc_fence_before();
    __syncthreads();
    // a pair: no CTA releases its tensor memory or leaves while the other's MMAs, copies or
    // arrivals may still reach it
    if (kCta2) cluster_sync_all();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc<kCta2>(tmem_base, TMEM_COLS);
    }
}

}  // namespace tc
}  // namespace vce
