// Fused linear cross-entropy: loss, dE and dW of softmax(E W^T) without storing the logits.
//
// Method: apple/ml-cross-entropy issue #14 (Cut Cross-Entropy): linear_cross_entropy(e, c,
// targets) with the classifier weight only; impl="cce_exact" (no gradient filtering, so the
// result is the plain CE gradient); use_kahan (dc = dW and de = dE kept in compensated
// precision).  The CE numerics are those of torchtitan PR #5723 (target-excluded
// log-sum-exp, softplus NLL, the p_t = 1/4 branch of the target gradient).
//
// Steps, all on the tensor cores through tc_gemm.cuh (bf16 operands, fp32 accumulators); every
// operand is read in its natural row-major layout (K-major or MN-major tiles):
//   1. z = E W^T tile by tile (256 rows on a CTA pair x 256 vocabulary columns, K = D); the
//      epilogue keeps per-row (max, sum-exp) over the tile's non-target columns and the target
//      logit, one partial per (row, vocabulary tile); a merge gives L', x, the loss and row_stats.
//   2. per vocabulary chunk of Vc columns:
//        G = c (softmax - onehot) of the recomputed z tile, split G = G_hi + G_lo in bf16
//            (a 16-bit significand in total), written once as [T, Vc];
//        dW[chunk] = G^T E      (A = G MN-major, B = E MN-major, K = 2T: G_hi^T E + G_lo^T E)
//        dE      += G W[chunk]  (A = G K-major, B = W MN-major, K = 2Vc)
//      Both gradient GEMMs accumulate compensated: every 1024 products of the K loop are summed
//      afresh in tensor memory and added into a (sum, compensation) pair with a two-sum; dE's
//      pair is carried across chunks in global memory, merged the same way.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <vector>

#include "tc_gemm.cuh"
#include "tc_launch.cuh"
#include "vce.h"
#include "vce_device.cuh"
#include "vce_check.cuh"
#include "vce_host.h"
#include "vce_linear.h"

namespace vce {
namespace {

using tc::BM;
using tc::BN;
using tc::BK;
using tc::Mat;

constexpr int64_t kChunkCols = 32768;   // vocabulary columns per gradient chunk (a multiple of BN)

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

// ------------------------------------------------------------------------------------------
// epilogues

// Step 1: per (row, vocabulary tile): (max, sum-exp) over non-target columns < V, target logit.
struct EpiStats {
    static constexpr int kScratch = 0;
    struct Params {
        const int64_t* labels;
        int64_t ignore_index, T, V;
        float4* part;   // [tiles_n][T]
    };
    struct Row {
        float m, s, mb, zt;
        int64_t t;
        bool own;
    };
    __device__ __forceinline__ static void begin(const Params& p, Row& r, int row, int) {
        r.m = -kInf;
        r.s = 0.f;
        r.mb = 0.f;
        r.zt = 0.f;
        r.own = false;
        r.t = row < p.T ? p.labels[row] : p.ignore_index;
        if (r.t == p.ignore_index) r.t = -1;
    }
    __device__ __forceinline__ static void consume(const Params& p, Row& r, int, int col0, const uint32_t (&acc)[32]) {
        float v[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(acc[k]);
        if ((int64_t)col0 + 32 > p.V) {   // vocabulary tail: columns past V are not logits
#pragma unroll
            for (int k = 0; k < 32; ++k)
                if ((int64_t)col0 + k >= p.V) v[k] = -kInf;
        }
        const uint64_t rel = (uint64_t)(r.t - col0);
        if (rel < 32) {   // the target column: take it out of the sum (column test)
#pragma unroll
            for (int k = 0; k < 32; ++k)
                if (rel == (uint64_t)k) {
                    r.zt = v[k];
                    r.own = true;
                    v[k] = -kInf;
                }
        }
        ms_push<32>(v, r.m, r.s, r.mb);
    }
    __device__ __forceinline__ static void end(const Params& p, Row& r, int row, int tn) {
        if (row < p.T) p.part[(int64_t)tn * p.T + row] = make_float4(r.m, r.s, r.own ? r.zt : 0.f, r.own ? 1.f : 0.f);
    }
};

// Step 2a: G = c * (softmax - onehot) on the chunk's columns, as bf16 hi + lo, row-major.
// With gradient filtering (keep_w != null) it also marks the 128 x 128 blocks of G that stay:
// those where a valid row has its target or a non-target probability p_ij >= eps.  Each warp
// ORs its 32 rows' marks; the first warp to set a block's bit also sets it in the transposed
// table and counts the block.
struct EpiGrad {
    // per epilogue warp: G_hi and G_lo of its 32 rows x 64 columns, 4 KB each (see put/flush)
    static constexpr int kScratch = 4 * 8192;
    struct Params {
        const int64_t* labels;
        int64_t T, width, col_off;   // rows, chunk width, chunk's first global column
        const float4* row_stats;
        const float* grad_output;
        int go_per_row;
        uint16_t *g_hi, *g_lo;       // [T_pad][ldg]
        int64_t ldg;
        float eps;                   // filter threshold on p_ij (used when keep_w != null)
        uint32_t* keep_w;            // [Vc/128][ldw]: bit (row block) per column block (dW's M tiles)
        int ldw;
        uint32_t* keep_e;            // [T_pad/128][lde]: bit (column block) per row block (dE's M tiles)
        int lde;
        unsigned long long* kept;    // blocks kept, or null
    };
    struct Row {
        float coef, bias, gt, thr;   // thr: p_ij >= eps  <=>  2^(z log2e - bias) >= thr
        float bias_c;                // bias - log2 |coef|: |coef| 2^(z log2e - bias) = 2^(z log2e - bias_c)
        uint32_t sign;               // 0x80008000 when coef < 0 (flips both halves of a packed bf16 pair)
        int64_t tl;
        bool zero;
        uint32_t bits;               // kept marks of this row's two 128-column halves of the tile
        uint8_t* scratch;            // this warp's 8 KB of shared memory
    };
    __device__ __forceinline__ static void begin(const Params& p, Row& r, int row, int tn) {
        r.zero = true;
        r.coef = r.bias = r.gt = r.bias_c = 0.f;
        r.sign = 0u;
        r.thr = kInf;
        r.tl = -1;
        r.bits = 0u;
        if (row < p.T) {
            const float4 st = p.row_stats[row];
            if (st.w != 0.f) {
                const float c = p.grad_output[p.go_per_row ? row : 0] * st.w;
                r.zero = false;
                r.coef = c * st.y;
                r.bias = (st.x == -kInf) ? 0.f : st.x * kLog2e;
                r.bias_c = r.bias - log2f(fabsf(r.coef));   // +inf for coef = 0: every entry 2^-inf = 0
                r.sign = r.coef < 0.f ? 0x80008000u : 0u;
                r.gt = c * st.z;
                r.tl = p.labels[row] - p.col_off;
                if (st.y > 0.f) r.thr = p.eps / st.y;   // p_ij = sigma(x) 2^(z log2e - bias)
                const int64_t rel = r.tl - (int64_t)tn * BN;
                if (rel >= 0 && rel < BN && r.tl < p.width) r.bits = 1u << (int)(rel >> 7);
            }
        }
    }
    __device__ __forceinline__ static void consume(const Params& p, Row& r, int row, int col0,
                                                   const uint32_t (&acc)[32]) {
        uint32_t hi[16], lo[16];
        // The common piece -- a weighted row, no filtering, neither its target column nor the
        // vocabulary's end among its 32 columns -- takes the coefficient into the exponent:
        // g = 2^(z log2e - bias_c), one FFMA and one exp2 per entry.  An entry below 2^-126
        // flushes to zero there; G only feeds the dW and dE sums, where such a term is far
        // below the fp32 rounding of any nonzero sum.
        if (!r.zero && !p.keep_w && (uint64_t)(r.tl - col0) >= 32u && (int64_t)col0 + 32 <= p.width) {
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
                const float g0 = ex2(fmaf(__uint_as_float(acc[k]), kLog2e, -r.bias_c));
                const float g1 = ex2(fmaf(__uint_as_float(acc[k + 1]), kLog2e, -r.bias_c));
                const uint32_t h = pack_bf16x2(g0, g1);
                hi[k / 2] = h ^ r.sign;
                lo[k / 2] = pack_bf16x2(g0 - bf16_lo(h), g1 - bf16_hi(h)) ^ r.sign;
            }
        } else {
            float emax = 0.f;   // largest 2^(z log2e - bias) over the piece's columns < width
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
                float g[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int col = col0 + k + e;
                    const float ev = ex2(fmaf(__uint_as_float(acc[k + e]), kLog2e, -r.bias));
                    float x = r.coef * ev;
                    if (p.keep_w && col < p.width) emax = fmaxf(emax, ev);
                    if (col == r.tl) x = r.gt;
                    if (r.zero || col >= p.width) x = 0.f;
                    g[e] = x;
                }
                const uint32_t h = pack_bf16x2(g[0], g[1]);
                const float r0 = g[0] - bf16_lo(h), r1 = g[1] - bf16_hi(h);
                hi[k / 2] = h;
                lo[k / 2] = pack_bf16x2(r0, r1);
            }
            // A target column in the piece keeps its block anyway (begin), so including its
            // value in emax changes nothing.
            if (p.keep_w && !r.zero && emax >= r.thr) r.bits |= 1u << ((col0 % BN) >> 7);
        }
        put(r, col0, hi, lo);
        if ((col0 >> 5) & 1) flush(p, r, row, col0 - 32);   // the second 32 columns of a 64-column pair
    }
    // G goes out through shared memory so that every store writes whole 128-byte lines: a
    // thread holds 64 B of its own row per piece, and storing that directly writes half
    // sectors of 32 different rows per instruction.  A row of the scratch is 128 B (64
    // columns); its 16-byte chunk c sits in slot c ^ (row & 7), so that the eight lanes of a
    // quarter warp hit eight different bank groups both when each writes its own row (put)
    // and when they read the eight chunks of one row (flush).
    __device__ __forceinline__ static void put(const Row& r, int col0, const uint32_t (&hi)[16],
                                               const uint32_t (&lo)[16]) {
        const int lane = threadIdx.x & 31;
        const int c0 = ((col0 >> 5) & 1) * 4;   // first chunk of this piece within the 128-byte row
        uint8_t* row_h = r.scratch + lane * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int slot = (c0 + q) ^ (lane & 7);
            tc::sts16(row_h + slot * 16, make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]));
            tc::sts16(row_h + 4096 + slot * 16, make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]));
        }
    }
    // The warp's 32 rows x 64 columns from col0 to row-major [T_pad][ldg], four rows of 128 B per
    // store.  Evict-first stores: the chunk's G (512 MB at T = 8192) is read back from DRAM by
    // the next two GEMMs anyway, and should not push E and W out of L2 meanwhile.
    __device__ __forceinline__ static void flush(const Params& p, const Row& r, int row, int col0) {
        __syncwarp();
        const int lane = threadIdx.x & 31;
        const int row0 = row - lane;   // the warp's first row
        const int c = lane & 7;
        const int64_t t_pad = (p.T + 127) / 128 * 128;   // G is [round_up(T, 128)][ldg]
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + (lane >> 3);
            const int off = rr * 128 + ((c ^ (rr & 7)) * 16);
            const uint4 h = tc::lds16(r.scratch + off);
            const uint4 l = tc::lds16(r.scratch + 4096 + off);
            if (!dbg::ok(row0 + rr < t_pad && col0 + 64 <= p.ldg, dbg::kTile)) continue;
            const int64_t at = (int64_t)(row0 + rr) * p.ldg + col0 + c * 8;
            st_stream16(p.g_hi + at, h);
            st_stream16(p.g_lo + at, l);
        }
        __syncwarp();   // the reads above before the next pair's writes
    }
    __device__ __forceinline__ static void end(const Params& p, Row& r, int row, int tn) {
        if (!p.keep_w) return;
        const uint32_t b = __reduce_or_sync(0xffffffffu, r.bits);   // the warp's 32 rows
        if ((threadIdx.x & 31) != 0) return;
        const int rb = row >> 7;   // row block of this warp's first row
#pragma unroll
        for (int h = 0; h < BN / 128; ++h) {
            if (!((b >> h) & 1u)) continue;
            const int cb = tn * (BN / 128) + h;
            const uint32_t bit = 1u << (rb & 31);
            if (atomicOr(&p.keep_w[(int64_t)cb * p.ldw + (rb >> 5)], bit) & bit) continue;   // set already
            atomicOr(&p.keep_e[(int64_t)rb * p.lde + (cb >> 5)], 1u << (cb & 31));
            if (p.kept) atomicAdd(p.kept, 1ull);
        }
    }
};

// Step 2b/2c: a partial product merged into a (sum, compensation) pair of fp32 arrays in
// global memory with a two-sum: the first part initialises the pair, the last writes
// sum + compensation to the output (bf16 or fp32) at row out_row_off + row.  dE: one part per
// vocabulary chunk, the pair [T, D] with its compensation array.  dW: one part per half of the
// rows of T (two parts), the pair the chunk's [width, D] sums alone (comp = null: with two
// parts the compensation would only ever hold the last merge's error, which is rounded away
// with it).
struct EpiKahan {
    static constexpr int kScratch = 0;
    struct Params {
        float *sum, *comp;   // [rows][cols]; comp may be null (the pair's compensation is then 0)
        int64_t rows, cols;
        int first, last;
        void* out;
        int bf16;
        int64_t out_row_off;
    };
    struct Row {};
    __device__ __forceinline__ static void begin(const Params&, Row&, int, int) {}
    // (a, ka) + (x, kx) -> (s, c): s + c = a + x exactly up to the compensations' own sum
    __device__ __forceinline__ static void merge(float a, float ka, float x, float kx, float& s, float& c) {
        s = a + x;   // a + x = s + e exactly (Knuth's two-sum); the compensation accumulates e
        const float bp = s - a;
        const float e = (a - (s - bp)) + (x - bp);
        c = (ka + kx) + e;
    }
    __device__ __forceinline__ static void consume(const Params& p, Row&, int row, int col0, const uint32_t (&acc)[32]) {
        if (row >= p.rows || col0 >= p.cols) return;
        float x[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) x[k] = __uint_as_float(acc[k]);
        const int64_t base = (int64_t)row * p.cols + col0;
        const int64_t obase = (p.out_row_off + row) * p.cols + col0;
        const bool has_comp = p.comp != nullptr;
        if (p.cols - col0 >= 32) {   // full 32-column piece: 16-byte accesses
            // four groups' loads are issued before their stores: the stores go to the same
            // arrays, so loads interleaved with them would each wait out a memory latency
#pragma unroll
            for (int q0 = 0; q0 < 8; q0 += 4) {
                float4 ld_a[4], ld_k[4];
                if (!p.first) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        ld_a[q] = *reinterpret_cast<const float4*>(p.sum + base + 4 * (q0 + q));
                        ld_k[q] = has_comp ? *reinterpret_cast<const float4*>(p.comp + base + 4 * (q0 + q))
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
#pragma unroll
                for (int q = q0; q < q0 + 4; ++q) {
                    float s[4], c[4];
                    if (p.first) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) { s[e] = x[4 * q + e]; c[e] = 0.f; }
                    } else {
                        const float av[4] = {ld_a[q - q0].x, ld_a[q - q0].y, ld_a[q - q0].z, ld_a[q - q0].w};
                        const float kv[4] = {ld_k[q - q0].x, ld_k[q - q0].y, ld_k[q - q0].z, ld_k[q - q0].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) merge(av[e], kv[e], x[4 * q + e], 0.f, s[e], c[e]);
                    }
                    if (p.last) {
                        if (p.bf16) {
                            uint2 w = make_uint2(pack_bf16x2(s[0] + c[0], s[1] + c[1]),
                                                 pack_bf16x2(s[2] + c[2], s[3] + c[3]));
                            *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.out) + obase + 4 * q) = w;
                        } else {
                            *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + obase + 4 * q) =
                                make_float4(s[0] + c[0], s[1] + c[1], s[2] + c[2], s[3] + c[3]);
                        }
                    } else {
                        *reinterpret_cast<float4*>(p.sum + base + 4 * q) = make_float4(s[0], s[1], s[2], s[3]);
                        if (has_comp)
                            *reinterpret_cast<float4*>(p.comp + base + 4 * q) = make_float4(c[0], c[1], c[2], c[3]);
                    }
                }
            }
            return;
        }
        const int n = (int)(p.cols - col0);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            if (k >= n) break;
            float sv = x[k], cv = 0.f;
            if (!p.first) merge(p.sum[base + k], has_comp ? p.comp[base + k] : 0.f, x[k], 0.f, sv, cv);
            if (p.last) {
                if (p.bf16)
                    reinterpret_cast<uint16_t*>(p.out)[obase + k] = to_bf16(sv + cv);
                else
                    reinterpret_cast<float*>(p.out)[obase + k] = sv + cv;
            } else {
                p.sum[base + k] = sv;
                if (has_comp) p.comp[base + k] = cv;
            }
        }
    }
    __device__ __forceinline__ static void end(const Params&, Row&, int, int) {}
};

// ------------------------------------------------------------------------------------------
// host side

// CUDA events around each GEMM launch of one call, on the call's stream (measurement only).
struct GemmTimer {
    enum { kStats = 0, kGrad = 1, kDW = 2, kDE = 3, kKinds = 4 };
    std::vector<cudaEvent_t> ev;   // begin and end of each launch, in launch order
    std::vector<int> kind;         // the kind of each launch
    bool mark(cudaStream_t s) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return false;
        ev.push_back(e);
        return cudaEventRecord(e, s) == cudaSuccess;
    }
    bool begin(cudaStream_t s) { return mark(s); }
    bool end(cudaStream_t s, int k) {
        kind.push_back(k);
        return mark(s);
    }
    ~GemmTimer() {
        for (cudaEvent_t e : ev) cudaEventDestroy(e);
    }
};

struct Layout {
    int64_t T, D, V, T_pad, V_pad, Vc, tiles_v;
    int ldw, lde;   // words per row of the two filter tables
    size_t off_part, off_stats, off_ghi, off_glo, off_sum, off_comp, off_wsum, off_keep_w, off_keep_e, keep_bytes, total;
};

bool layout(int64_t T, int64_t D, int64_t V, Layout* L) {
    if (T < 1 || D < 8 || V < 1 || (D % 8) != 0) return false;
    if (T > (1 << 30) || V > (1ll << 31) || D > (1 << 20)) return false;
    L->T = T;
    L->D = D;
    L->V = V;
    L->T_pad = round_up(T, BM);
    L->tiles_v = cdiv(V, BN);
    L->V_pad = L->tiles_v * BN;
    L->Vc = std::min<int64_t>(kChunkCols, L->V_pad);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) & ~size_t(255);
        return o;
    };
    L->off_part = take((size_t)L->tiles_v * T * 16);
    L->off_stats = take((size_t)T * 16);
    L->off_ghi = take((size_t)L->T_pad * L->Vc * 2);
    L->off_glo = take((size_t)L->T_pad * L->Vc * 2);
    L->off_sum = take((size_t)T * D * 4);
    L->off_comp = take((size_t)T * D * 4);
    L->off_wsum = take((size_t)L->Vc * D * 4);   // dW partial of one chunk's first half of T
    // gradient-filter tables of one chunk: [Vc/128][ldw] and [T_pad/128][lde] bits
    L->ldw = (int)cdiv(L->T_pad / 128, 32);
    L->lde = (int)cdiv(L->Vc / 128, 32);
    L->off_keep_w = take((size_t)(L->Vc / 128) * L->ldw * 4);
    L->off_keep_e = take((size_t)(L->T_pad / 128) * L->lde * 4);
    L->keep_bytes = off - L->off_keep_w;   // both tables, contiguous
    L->total = off;
    return true;
}

}  // namespace
}  // namespace vce

using namespace vce;

extern "C" size_t linear_ce_workspace_bytes(int64_t T, int64_t D, int64_t V) {
    Layout L;
    return layout(T, D, V, &L) ? L.total : 0;
}

namespace vce {

VCE_DEBUG_READER(debug_word_lce)

namespace {

// The whole call; with a timer, events are recorded around every GEMM launch.
int linear_ce_run(const void* E, const void* W, int64_t T, int64_t D, int64_t V, const int64_t* labels,
                  int64_t ignore_index, vce_reduction red, const float* grad_output, float* loss_rows,
                  float* loss_out, void* dE, void* dW, vce_dtype grad_dt, float filter_eps,
                  unsigned long long* kept_blocks, void* workspace, size_t workspace_bytes, int32_t* status,
                  cudaStream_t s, GemmTimer* timer) {
    if (!(filter_eps >= 0.f) || filter_eps == kInf) return VCE_ERR_ARG;   // NaN, negative or infinite
    if (red != VCE_RED_NONE && red != VCE_RED_SUM && red != VCE_RED_MEAN) return VCE_ERR_DTYPE;
    if (grad_dt != VCE_BF16 && grad_dt != VCE_F32) return VCE_ERR_DTYPE;
    Layout L;
    if (!layout(T, D, V, &L)) return VCE_ERR_SHAPE;
    if (!E || !W || !labels || !grad_output || !loss_rows || !dE || !dW || !status) return VCE_ERR_NULL;
    if (red != VCE_RED_NONE && !loss_out) return VCE_ERR_NULL;
    if (!workspace || workspace_bytes < L.total) return VCE_ERR_WORKSPACE;
    if (!aligned(E, 16) || !aligned(W, 16) || !aligned(workspace, 256) || !aligned(labels, 8) ||
        !aligned(loss_rows, 4) || !aligned(grad_output, 4) || !aligned(dE, 16) || !aligned(dW, 16) ||
        (loss_out && !aligned(loss_out, 4)) || (kept_blocks && !aligned(kept_blocks, 8)))
        return VCE_ERR_ALIGN;
    int rc = require_sm100();
    if (rc) return rc;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* part = reinterpret_cast<float*>(ws + L.off_part);
    float* stats = reinterpret_cast<float*>(ws + L.off_stats);
    uint16_t* ghi = reinterpret_cast<uint16_t*>(ws + L.off_ghi);
    uint16_t* glo = reinterpret_cast<uint16_t*>(ws + L.off_glo);
    float* dsum = reinterpret_cast<float*>(ws + L.off_sum);
    float* dcomp = reinterpret_cast<float*>(ws + L.off_comp);
    float* wsum = reinterpret_cast<float*>(ws + L.off_wsum);
    const bool filter = filter_eps > 0.f;
    uint32_t* keep_w = filter ? reinterpret_cast<uint32_t*>(ws + L.off_keep_w) : nullptr;
    uint32_t* keep_e = filter ? reinterpret_cast<uint32_t*>(ws + L.off_keep_e) : nullptr;

    if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return VCE_ERR_CUDA;
    if (kept_blocks && cudaMemsetAsync(kept_blocks, 0, sizeof(unsigned long long), s) != cudaSuccess)
        return VCE_ERR_CUDA;

    // operands, row-major: E [T, D], W [V, D], the gradient chunk halves [T_pad, Vc]
    const Mat mE{E, D, T, D}, mW{W, D, V, D}, mGhi{ghi, L.Vc, L.T_pad, L.Vc}, mGlo{glo, L.Vc, L.T_pad, L.Vc};
    const int nkD = (int)cdiv(D, BK);
    const int tiles_t = (int)(L.T_pad / BM);
    // 256-row tiles on CTA pairs where the rows split evenly, else single CTAs
    const bool pairs_t = tiles_t % 2 == 0;

    // 1. forward statistics over the whole vocabulary
    {
        tc::GemmArgs g{tiles_t, (int)L.tiles_v, nkD, nkD, 0, 0, 0, 0, status};
        EpiStats::Params ep{labels, ignore_index, T, V, reinterpret_cast<float4*>(part)};
        if (timer && !timer->begin(s)) return VCE_ERR_CUDA;
        // two K blocks per stage where D gives an even number of them (eight MMAs per stage)
        const cudaError_t e = nkD % 2 == 0 ? tc::launch_gemm<EpiStats, false, false, false, true>(mE, mE, mW, g, ep, pairs_t, s)
                                           : tc::launch_gemm<EpiStats, false, false>(mE, mE, mW, g, ep, pairs_t, s);
        if (e != cudaSuccess) return VCE_ERR_CUDA;
        if (timer && !timer->end(s, GemmTimer::kStats)) return VCE_ERR_CUDA;
        if (launch_stats_merge(part, (int)L.tiles_v, T, V, labels, ignore_index, loss_rows, stats, status, s) !=
            cudaSuccess)
            return VCE_ERR_CUDA;
        if (red != VCE_RED_NONE &&
            launch_loss_reduce(loss_rows, labels, T, V, ignore_index, red, loss_out, stats, s) != cudaSuccess)
            return VCE_ERR_CUDA;
    }

    // 2. gradients, one vocabulary chunk at a time.  Exact: CTA pairs; dW as two partial products
    // over the halves of T merged with a two-sum, dE's chunk partials merged the same way.
    // Filtered: single CTAs skipping the dropped K blocks, dW in one product.
    const int64_t nchunks = cdiv(L.V_pad, L.Vc);
    for (int64_t ci = 0; ci < nchunks; ++ci) {
        const int64_t off = ci * L.Vc;
        const int64_t width = std::min<int64_t>(L.Vc, V - off);
        const int64_t width_pad = round_up(width, BN);
        if (filter && cudaMemsetAsync(keep_w, 0, L.keep_bytes, s) != cudaSuccess) return VCE_ERR_CUDA;
        {
            tc::GemmArgs g{tiles_t, (int)(width_pad / BN), nkD, nkD, 0, 0, (int)off, 0, status};
            EpiGrad::Params ep{labels, T,      width,  off,    reinterpret_cast<const float4*>(stats), grad_output,
                               red == VCE_RED_NONE, ghi, glo, L.Vc, filter_eps, keep_w, L.ldw, keep_e, L.lde,
                               filter ? kept_blocks : nullptr};
            if (timer && !timer->begin(s)) return VCE_ERR_CUDA;
            const cudaError_t e =
                nkD % 2 == 0 ? tc::launch_gemm<EpiGrad, false, false, false, true>(mE, mE, mW, g, ep, pairs_t, s)
                             : tc::launch_gemm<EpiGrad, false, false>(mE, mE, mW, g, ep, pairs_t, s);
            if (e != cudaSuccess) return VCE_ERR_CUDA;
            if (timer && !timer->end(s, GemmTimer::kGrad)) return VCE_ERR_CUDA;
        }
        {   // dW[off : off + width] = G^T E: A = G (MN-major), B = E (MN-major), K = 2 T_pad (hi then lo);
            // M tile = 128 vocabulary columns = one row of keep_w, K block = 64 rows of T.  width_pad
            // is a multiple of 256, so the M tiles always pair.
            const int nkT = (int)(L.T_pad / BK);
            if (filter) {
                tc::GemmArgs g{(int)(width_pad / BM), (int)cdiv(D, BN), 2 * nkT, nkT, 0, 0, 0, 1, status};
                g.skip = keep_w;
                g.skip_ld = L.ldw;
                tc::EpiStore::Params ep{dW, D, width, D, off, grad_dt == VCE_BF16};
                if (timer && !timer->begin(s)) return VCE_ERR_CUDA;
                if (tc::launch_gemm<tc::EpiStore, true, true>(mGhi, mGlo, mE, g, ep, false, s) != cudaSuccess)
                    return VCE_ERR_CUDA;
                if (timer && !timer->end(s, GemmTimer::kDW)) return VCE_ERR_CUDA;
            } else {
                // nkT is even (T_pad is a multiple of 128): part h takes K blocks [h nkT/2, (h+1) nkT/2)
                // of E's rows and of both halves of G, G_hi's and G_lo's tiles of a block in one
                // stage beside E's
                for (int h = 0; h < 2; ++h) {
                    tc::GemmArgs g{(int)(width_pad / BM), (int)cdiv(D, BN), nkT / 2, nkT / 2, 0, 0, 0, 1, status};
                    g.ka0 = h * (nkT / 2);
                    EpiKahan::Params ep{wsum, nullptr, width, D, h == 0, h == 1, dW, grad_dt == VCE_BF16, off};
                    if (timer && !timer->begin(s)) return VCE_ERR_CUDA;
                    if (tc::launch_gemm<EpiKahan, true, true, true>(mGhi, mGlo, mE, g, ep, true, s) != cudaSuccess)
                        return VCE_ERR_CUDA;
                    if (timer && !timer->end(s, GemmTimer::kDW)) return VCE_ERR_CUDA;
                }
            }
        }
        {   // dE += G W[off : off + width]: A = G (K-major), B = W rows (MN-major), K = 2 width (hi then lo);
            // M tile = 128 rows of T = one row of keep_e, K block = 64 vocabulary columns
            const int nkc = (int)cdiv(width, BK);
            EpiKahan::Params ep{dsum, dcomp, T, D, ci == 0, ci == nchunks - 1, dE, grad_dt == VCE_BF16, 0};
            if (timer && !timer->begin(s)) return VCE_ERR_CUDA;
            if (filter) {
                tc::GemmArgs g{tiles_t, (int)cdiv(D, BN), 2 * nkc, nkc, (int)off, 0, 0, 1, status};
                g.skip = keep_e;
                g.skip_ld = L.lde;
                if (tc::launch_gemm<EpiKahan, false, true>(mGhi, mGlo, mW, g, ep, false, s) != cudaSuccess)
                    return VCE_ERR_CUDA;
            } else {   // G_hi's and G_lo's tiles of a K block in one stage beside W's
                tc::GemmArgs g{tiles_t, (int)cdiv(D, BN), nkc, nkc, (int)off, 0, 0, 1, status};
                if (tc::launch_gemm<EpiKahan, false, true, true>(mGhi, mGlo, mW, g, ep, pairs_t, s) != cudaSuccess)
                    return VCE_ERR_CUDA;
            }
            if (timer && !timer->end(s, GemmTimer::kDE)) return VCE_ERR_CUDA;
        }
    }
    return VCE_OK;
}

}  // namespace
}  // namespace vce

extern "C" int linear_ce_fwd_bwd_filtered(const void* E, const void* W, int64_t T, int64_t D, int64_t V,
                                          const int64_t* labels, int64_t ignore_index, vce_reduction red,
                                          const float* grad_output, float* loss_rows, float* loss_out, void* dE,
                                          void* dW, vce_dtype grad_dt, float filter_eps,
                                          unsigned long long* kept_blocks, void* workspace, size_t workspace_bytes,
                                          int32_t* status, vce_stream_t s) {
    return linear_ce_run(E, W, T, D, V, labels, ignore_index, red, grad_output, loss_rows, loss_out, dE, dW, grad_dt,
                         filter_eps, kept_blocks, workspace, workspace_bytes, status, s, nullptr);
}

extern "C" int linear_ce_fwd_bwd_timed(const void* E, const void* W, int64_t T, int64_t D, int64_t V,
                                       const int64_t* labels, int64_t ignore_index, vce_reduction red,
                                       const float* grad_output, float* loss_rows, float* loss_out, void* dE,
                                       void* dW, vce_dtype grad_dt, float filter_eps, unsigned long long* kept_blocks,
                                       void* workspace, size_t workspace_bytes, int32_t* status, vce_stream_t s,
                                       float* gemm_ms, int* gemm_launches) {
    if (!gemm_ms || !gemm_launches) return VCE_ERR_NULL;
    GemmTimer timer;
    int rc = linear_ce_run(E, W, T, D, V, labels, ignore_index, red, grad_output, loss_rows, loss_out, dE, dW,
                           grad_dt, filter_eps, kept_blocks, workspace, workspace_bytes, status, s, &timer);
    for (int k = 0; k < GemmTimer::kKinds; ++k) {
        gemm_ms[k] = 0.f;
        gemm_launches[k] = 0;
    }
    if (rc == VCE_OK && cudaStreamSynchronize(s) != cudaSuccess) rc = VCE_ERR_CUDA;
    for (size_t i = 0; rc == VCE_OK && i < timer.kind.size(); ++i) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, timer.ev[2 * i], timer.ev[2 * i + 1]) != cudaSuccess) rc = VCE_ERR_CUDA;
        gemm_ms[timer.kind[i]] += ms;
        gemm_launches[timer.kind[i]] += 1;
    }
    return rc;
}

extern "C" int linear_ce_fwd_bwd(const void* E, const void* W, int64_t T, int64_t D, int64_t V, const int64_t* labels,
                                 int64_t ignore_index, vce_reduction red, const float* grad_output, float* loss_rows,
                                 float* loss_out, void* dE, void* dW, vce_dtype grad_dt, void* workspace,
                                 size_t workspace_bytes, int32_t* status, vce_stream_t s) {
    return linear_ce_fwd_bwd_filtered(E, W, T, D, V, labels, ignore_index, red, grad_output, loss_rows, loss_out, dE,
                                      dW, grad_dt, 0.f, nullptr, workspace, workspace_bytes, status, s);
}
