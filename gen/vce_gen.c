/*
 * Seeded synthetic inputs for the cross-entropy library, its tests and its bench.
 *
 * This file holds no cross-entropy arithmetic: it only draws numbers.  Both the
 * CUDA path and the fp64 oracle take their inputs from here, so every draw is a
 * pure function of (seed, stream, counter) and any row of any matrix can be
 * regenerated on its own, in any order, by any thread.
 *
 * Counter hash: the 64-bit finaliser of SplitMix64 (Steele, Lea & Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014), applied to
 * key + (counter + 1) * golden-gamma.  Uniform doubles take the top 53 bits.
 * Normals use the Box-Muller transform (cosine branch only, one normal per
 * element, so element e depends on counters 2e and 2e+1 alone).
 * Integers in [0, n) use the 64x64->128 multiply-high range reduction
 * (Lemire 2019), whose bias is below n / 2^64.
 *
 * Values are produced in double, rounded to fp32 by the C cast (round to
 * nearest even), and for bf16 storage rounded once more from those fp32 bits
 * to the nearest bf16 with ties to even.  Plain C99, no platform intrinsics.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed ^ 0x5DEECE66DULL) + stream * GOLDEN_GAMMA);
}

static uint64_t draw(uint64_t key, uint64_t ctr) { return mix64(key + (ctr + 1) * GOLDEN_GAMMA); }

static double u01(uint64_t h) { return (double)(h >> 11) * (1.0 / 9007199254740992.0); }

static double normal_at(uint64_t key, uint64_t e) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = 1.0 - u01(draw(key, 2 * e)); /* (0, 1] */
    double u2 = u01(draw(key, 2 * e + 1));   /* [0, 1) */
    return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

static uint16_t f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static float bf16_bits_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ---- exported primitives ---------------------------------------------------- */

uint64_t vce_gen_hash(uint64_t seed, uint64_t stream, uint64_t ctr) {
    return draw(stream_key(seed, stream), ctr);
}

/* out[i] = lo + (hi - lo) * U[0,1), i = 0..n-1, counters ctr0..ctr0+n-1. */
void vce_gen_uniform_f64(uint64_t seed, uint64_t stream, uint64_t ctr0, int64_t n, double lo,
                         double hi, double* out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = lo + (hi - lo) * u01(draw(key, ctr0 + (uint64_t)i));
}

/* out[i] uniform in [0, range), i = 0..n-1. */
void vce_gen_uniform_int(uint64_t seed, uint64_t stream, uint64_t ctr0, int64_t n, uint64_t range,
                         int64_t* out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) {
        unsigned __int128 p = (unsigned __int128)draw(key, ctr0 + (uint64_t)i) * range;
        out[i] = (int64_t)(uint64_t)(p >> 64);
    }
}

/* A uniformly drawn permutation of 0..n-1 (Fisher-Yates, Durstenfeld form). */
void vce_gen_permutation(uint64_t seed, uint64_t stream, int64_t n, int64_t* perm) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) perm[i] = i;
    for (int64_t i = n - 1; i > 0; --i) {
        unsigned __int128 p = (unsigned __int128)draw(key, (uint64_t)i) * (uint64_t)(i + 1);
        int64_t j = (int64_t)(uint64_t)(p >> 64);
        int64_t tmp = perm[i];
        perm[i] = perm[j];
        perm[j] = tmp;
    }
}

/*
 * Rows r0 .. r0+nrows-1 of a [*, ncols] matrix with N(mean, std^2) entries; the
 * element (r, j) is normal number r*ncols + j of the stream.  Rows land in `out`
 * with a stride of ld_out elements.
 *
 * Optional "raised target" rows: when raise_col != NULL and raise_col[r - r0] >= 0,
 * entry (r, raise_col) is replaced after the row is drawn by
 * round(max over the whole drawn row + raise_by[r - r0]), computed in double and
 * rounded to the storage type.  This builds rows whose target logit stands a
 * chosen margin above every other entry.
 */
void vce_gen_normal_rows_f32(uint64_t seed, uint64_t stream, int64_t r0, int64_t nrows,
                             int64_t ncols, int64_t ld_out, double mean, double std,
                             const int64_t* raise_col, const double* raise_by, float* out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t r = 0; r < nrows; ++r) {
        float* row = out + r * ld_out;
        uint64_t base = (uint64_t)(r0 + r) * (uint64_t)ncols;
        for (int64_t j = 0; j < ncols; ++j) row[j] = (float)(mean + std * normal_at(key, base + (uint64_t)j));
        if (raise_col && raise_col[r] >= 0 && raise_col[r] < ncols) {
            double mx = -INFINITY;
            for (int64_t j = 0; j < ncols; ++j) mx = row[j] > mx ? row[j] : mx;
            row[raise_col[r]] = (float)(mx + raise_by[r]);
        }
    }
}

void vce_gen_normal_rows_bf16(uint64_t seed, uint64_t stream, int64_t r0, int64_t nrows,
                              int64_t ncols, int64_t ld_out, double mean, double std,
                              const int64_t* raise_col, const double* raise_by, uint16_t* out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t r = 0; r < nrows; ++r) {
        uint16_t* row = out + r * ld_out;
        uint64_t base = (uint64_t)(r0 + r) * (uint64_t)ncols;
        for (int64_t j = 0; j < ncols; ++j)
            row[j] = f32_to_bf16_bits((float)(mean + std * normal_at(key, base + (uint64_t)j)));
        if (raise_col && raise_col[r] >= 0 && raise_col[r] < ncols) {
            double mx = -INFINITY;
            for (int64_t j = 0; j < ncols; ++j) {
                double v = (double)bf16_bits_to_f32(row[j]);
                mx = v > mx ? v : mx;
            }
            row[raise_col[r]] = f32_to_bf16_bits((float)(mx + raise_by[r]));
        }
    }
}

/*
 * Rows r0 .. r0+nrows-1 of a [*, ncols] matrix whose element (r, j) is
 *     std * (normal number r*ncols + j of the stream) + a[r - r0] * bf16(add[(r - r0), j]),
 * computed in double, rounded to fp32 and then to bf16 (ties to even).  `add` holds nrows
 * rows of ncols bf16 values (stride ncols).  With add = the classifier rows of the rows'
 * labels this draws hidden states aligned with their targets.
 */
void vce_gen_aligned_rows_bf16(uint64_t seed, uint64_t stream, int64_t r0, int64_t nrows, int64_t ncols,
                               double std, const uint16_t* add, const double* a, uint16_t* out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t r = 0; r < nrows; ++r) {
        uint16_t* row = out + r * ncols;
        const uint16_t* ar = add + r * ncols;
        uint64_t base = (uint64_t)(r0 + r) * (uint64_t)ncols;
        for (int64_t j = 0; j < ncols; ++j) {
            double v = std * normal_at(key, base + (uint64_t)j);
            if (a[r] != 0.0) v += a[r] * (double)bf16_bits_to_f32(ar[j]);
            row[j] = f32_to_bf16_bits((float)v);
        }
    }
}

/* Copy columns [c0, c0+w) of nrows rows (strides ld_in / ld_out, elements of `esize` bytes). */
void vce_gen_copy_cols(const void* in, int64_t ld_in, int64_t nrows, int64_t c0, int64_t w,
                       int64_t esize, void* out, int64_t ld_out) {
    const char* src = (const char*)in;
    char* dst = (char*)out;
    for (int64_t r = 0; r < nrows; ++r)
        memcpy(dst + (r * ld_out) * esize, src + (r * ld_in + c0) * esize, (size_t)(w * esize));
}
