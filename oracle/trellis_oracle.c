/*
 * Plain CPU oracle for the packed-Trellis weight decode and the
 * decode-and-multiply product.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and
 * the benchmark's CPU-baseline leg load this library.  The product path (the
 * CUDA library and its Python binding) never calls it and shares no code,
 * header, table or constant generator with it.
 *
 * Every step is written out in the order of the Metal kernel source printed
 * on the page "mlx-bun 0.2.0 -> 0.4.0", file
 * package/src/model/trellis-wide-prefill.ts (the `mlx_bun_trellis_wide_prefill`
 * kernel body and its `wideTrellisPrefill` wrapper).  Readings taken where the
 * source is silent:
 *   - the 12-bit code-to-value quotient is the IEEE fp32 round-to-nearest
 *     quotient code / 147.800537109375 (the page's residual-corrected form
 *     reaches the same value for every code; the test suite checks this);
 *   - conversions to bf16 (the kernel's `T(...)`) round to nearest, ties to
 *     even;
 *   - the product's "fp32 result" is the exact sum of the bf16 products,
 *     accumulated in double and rounded once to fp32 (no summation order is
 *     fixed by the page, so none is imitated).
 *
 * Single-threaded, no vectorisation, no blocking.  Built with
 * -ffp-contract=off so that every float operation is the one written.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "trellis_oracle.h"

/* ---- bf16 <-> fp32 (round to nearest even) -------------------------------- */

float oracle_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN, never reached here */
    /* add half an ulp of bf16, plus one more when the kept lsb is odd */
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* ---- step 1: the L-bit window of weight t (tail-biting block) -------------- */
/* The block is the bit-string of `wpb` little-endian words.  Weight t of the
 * block starts at bit (T-1-t)*k; when the window runs past the end of its word
 * it continues in the next word, and past the block's last word it continues
 * in word 0 of the same block. */
uint32_t oracle_window(const uint32_t *blk, int t, int k, int L, int T) {
    const uint32_t wpb = (uint32_t)(T * k / 32);
    const uint32_t pos = (uint32_t)(T - 1 - t) * (uint32_t)k;
    const uint32_t wi = pos >> 5;
    const uint32_t off = pos & 31u;
    uint32_t win = blk[wi] >> off;
    if (off + (uint32_t)L > 32u) {
        const uint32_t next = (wi + 1u == wpb) ? 0u : wi + 1u;
        win |= blk[next] << (32u - off);
    }
    win &= (1u << L) - 1u;
    return win;
}

/* ---- step 2: the "1MAD" hash of a window to an integer code ---------------- */
int32_t oracle_code(uint32_t win) {
    const uint32_t z = win * 34038481u + 76625530u; /* wraps modulo 2^32 */
    const uint32_t p = (z & 0x00FF00FFu) + ((z >> 8) & 0x00FF00FFu);
    return (int32_t)((p & 0xFFFFu) + (p >> 16)) - 510;
}

/* ---- step 3: code to value ------------------------------------------------- */
float oracle_value(int32_t code) {
    const float c = 147.800537109375f;
    return (float)code / c;
}

/* ---- step 4: one weight = bf16(value * scale) ------------------------------ */
uint16_t oracle_weight(const uint32_t *blk, int t, int k, int L, int T, uint16_t scale_bf16) {
    const float s = oracle_bf16_to_f32(scale_bf16);
    const float v = oracle_value(oracle_code(oracle_window(blk, t, k, L, T)));
    const float prod = v * s;
    return oracle_f32_to_bf16(prod);
}

int oracle_check_geometry(int64_t K, int64_t N, int k, int L, int T) {
    if (K <= 0 || N <= 0) return -2;
    if (k < 1 || k > 8 || L < 1 || L > 24 || L <= k) return -3;
    if (T <= 0 || (T * k) % 32 != 0) return -3;
    if (K % T != 0) return -2;
    return 0;
}

/* ---- dense decode of rows [n0, n1) into out[(n-n0)*K + kk] ----------------- */
int oracle_decode_rows(const uint32_t *codes, const uint16_t *scales, int64_t K, int64_t N,
                       int k, int L, int T, int64_t n0, int64_t n1, uint16_t *out) {
    const int rc = oracle_check_geometry(K, N, k, L, T);
    if (rc != 0) return rc;
    if (n0 < 0 || n1 > N || n0 > n1) return -2;
    const int64_t row_words = K * k / 32;
    const int64_t wpb = (int64_t)T * k / 32;
    const int64_t nblocks = K / T;
    for (int64_t n = n0; n < n1; ++n) {
        for (int64_t b = 0; b < nblocks; ++b) {
            const uint32_t *blk = codes + n * row_words + b * wpb;
            for (int t = 0; t < T; ++t)
                out[(n - n0) * K + b * T + t] = oracle_weight(blk, t, k, L, T, scales[n]);
        }
    }
    return 0;
}

/* ---- product with dense bf16 rows ------------------------------------------ */
/* W holds rows [n0, n0+nrows) of the [N, K] weight matrix; x is [M, K].
 * ref[m*nrows + i]    = fp32( sum_k W[i,k] * x[m,k] )   (double accumulation)
 * refabs[m*nrows + i] = sum_k |W[i,k] * x[m,k]|
 * Each bf16 x bf16 product is exact in double. */
int oracle_gemm_dense(const uint16_t *x, const uint16_t *W, int64_t M, int64_t K, int64_t nrows,
                      float *ref, double *refabs) {
    if (M <= 0 || K <= 0 || nrows < 0) return -2;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t i = 0; i < nrows; ++i) {
            double acc = 0.0, aabs = 0.0;
            for (int64_t kk = 0; kk < K; ++kk) {
                const double p = (double)oracle_bf16_to_f32(W[i * K + kk]) *
                                 (double)oracle_bf16_to_f32(x[m * K + kk]);
                acc += p;
                aabs += fabs(p);
            }
            ref[m * nrows + i] = (float)acc;
            if (refabs) refabs[m * nrows + i] = aabs;
        }
    }
    return 0;
}

/* ---- gate/up: act = bf16(silu(g) * u) --------------------------------------- */
/* The SiLU-gated product of two projections that share x.  The page
 * "mlx-bun 0.4.0 -> 0.5.0" (package/src/model/trellis-linear.ts) imports fused
 * gate/up kernels without showing their bodies; reading taken: silu(v) =
 * v / (1 + e^-v) of the bf16 gate output times the bf16 up output, evaluated
 * exactly (double) and rounded to fp32, then to bf16 (nearest even). */
void oracle_silu_mul(const uint16_t *g, const uint16_t *u, int64_t n, uint16_t *act) {
    for (int64_t i = 0; i < n; ++i) {
        const double v = (double)oracle_bf16_to_f32(g[i]);
        const double s = v / (1.0 + exp(-v));
        act[i] = oracle_f32_to_bf16((float)(s * (double)oracle_bf16_to_f32(u[i])));
    }
}

