/*
 * oracle.c -- TEST INFRASTRUCTURE, NOT PRODUCT CODE.
 *
 * A plain, slow, obviously correct CPU statement of the FP8 NT GEMM with
 * fine-grained scaling and its two MoE grouped layouts, as described on the
 * page "DeepSeek开源周第三天DeepGEMM" (explinks.com): section "核心功能"
 * (fine-grained scaling, two-level accumulation), section "基本用法" (LHS is
 * an FP8 m x k matrix with FP32 scales of shape [m, ceil(k/128)], RHS an FP8
 * n x k matrix with FP32 scales [ceil(n/128), ceil(k/128)], BF16 output),
 * the three GEMM kinds listed under "DeepGEMM提供三种FP8GEMM实现", and the
 * promotion excerpt "两级精度累加与细粒度缩放" (final += sA * sB * partial per
 * 128-wide K block).
 *
 * Only the test suite, the package's smoke() entry and bench.py's CPU
 * baseline may load this file's library.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Definition computed (exact up to FP64 rounding order):
 *
 *   D[m,n] = bf16_rne( sum_kb  sA[m,kb] * sB[n/128,kb] * sum_{k in kb} dec(A[m,k]) * dec(B[n,k]) )
 *
 * where kb runs over ceil(k/128) blocks of 128 K-columns (the last block may be
 * shorter), dec() decodes an FP8 byte to its real value, and bf16_rne rounds the
 * FP64 value directly to bfloat16, ties to even.
 *
 * The same file states the step before the GEMM: per-token (1 x 128)
 * quantization of activations into the FP8 LHS and its scales
 * (oracle_quantize_per_token, with the FP8 encoder oracle_encode_fp8), from
 * the same page's section "基本用法" and section 5.2 of the page
 * "企业官网建设流程全解析" (scales come from a scan for each group's
 * largest magnitude).
 *
 * Pins: every function here is checked by tests/test_oracle_pins.py against
 * values fixed by the pages (format widths and maxima of E4M3/E5M2, page
 * "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践" section 3.1 table), closed forms, brute force
 * over all FP8 codes, library routines on special cases (numpy float64 matmul
 * with unit scales, torch's float8 and bfloat16 conversions) and invariants
 * (zero scales, power-of-two scale linearity, grouped == per-group dense).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_E4M3 0
#define ORACLE_E5M2 1
#define ORACLE_KBLOCK 128 /* K-block of the fine-grained scales and of promotion */
#define ORACLE_NBLOCK 128 /* N-block of the RHS scales */

/* ---------------------------------------------------------------- decoding */

/* E4M3 ("fn" variant, the one torch calls float8_e4m3fn): 1 sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits.  No infinities; the two codes with
 * all exponent and mantissa bits set (0x7F, 0xFF) are NaN.  Largest finite
 * magnitude 1.75 * 2^8 = 448; exponent field 0 encodes subnormals f * 2^-9. */
static double decode_e4m3(unsigned code) {
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 0xFu, f = code & 7u;
    double v;
    if (e == 15u && f == 7u) return NAN;
    if (e == 0u)
        v = ldexp((double)f, -9);                 /* 0.f * 2^(1-7) */
    else
        v = ldexp((double)(8u + f), (int)e - 10); /* 1.f * 2^(e-7) */
    return s ? -v : v;
}

/* E5M2: 1 sign bit, 5 exponent bits with bias 15, 2 mantissa bits, IEEE-like:
 * exponent field 31 is infinity (mantissa 0) or NaN; largest finite 1.75*2^15 =
 * 57344; subnormals f * 2^-16. */
static double decode_e5m2(unsigned code) {
    unsigned s = (code >> 7) & 1u, e = (code >> 2) & 0x1Fu, f = code & 3u;
    double v;
    if (e == 31u) {
        if (f != 0u) return NAN;
        return s ? -INFINITY : INFINITY;
    }
    if (e == 0u)
        v = ldexp((double)f, -16);                /* 0.f * 2^(1-15) */
    else
        v = ldexp((double)(4u + f), (int)e - 17); /* 1.f * 2^(e-15) */
    return s ? -v : v;
}

double oracle_decode(int fmt, int code) {
    if (fmt == ORACLE_E4M3) return decode_e4m3((unsigned)code & 0xFFu);
    if (fmt == ORACLE_E5M2) return decode_e5m2((unsigned)code & 0xFFu);
    return NAN;
}

static int fill_table(int fmt, double table[256]) {
    if (fmt != ORACLE_E4M3 && fmt != ORACLE_E5M2) return -1;
    for (int c = 0; c < 256; ++c) table[c] = oracle_decode(fmt, c);
    return 0;
}

/* ------------------------------------------------------- bfloat16 rounding */

/* Round an FP64 value directly (no intermediate float) to bfloat16 with round
 * to nearest, ties to even.  bfloat16 has float32's exponent range (normal
 * exponents -126..127) and 8 significant bits, so its spacing in the binade
 * [2^E, 2^(E+1)) is 2^(E-7), and 2^-133 below 2^-126 (subnormals).  NaN becomes
 * the canonical quiet NaN 0x7FC0; magnitudes that round past the largest finite
 * value (0x7F7F = (2 - 2^-7) * 2^127) become infinity. */
uint16_t oracle_bf16_rne(double x) {
    uint16_t sign;
    double a, q, y;
    int e, E, qexp;
    if (isnan(x)) return 0x7FC0u;
    sign = signbit(x) ? 0x8000u : 0u;
    a = fabs(x);
    if (a == 0.0) return sign;
    if (a >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u); /* also +-inf */
    (void)frexp(a, &e);               /* a = m * 2^e, m in [0.5, 1) */
    E = e - 1;                        /* a in [2^E, 2^(E+1)) */
    qexp = (E < -126 ? -126 : E) - 7; /* exponent of one bf16 ulp here */
    q = ldexp(1.0, qexp);
    y = nearbyint(a / q) * q;         /* a/q is exact; default mode is ties-to-even */
    if (y > ldexp(255.0, 120))        /* largest finite bf16 = 255 * 2^120 */
        return (uint16_t)(sign | 0x7F80u);
    if (y == 0.0) return sign;
    {
        /* y is now exactly representable in bfloat16, hence in float32: take
         * the upper half of its float32 encoding, built here by hand. */
        int ye;
        double ym = frexp(y, &ye);    /* y = ym * 2^ye, ym in [0.5,1) */
        int Eb = ye - 1;              /* y = 1.f * 2^Eb */
        uint32_t bits;
        if (Eb >= -126) {
            uint32_t mant = (uint32_t)ldexp(ym * 2.0 - 1.0, 7); /* 7 fraction bits */
            bits = ((uint32_t)(Eb + 127) << 7) | mant;
        } else {
            bits = (uint32_t)ldexp(y, 133);                     /* subnormal: y / 2^-133 */
        }
        return (uint16_t)(sign | (uint16_t)bits);
    }
}

/* ------------------------------------------------------------ the dot core */

/* One output element: the two-level sum of the page's promotion excerpt.  The
 * inner block sum is exact in FP64 for E4M3 x E4M3 (every product is an integer
 * multiple of 2^-18 below 2^18, and 128 of them need at most 43 bits). */
static double output_element(const uint8_t *a_row, const float *sa_row,
                             const uint8_t *b_row, const float *sb_row,
                             int k, const double *ta, const double *tb) {
    int num_kb = (k + ORACLE_KBLOCK - 1) / ORACLE_KBLOCK;
    double acc = 0.0;
    for (int kb = 0; kb < num_kb; ++kb) {
        int k0 = kb * ORACLE_KBLOCK;
        int k1 = k0 + ORACLE_KBLOCK < k ? k0 + ORACLE_KBLOCK : k;
        double partial = 0.0;
        for (int kk = k0; kk < k1; ++kk) partial += ta[a_row[kk]] * tb[b_row[kk]];
        acc += ((double)sa_row[kb] * (double)sb_row[kb]) * partial;
    }
    return acc;
}

static int shapes_ok(int m, int n, int k) { return m >= 0 && n >= 0 && k >= 1; }

/* ------------------------------------------------------------- dense (NT) */

/* A: [m][k] bytes, row-major.  sA: [m][ceil(k/128)] row-major.
 * B: [n][k] bytes, row-major (the "transposed" RHS of the NT layout).
 * sB: [ceil(n/128)][ceil(k/128)] row-major.
 * Outputs (either may be NULL): D64 [m][n] unrounded FP64, D16 [m][n] bf16 bits. */
int oracle_gemm_fp8_nt(const uint8_t *A, int a_fmt, const float *sA,
                       const uint8_t *B, int b_fmt, const float *sB,
                       int m, int n, int k, double *D64, uint16_t *D16) {
    double ta[256], tb[256];
    int num_kb = (k + ORACLE_KBLOCK - 1) / ORACLE_KBLOCK;
    if (!shapes_ok(m, n, k) || fill_table(a_fmt, ta) || fill_table(b_fmt, tb)) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long r = 0; r < m; ++r) {
        for (int c = 0; c < n; ++c) {
            double v = output_element(A + r * (long long)k, sA + r * (long long)num_kb,
                                      B + c * (long long)k, sB + (long long)(c / ORACLE_NBLOCK) * num_kb,
                                      k, ta, tb);
            if (D64) D64[r * (long long)n + c] = v;
            if (D16) D16[r * (long long)n + c] = oracle_bf16_rne(v);
        }
    }
    return 0;
}

/* The same definition evaluated only at `count` (row, col) positions, for
 * sampled checks of shapes too large to compute in full. */
int oracle_gemm_fp8_nt_at(const uint8_t *A, int a_fmt, const float *sA,
                          const uint8_t *B, int b_fmt, const float *sB,
                          int m, int n, int k, long long count,
                          const long long *rows, const long long *cols,
                          double *D64, uint16_t *D16) {
    double ta[256], tb[256];
    int num_kb = (k + ORACLE_KBLOCK - 1) / ORACLE_KBLOCK;
    if (!shapes_ok(m, n, k) || fill_table(a_fmt, ta) || fill_table(b_fmt, tb)) return -1;
    for (long long i = 0; i < count; ++i)
        if (rows[i] < 0 || rows[i] >= m || cols[i] < 0 || cols[i] >= n) return -2;
#pragma omp parallel for schedule(dynamic, 64)
    for (long long i = 0; i < count; ++i) {
        long long r = rows[i], c = cols[i];
        double v = output_element(A + r * k, sA + r * num_kb, B + c * k,
                                  sB + (c / ORACLE_NBLOCK) * num_kb, k, ta, tb);
        if (D64) D64[i] = v;
        if (D16) D16[i] = oracle_bf16_rne(v);
    }
    return 0;
}

/* ------------------------------------------------- contiguous grouped layout */

/* Groups concatenated along M ("连续布局分组GEMM": tokens of different experts
 * grouped on the M axis).  m_indices[r] in [0,G) names the weight matrix that
 * row r multiplies; any other value (the layout uses -1 for alignment padding)
 * leaves row r of D untouched.  B: [G][n][k], sB: [G][ceil(n/128)][ceil(k/128)].
 * D16 is read-modify-write: only rows with a valid group are written. */
int oracle_grouped_contiguous(const uint8_t *A, int a_fmt, const float *sA,
                              const uint8_t *B, int b_fmt, const float *sB,
                              const int32_t *m_indices, int M, int n, int k, int G,
                              double *D64, uint16_t *D16) {
    double ta[256], tb[256];
    int num_kb = (k + ORACLE_KBLOCK - 1) / ORACLE_KBLOCK;
    int num_nb = (n + ORACLE_NBLOCK - 1) / ORACLE_NBLOCK;
    if (!shapes_ok(M, n, k) || G < 1 || fill_table(a_fmt, ta) || fill_table(b_fmt, tb)) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long r = 0; r < M; ++r) {
        int g = m_indices[r];
        if (g < 0 || g >= G) continue;
        const uint8_t *Bg = B + (long long)g * n * k;
        const float *sBg = sB + (long long)g * num_nb * num_kb;
        for (int c = 0; c < n; ++c) {
            double v = output_element(A + r * k, sA + r * num_kb, Bg + (long long)c * k,
                                      sBg + (long long)(c / ORACLE_NBLOCK) * num_kb, k, ta, tb);
            if (D64) D64[r * (long long)n + c] = v;
            if (D16) D16[r * (long long)n + c] = oracle_bf16_rne(v);
        }
    }
    return 0;
}

/* Sampled form: the value row r would receive at column c (rows whose group is
 * invalid report NaN / 0xFFFF, meaning "not written"). */
int oracle_grouped_contiguous_at(const uint8_t *A, int a_fmt, const float *sA,
                                 const uint8_t *B, int b_fmt, const float *sB,
                                 const int32_t *m_indices, int M, int n, int k, int G,
                                 long long count, const long long *rows, const long long *cols,
                                 double *D64, uint16_t *D16) {
    double ta[256], tb[256];
    int num_kb = (k + ORACLE_KBLOCK - 1) / ORACLE_KBLOCK;
    int num_nb = (n + ORACLE_NBLOCK - 1) / ORACLE_NBLOCK;
    if (!shapes_ok(M, n, k) || G < 1 || fill_table(a_fmt, ta) || fill_table(b_fmt, tb)) return -1;
    for (long long i = 0; i < count; ++i)
        if (rows[i] < 0 || rows[i] >= M || cols[i] < 0 || cols[i] >= n) return -2;
#pragma omp parallel for schedule(dynamic, 64)
    for (long long i = 0; i < count; ++i) {
        long long r = rows[i], c = cols[i];
        int g = m_indices[r];
        if (g < 0 || g >= G) {
            if (D64) D64[i] = NAN;
            if (D16) D16[i] = 0xFFFFu;
            continue;
        }
        {
            double v = output_element(A + r * k, sA + r * num_kb,
                                      B + ((long long)g * n + c) * k,
                                      sB + ((long long)g * num_nb + c / ORACLE_NBLOCK) * num_kb,
                                      k, ta, tb);
            if (D64) D64[i] = v;
            if (D16) D16[i] = oracle_bf16_rne(v);
        }
    }
    return 0;
}

/* --------------------------------------------------- masked grouped layout */

/* Fixed capacity per group ("掩码布局分组GEMM": a mask tensor names the valid
 * part).  A: [G][M_cap][k], sA: [G][M_cap][ceil(k/128)], B/sB as above,
 * masked_m[g] = number of valid leading rows of group g.  Rows r with
 * r < masked_m[g] are written; all other rows of D16 [G][M_cap][n] are left
 * untouched.  A count outside [0, M_cap] is clamped into it. */
int oracle_grouped_masked(const uint8_t *A, int a_fmt, const float *sA,
                          const uint8_t *B, int b_fmt, const float *sB,
                          const int32_t *masked_m, int G, int M_cap, int n, int k,
                          double *D64, uint16_t *D16) {
    double ta[256], tb[256];
    int num_kb = (k + ORACLE_KBLOCK - 1) / ORACLE_KBLOCK;
    int num_nb = (n + ORACLE_NBLOCK - 1) / ORACLE_NBLOCK;
    if (!shapes_ok(M_cap, n, k) || G < 1 || fill_table(a_fmt, ta) || fill_table(b_fmt, tb)) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long gr = 0; gr < (long long)G * M_cap; ++gr) {
        long long g = gr / M_cap, r = gr % M_cap;
        int valid = masked_m[g] < 0 ? 0 : (masked_m[g] > M_cap ? M_cap : masked_m[g]);
        if (r >= valid) continue;
        for (int c = 0; c < n; ++c) {
            double v = output_element(A + gr * k, sA + gr * num_kb,
                                      B + (g * n + c) * (long long)k,
                                      sB + (g * num_nb + c / ORACLE_NBLOCK) * (long long)num_kb,
                                      k, ta, tb);
            if (D64) D64[gr * n + c] = v;
            if (D16) D16[gr * n + c] = oracle_bf16_rne(v);
        }
    }
    return 0;
}

/* Sampled form over (g, r, c) triples; rows past the count report NaN / 0xFFFF. */
int oracle_grouped_masked_at(const uint8_t *A, int a_fmt, const float *sA,
                             const uint8_t *B, int b_fmt, const float *sB,
                             const int32_t *masked_m, int G, int M_cap, int n, int k,
                             long long count, const long long *groups, const long long *rows,
                             const long long *cols, double *D64, uint16_t *D16) {
    double ta[256], tb[256];
    int num_kb = (k + ORACLE_KBLOCK - 1) / ORACLE_KBLOCK;
    int num_nb = (n + ORACLE_NBLOCK - 1) / ORACLE_NBLOCK;
    if (!shapes_ok(M_cap, n, k) || G < 1 || fill_table(a_fmt, ta) || fill_table(b_fmt, tb)) return -1;
    for (long long i = 0; i < count; ++i)
        if (groups[i] < 0 || groups[i] >= G || rows[i] < 0 || rows[i] >= M_cap ||
            cols[i] < 0 || cols[i] >= n) return -2;
#pragma omp parallel for schedule(dynamic, 64)
    for (long long i = 0; i < count; ++i) {
        long long g = groups[i], r = rows[i], c = cols[i];
        long long gr = g * M_cap + r;
        int valid = masked_m[g] < 0 ? 0 : (masked_m[g] > M_cap ? M_cap : masked_m[g]);
        if (r >= valid) {
            if (D64) D64[i] = NAN;
            if (D16) D16[i] = 0xFFFFu;
            continue;
        }
        {
            double v = output_element(A + gr * k, sA + gr * num_kb, B + (g * n + c) * (long long)k,
                                      sB + (g * num_nb + c / ORACLE_NBLOCK) * (long long)num_kb,
                                      k, ta, tb);
            if (D64) D64[i] = v;
            if (D16) D16[i] = oracle_bf16_rne(v);
        }
    }
    return 0;
}

/* ------------------------------------------------ K-grouped layout */

/* Groups concatenated along K: the weight-gradient step of MoE training
 * contracts over tokens, and each expert's tokens form one segment of the K
 * axis (the pages name the grouped kinds by the training forward pass and
 * inference; this is the same scaled NT product with the K range restricted
 * per group).  A: [M][K] bytes and B: [N][K] bytes, both K-major, shared by all
 * groups; sA: [M][ceil(K/128)] and sB: [ceil(N/128)][ceil(K/128)] row-major, the
 * scaling of the NT GEMM.  Group g covers the K columns
 * [off_g, off_g + ks[g]) with off_g = ks[0] + ... + ks[g-1]; every ks[g] is a
 * multiple of 128 (so K blocks and scale blocks never straddle two groups) and
 * their sum is at most K.  Output D [G][M][N]:
 *
 *   D[g][m][n] = sum over the K blocks kb of segment g of
 *                sA[m,kb] * sB[n/128,kb] * sum_{k in kb} dec(A[m,k]) * dec(B[n,k])
 *
 * (an empty segment gives 0).  Returns -3 for sizes that break those rules. */
static double k_segment_element(const uint8_t *a_row, const float *sa_row, const uint8_t *b_row,
                                const float *sb_row, int kb0, int kb1, int K, const double *ta,
                                const double *tb) {
    double acc = 0.0;
    for (int kb = kb0; kb < kb1; ++kb) {
        int k0 = kb * ORACLE_KBLOCK;
        int k1 = k0 + ORACLE_KBLOCK < K ? k0 + ORACLE_KBLOCK : K;
        double partial = 0.0;
        for (int kk = k0; kk < k1; ++kk) partial += ta[a_row[kk]] * tb[b_row[kk]];
        acc += ((double)sa_row[kb] * (double)sb_row[kb]) * partial;
    }
    return acc;
}

static int k_segments_ok(const int32_t *ks, int G, int K) {
    long long total = 0;
    for (int g = 0; g < G; ++g) {
        if (ks[g] < 0 || ks[g] % ORACLE_KBLOCK != 0) return 0;
        total += ks[g];
    }
    return total <= K;
}

int oracle_k_grouped(const uint8_t *A, int a_fmt, const float *sA, const uint8_t *B, int b_fmt,
                     const float *sB, const int32_t *ks, int G, int M, int N, int K,
                     double *D64, uint16_t *D16) {
    double ta[256], tb[256];
    int num_kb = (K + ORACLE_KBLOCK - 1) / ORACLE_KBLOCK;
    if (!shapes_ok(M, N, K) || G < 1 || fill_table(a_fmt, ta) || fill_table(b_fmt, tb)) return -1;
    if (!k_segments_ok(ks, G, K)) return -3;
    int off = 0;
    for (int g = 0; g < G; ++g) {
        int kb0 = off / ORACLE_KBLOCK, kb1 = (off + ks[g]) / ORACLE_KBLOCK;
        off += ks[g];
#pragma omp parallel for schedule(dynamic, 1)
        for (long long r = 0; r < M; ++r) {
            for (int c = 0; c < N; ++c) {
                double v = k_segment_element(A + r * K, sA + r * num_kb, B + (long long)c * K,
                                             sB + (long long)(c / ORACLE_NBLOCK) * num_kb, kb0, kb1, K, ta, tb);
                long long o = ((long long)g * M + r) * N + c;
                if (D64) D64[o] = v;
                if (D16) D16[o] = oracle_bf16_rne(v);
            }
        }
    }
    return 0;
}

/* Sampled form over (g, m, n) triples. */
int oracle_k_grouped_at(const uint8_t *A, int a_fmt, const float *sA, const uint8_t *B, int b_fmt,
                        const float *sB, const int32_t *ks, int G, int M, int N, int K, long long count,
                        const long long *groups, const long long *rows, const long long *cols,
                        double *D64, uint16_t *D16) {
    double ta[256], tb[256];
    int num_kb = (K + ORACLE_KBLOCK - 1) / ORACLE_KBLOCK;
    if (!shapes_ok(M, N, K) || G < 1 || fill_table(a_fmt, ta) || fill_table(b_fmt, tb)) return -1;
    if (!k_segments_ok(ks, G, K)) return -3;
    for (long long i = 0; i < count; ++i)
        if (groups[i] < 0 || groups[i] >= G || rows[i] < 0 || rows[i] >= M || cols[i] < 0 || cols[i] >= N)
            return -2;
#pragma omp parallel for schedule(dynamic, 64)
    for (long long i = 0; i < count; ++i) {
        long long g = groups[i], r = rows[i], c = cols[i];
        int off = 0;
        for (long long h = 0; h < g; ++h) off += ks[h];
        double v = k_segment_element(A + r * K, sA + r * num_kb, B + c * K, sB + (c / ORACLE_NBLOCK) * num_kb,
                                     off / ORACLE_KBLOCK, (off + ks[g]) / ORACLE_KBLOCK, K, ta, tb);
        if (D64) D64[i] = v;
        if (D16) D16[i] = oracle_bf16_rne(v);
    }
    return 0;
}

/* ------------------------------------------- per-token FP8 quantization */

/* FP8 code of the float v rounded to nearest, ties to even, saturating at the
 * largest finite magnitude (448 for E4M3, 57344 for E5M2; page
 * "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践", section 3.1).
 * Written from the definition of rounding: among the finite non-negative codes,
 * whose values grow with the code, take the two that bracket |v| and keep the
 * nearer; on a tie keep the one whose last mantissa bit (the code's bit 0) is
 * 0.  The sign bit is v's sign bit (so -0 and negative values that round to
 * zero give 0x80).  v must be finite; NaN gives 0xFF. */
static int encode_in_table(const double table[256], int top, float v) {
    double a;
    int lo, hi;
    unsigned sign;
    if (isnan(v)) return 0xFF;
    sign = signbit(v) ? 0x80u : 0u;
    a = fabs((double)v);
    if (a >= table[top]) return (int)(sign | (unsigned)top);
    /* table[lo] <= a < table[hi], hi = lo + 1 (binary search, codes 0..top) */
    lo = 0;
    hi = top;
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (table[mid] <= a) lo = mid; else hi = mid;
    }
    {
        double dlo = a - table[lo], dhi = table[hi] - a;
        int c = dlo < dhi ? lo : dhi < dlo ? hi : ((lo & 1) == 0 ? lo : hi);
        return (int)(sign | (unsigned)c);
    }
}

static int top_code(int fmt) { return fmt == ORACLE_E4M3 ? 0x7E : 0x7B; } /* largest finite positive code */

int oracle_encode_fp8(int fmt, float v) {
    double table[256];
    if (fill_table(fmt, table) != 0) return -1;
    return encode_in_table(table, top_code(fmt), v);
}

/* Per-token (1 x 128) quantization of activations, the step that produces the
 * LHS of the GEMM: page "DeepSeek开源周第三天DeepGEMM", section "基本用法" (the
 * LHS is FP8 with one FP32 scale per row and 128-wide K block), and page
 * "企业官网建设流程全解析", section 5.2 (a scale is found by scanning the
 * group for its largest magnitude).  For each row r and K block kb, over the
 * columns of the block that lie inside k:
 *
 *   amax      = max |x[r][c]|
 *   s[r][kb]  = amax / fmax      (float32 division; 1 when amax == 0, so an
 *                                 all-zero group never divides by zero)
 *   q[r][c]   = encode( x[r][c] / s[r][kb] )   (float32 division, then the
 *                                               rounding of oracle_encode_fp8)
 *
 * Every step is float32 because the codes are integers decided by floating
 * point: the quantizer being checked decides them in float32 as well.
 * x is float [rows][ld_x] (bfloat16 inputs widen to float exactly), q is
 * [rows][k] bytes, s is row-major [rows][ceil(k/128)].  Returns 0, or -1 for
 * a bad argument. */
int oracle_quantize_per_token(const float *x, int ld_x, int fmt, uint8_t *q, float *s, int rows, int k) {
    double table[256];
    int kb, top;
    float fmax;
    if (fill_table(fmt, table) != 0) return -1;
    if (rows < 0 || k < 1 || ld_x < k) return -1;
    top = top_code(fmt);
    fmax = fmt == ORACLE_E4M3 ? 448.0f : 57344.0f;
    kb = (k + ORACLE_KBLOCK - 1) / ORACLE_KBLOCK;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        for (int b = 0; b < kb; ++b) {
            int c0 = b * ORACLE_KBLOCK;
            int c1 = c0 + ORACLE_KBLOCK < k ? c0 + ORACLE_KBLOCK : k;
            const float *xr = x + (size_t)r * (size_t)ld_x;
            float amax = 0.0f, scale;
            for (int c = c0; c < c1; ++c) {
                float m = fabsf(xr[c]);
                if (m > amax) amax = m;
            }
            scale = amax > 0.0f ? amax / fmax : 1.0f;
            s[(size_t)r * (size_t)kb + (size_t)b] = scale;
            for (int c = c0; c < c1; ++c)
                q[(size_t)r * (size_t)k + (size_t)c] = (uint8_t)encode_in_table(table, top, xr[c] / scale);
        }
    }
    return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
