/*
 * CPU oracle for the tensor-core multiply-accumulate D = A·B + C.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or table with the CUDA library.
 *
 * What it computes (the plain definition, "Tensor Core 数据布局的演进",
 * overview: the three tensor-core generations all compute D = AB + C):
 *
 *     D[i][j] = C[i][j] + sum_{k=0}^{K-1} a[i][k] * b[k][j]
 *     S[i][j] =           sum_{k=0}^{K-1} |a[i][k] * b[k][j]|
 *
 * in fp64 over the already rounded operands.  bf16, fp16 and e4m3 values are
 * exact in fp64, and so are their products, so the only rounding is the
 * fp64 summation (error far below any tolerance applied to the result).
 *
 * Block scaling ("Tensor Core 数据布局的演进", section "Block-Scaled MMA 的
 * Scale Factors"): SFA[m][sfk] scales the elements of row m of A inside the
 * sfk-th K block, SFB[n][sfk] the elements of column n of B:
 *     a[i][k] = A[i][k] * sf(SFA[i][k/blk])
 *     b[k][j] = B[k][j] * sf(SFB[j][k/blk])
 * Two scale modes (the same section: a 32-bit scale word holds one, two or
 * four scales per row, scale_vec::1X / 2X / 4X):
 *   block_scaled = 1  UE8M0 scales, blk = 32: e4m3 operands (one scale per
 *                     32-element MMA K step) or e2m1 operands (two per 64);
 *   block_scaled = 2  UE4M3 scales, blk = 16: e2m1 operands (four per 64).
 * SFA is stored M x ceil(K/blk) row-major, SFB N x ceil(K/blk) row-major.
 *
 * Operand storage: A is M x K, row-major (A[i*K+k]) when a_row_major, else
 * column-major (A[k*M+i]).  B is K x N, row-major (B[k*N+j]) when b_row_major,
 * else column-major (B[j*K+k]).  C is M x N fp32 row-major, or NULL for 0.
 *
 * Operand formats, decoded from their definitions:
 *   bf16  the upper 16 bits of an IEEE-754 binary32 pattern;
 *   fp16  IEEE-754 binary16 (1/5/10, bias 15, subnormals, inf/NaN at 31);
 *   e4m3  OCP 8-bit floating point E4M3 (1/4/3, bias 7, subnormals,
 *         no infinities, S.1111.111 is NaN, max normal 448);
 *   e2m1  OCP 4-bit floating point E2M1 (1/2/1, bias 1, one subnormal
 *         0.5, no infinities or NaN, max 6), two per byte: element 2t in
 *         bits 0..3 of byte t, element 2t+1 in bits 4..7 (t counts along
 *         the storage order's contiguous dimension);
 *   ue8m0 OCP microscaling scale: 2^(code-127), code 255 is NaN;
 *   ue4m3 unsigned E4M3 scale: the 7 low bits read as a non-negative e4m3
 *         value (0x7F is NaN); codes with bit 7 set have no value (NaN).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1, ORACLE_E4M3 = 2, ORACLE_E2M1 = 3 };
enum { SCALE_NONE = 0, SCALE_UE8M0_32 = 1, SCALE_UE4M3_16 = 2 };

double oracle_decode_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-14 * 2^-10 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

double oracle_decode_e4m3(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);                  /* m/8 * 2^(1-7) */
    else
        v = ldexp((double)(8 + m), e - 10);        /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

double oracle_decode_ue8m0(uint8_t c) {
    return c == 255 ? NAN : ldexp(1.0, (int)c - 127);
}

/* one E2M1 code in the low 4 bits of c */
double oracle_decode_e2m1(uint8_t c) {
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 0x3;
    int m = c & 0x1;
    double v = e == 0 ? 0.5 * m                            /* subnormal: m/2 * 2^(1-1) */
                      : ldexp(2.0 + m, e - 2);              /* (1 + m/2) * 2^(e-1) */
    return sign ? -v : v;
}

double oracle_decode_ue4m3(uint8_t c) {
    if (c & 0x80) return NAN;
    return oracle_decode_e4m3(c);
}

/* element idx (in storage order) of an operand */
static double decode(int dtype, const void *p, int64_t idx) {
    switch (dtype) {
    case ORACLE_F16: return oracle_decode_f16(((const uint16_t *)p)[idx]);
    case ORACLE_BF16: return oracle_decode_bf16(((const uint16_t *)p)[idx]);
    case ORACLE_E2M1: {
        uint8_t byte = ((const uint8_t *)p)[idx / 2];
        return oracle_decode_e2m1(idx % 2 ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF));
    }
    default: return oracle_decode_e4m3(((const uint8_t *)p)[idx]);
    }
}

typedef struct {
    int64_t M, N, K, sfk, blk;
    int dtype, a_row_major, b_row_major, block_scaled;
    const void *A, *B;
    const uint8_t *SFA, *SFB;
} problem;

static double scale(const problem *p, uint8_t code) {
    return p->block_scaled == SCALE_UE4M3_16 ? oracle_decode_ue4m3(code) : oracle_decode_ue8m0(code);
}

/* a[i][k] with its block scale applied */
static double a_elem(const problem *p, int64_t i, int64_t k) {
    int64_t idx = p->a_row_major ? i * p->K + k : k * p->M + i;
    double v = decode(p->dtype, p->A, idx);
    if (p->block_scaled) v *= scale(p, p->SFA[i * p->sfk + k / p->blk]);
    return v;
}

/* b[k][j] with its block scale applied */
static double b_elem(const problem *p, int64_t k, int64_t j) {
    int64_t idx = p->b_row_major ? k * p->N + j : j * p->K + k;
    double v = decode(p->dtype, p->B, idx);
    if (p->block_scaled) v *= scale(p, p->SFB[j * p->sfk + k / p->blk]);
    return v;
}

/* Fill *p; -1 when the operand type and scale mode do not go together:
 * fp16 / bf16 take no scales, e4m3 none or UE8M0 / 32, e2m1 any mode. */
static int make_problem(problem *p, int64_t M, int64_t N, int64_t K, int dtype, const void *A, int a_row_major,
                        const void *B, int b_row_major, const uint8_t *SFA, const uint8_t *SFB, int block_scaled) {
    if (block_scaled < SCALE_NONE || block_scaled > SCALE_UE4M3_16) return -1;
    if (dtype < ORACLE_F16 || dtype > ORACLE_E2M1) return -1;
    if (block_scaled && (!SFA || !SFB)) return -1;
    if (dtype == ORACLE_E4M3 && block_scaled != SCALE_NONE && block_scaled != SCALE_UE8M0_32) return -1;
    if (dtype < ORACLE_E4M3 && block_scaled != SCALE_NONE) return -1;
    int64_t blk = block_scaled == SCALE_UE4M3_16 ? 16 : 32;
    problem q = {M, N, K, (K + blk - 1) / blk, blk, dtype, a_row_major, b_row_major, block_scaled, A, B, SFA, SFB};
    *p = q;
    return 0;
}

static int set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) return nthreads;
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Number of threads an oracle call with this request would use. */
int oracle_threads(int nthreads) { return set_threads(nthreads); }

/*
 * Rows [row0, row1) of the product (pass 0, M for all of it): D and S are
 * (row1 - row0) x N fp64 row-major outputs, row r holding row row0 + r.
 * Returns 0, or -1 on a bad argument or allocation failure.
 */
int oracle_gemm(int64_t M, int64_t N, int64_t K, int dtype,
                const void *A, int a_row_major, const void *B, int b_row_major,
                const float *C, const uint8_t *SFA, const uint8_t *SFB, int block_scaled,
                int64_t row0, int64_t row1, double *D, double *S, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || row0 < 0 || row1 > M || row0 > row1) return -1;
    problem p;
    if (make_problem(&p, M, N, K, dtype, A, a_row_major, B, b_row_major, SFA, SFB, block_scaled)) return -1;
    int64_t rows = row1 - row0;
    /* decode the operands once into plain fp64 matrices: ad (rows x K), bd (K x N) */
    double *ad = (double *)malloc(sizeof(double) * (size_t)(rows * K > 0 ? rows * K : 1));
    double *bd = (double *)malloc(sizeof(double) * (size_t)(K * N > 0 ? K * N : 1));
    if (!ad || !bd) { free(ad); free(bd); return -1; }
    int nt = set_threads(nthreads);
    #pragma omp parallel for num_threads(nt) schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; ++k) ad[r * K + k] = a_elem(&p, row0 + r, k);
    #pragma omp parallel for num_threads(nt) schedule(static)
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < N; ++j) bd[k * N + j] = b_elem(&p, k, j);

    #pragma omp parallel for num_threads(nt) schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t i = row0 + r;
        double *d = D + r * N, *s = S + r * N;
        for (int64_t j = 0; j < N; ++j) { d[j] = 0.0; s[j] = 0.0; }
        for (int64_t k = 0; k < K; ++k) {
            double a = ad[r * K + k];
            const double *b = bd + k * N;
            for (int64_t j = 0; j < N; ++j) {
                double prod = a * b[j];
                d[j] += prod;
                s[j] += fabs(prod);
            }
        }
        for (int64_t j = 0; j < N; ++j) d[j] += C ? (double)C[i * N + j] : 0.0;
    }
    free(ad);
    free(bd);
    return 0;
}

/*
 * Selected entries: for each (rows[e], cols[e]) the same sums as oracle_gemm,
 * evaluated one entry at a time straight from the operand codes.
 */
int oracle_gemm_entries(int64_t M, int64_t N, int64_t K, int dtype,
                        const void *A, int a_row_major, const void *B, int b_row_major,
                        const float *C, const uint8_t *SFA, const uint8_t *SFB, int block_scaled,
                        int64_t n, const int64_t *rows, const int64_t *cols,
                        double *D, double *S, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || n < 0) return -1;
    problem p;
    if (make_problem(&p, M, N, K, dtype, A, a_row_major, B, b_row_major, SFA, SFB, block_scaled)) return -1;
    for (int64_t e = 0; e < n; ++e)
        if (rows[e] < 0 || rows[e] >= M || cols[e] < 0 || cols[e] >= N) return -1;
    int nt = set_threads(nthreads);
    #pragma omp parallel for num_threads(nt) schedule(dynamic, 64)
    for (int64_t e = 0; e < n; ++e) {
        int64_t i = rows[e], j = cols[e];
        double d = 0.0, s = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double prod = a_elem(&p, i, k) * b_elem(&p, k, j);
            d += prod;
            s += fabs(prod);
        }
        D[e] = d + (C ? (double)C[i * N + j] : 0.0);
        S[e] = s;
    }
    return 0;
}

/*
 * Round x to the nearest value with `p` significant bits and exponent floor
 * `emin` (IEEE-style format with subnormals), ties to even; magnitudes that
 * round beyond `maxv` become infinities.  bf16: p = 8, emin = -126,
 * maxv = (2 - 2^-7) * 2^127; fp16: p = 11, emin = -14, maxv = 65504.
 * x / q is exact (q a power of two), and rint rounds ties to even in the
 * default rounding mode.
 */
static double round_to_format(double x, int p, int emin, double maxv) {
    if (x == 0.0 || isnan(x) || isinf(x)) return x;
    int e;
    frexp(fabs(x), &e);                    /* |x| = m * 2^e, m in [0.5, 1) */
    int ex = e - 1 < emin ? emin : e - 1;  /* unbiased exponent of |x|, subnormals share emin */
    double q = ldexp(1.0, ex - (p - 1));
    double r = rint(x / q) * q;
    if (fabs(r) > maxv) return x > 0 ? INFINITY : -INFINITY;
    return r;
}

double oracle_round_bf16(double x) { return round_to_format(x, 8, -126, ldexp(255.0, 120)); }
double oracle_round_f16(double x) { return round_to_format(x, 11, -14, 65504.0); }

/*
 * Two chained products ("Tensor Core 数据布局的演进", section "TMEM 中的累加器":
 * some tcgen05.mma forms read A from tensor memory, so a first product's
 * result can feed a second without leaving the SM):
 *
 *     T[i][j] = sum_k a[i][k] * b[k][j]                 (M x N1, K terms)
 *     P[i][j] = round(T[i][j])                          (to the operand format, RNE)
 *     D[i][n] = C[i][n] + sum_j P[i][j] * e[j][n]       (M x N2, N1 terms)
 *
 * A is M x K row-major, B is K x N1 column-major (B[j*K + k]), E is
 * N1 x N2 column-major (E[n*N1 + j]), C is M x N2 fp32 row-major or NULL;
 * dtype is ORACLE_F16 or ORACLE_BF16 (operands and P).  For each listed row
 * i = rows[r] it writes T, S1 = sum_k |a b| (r x N1), D, S2 = sum_j |P e|
 * (r x N2), all fp64.  Returns 0, or -1 on a bad argument.
 */
int oracle_chain(int64_t M, int64_t N1, int64_t N2, int64_t K, int dtype, const void *A, const void *B,
                 const void *E, const float *C, int64_t nrows, const int64_t *rows, double *T, double *S1,
                 double *D, double *S2, int nthreads) {
    if (M < 0 || N1 < 0 || N2 < 0 || K < 0 || nrows < 0) return -1;
    if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;
    problem first, second;
    if (make_problem(&first, M, N1, K, dtype, A, 1, B, 0, NULL, NULL, SCALE_NONE)) return -1;
    if (make_problem(&second, M, N2, N1, dtype, NULL, 1, E, 0, NULL, NULL, SCALE_NONE)) return -1;
    int nt = set_threads(nthreads);
    #pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows[r];
        double *t = T + r * N1, *s1 = S1 + r * N1, *d = D + r * N2, *s2 = S2 + r * N2;
        for (int64_t j = 0; j < N1; ++j) {
            double acc = 0.0, sabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double prod = a_elem(&first, i, k) * b_elem(&first, k, j);
                acc += prod;
                sabs += fabs(prod);
            }
            t[j] = acc;
            s1[j] = sabs;
        }
        for (int64_t n = 0; n < N2; ++n) {
            double acc = 0.0, sabs = 0.0;
            for (int64_t j = 0; j < N1; ++j) {
                double pv = dtype == ORACLE_BF16 ? oracle_round_bf16(t[j]) : oracle_round_f16(t[j]);
                double prod = pv * b_elem(&second, j, n);
                acc += prod;
                sabs += fabs(prod);
            }
            d[n] = acc + (C ? (double)C[i * N2 + n] : 0.0);
            s2[n] = sabs;
        }
    }
    return 0;
}
