/*
 * GEMM oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library. It shares no code with the CUDA path.
 *
 * What it computes (plain definition, no blocking or reordering):
 *
 *   D[i][j] = alpha * sum_{k=0}^{K-1} A(i,k) * B(k,j) + beta * C[i][j]
 *
 * in IEEE double precision, over the exact values of the fp16/bf16 (or fp8
 * E4M3/E5M2, A and B each in its own format) inputs.
 * The accumulate-into-D form is the one the tensor-core pages state for one
 * MMA (gpu-kernels part 6, "Tensor Cores, layouts, and swizzling", opening
 * paragraph: D = A.B + C; zhenwei tcgen05 page, "Overview" and the
 * interactive K-step walk-through: the first K step overwrites, later steps
 * add); alpha/beta are the BLAS reading of "D = alpha.A.B + beta.C" with
 * beta == 0 never reading C.
 *
 * Operand storage (the "major-ness" of the tcgen05 descriptor pages,
 * gauravjain "LBO, SBO and SWZ for a tcgen05 tile", section 1):
 *   A is logical M x K.  K-major: A[m*lda + k].  MN-major: A[k*lda + m].
 *   B is logical K x N.  K-major: B[n*ldb + k].  MN-major: B[k*ldb + n].
 *   C and D are row-major M x N with leading dimension ldc.
 *
 * Alongside D it returns the error scale used by the parity tolerance:
 *   S[i][j] = |alpha| * sum_k |A(i,k) * B(k,j)| + |beta * C[i][j]|.
 *
 * Rounding to an output format (oracle_round_*) is round-to-nearest-even
 * from the double value in one step (no double rounding through float).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_F32 = 2, ORC_E4M3 = 3, ORC_E5M2 = 4, ORC_TF32 = 5 };

/* TF32 operand read from fp32 storage (tcgen05 kind::tf32 operands are fp32
 * words). Reading: the tensor core keeps the sign, the 8 exponent bits and the
 * top 10 of the 23 fraction bits, i.e. the low 13 fraction bits are dropped
 * (truncation, not rounding); values representable in TF32 are unchanged. */
static double decode_tf32(uint32_t u)
{
    u &= ~(uint32_t)0x1FFF;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25);    /* 1.f * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double decode_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

/*
 * 8-bit floats (the fp8 family a 16-byte core-matrix cell holds 16 of, "LBO,
 * SBO and SWZ for a tcgen05 tile", section 4; the MMA kind selects the A/B
 * type family, "06 Blackwell Tensor Core - tcgen05 MMA"):
 *   E4M3: 1 sign, 4 exponent (bias 7), 3 fraction bits; no infinities, the
 *         all-ones exponent and fraction is NaN; largest finite 448.
 *   E5M2: 1 sign, 5 exponent (bias 15), 2 fraction bits, IEEE-style
 *         infinities and NaNs; largest finite 57344.
 */
static double decode_e4m3(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xf;
    int f = b & 7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);                  /* f * 2^-6 * 2^-3 */
    else
        v = ldexp((double)(f | 8), e - 10);        /* 1.f * 2^(e-7) */
    return sign ? -v : v;
}

static double decode_e5m2(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 2) & 0x1f;
    int f = b & 3;
    double v;
    if (e == 31)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -16);                 /* f * 2^-14 * 2^-2 */
    else
        v = ldexp((double)(f | 4), e - 17);        /* 1.f * 2^(e-15) */
    return sign ? -v : v;
}

double oracle_decode(int fmt, uint32_t bits)
{
    switch (fmt) {
    case ORC_F16: return decode_f16((uint16_t)bits);
    case ORC_BF16: return decode_bf16((uint16_t)bits);
    case ORC_E4M3: return decode_e4m3((uint8_t)bits);
    case ORC_E5M2: return decode_e5m2((uint8_t)bits);
    case ORC_TF32: return decode_tf32(bits);
    default: {
        float x;
        memcpy(&x, &bits, sizeof x);
        return (double)x;
    }
    }
}

static double decode_f32(uint32_t u)
{
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

static double load(const void *p, int fmt, int64_t idx)
{
    switch (fmt) {
    case ORC_F16: return decode_f16(((const uint16_t *)p)[idx]);
    case ORC_BF16: return decode_bf16(((const uint16_t *)p)[idx]);
    case ORC_E4M3: return decode_e4m3(((const uint8_t *)p)[idx]);
    case ORC_E5M2: return decode_e5m2(((const uint8_t *)p)[idx]);
    case ORC_TF32: return decode_tf32(((const uint32_t *)p)[idx]);
    default: return decode_f32(((const uint32_t *)p)[idx]);
    }
}

static double a_at(const void *A, int fmt, int major, int64_t lda, int64_t m, int64_t k)
{
    return load(A, fmt, major == 0 ? m * lda + k : k * lda + m);
}

static double b_at(const void *B, int fmt, int major, int64_t ldb, int64_t k, int64_t n)
{
    return load(B, fmt, major == 0 ? n * ldb + k : k * ldb + n);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Full product. D and S are row-major M x N doubles (S may be NULL).
 * The loop order is i-k-j: row i of D accumulates A(i,k) * row k of B,
 * k = 0, 1, ..., K-1 in that order.
 */
int oracle_gemm(int64_t M, int64_t N, int64_t K,
                const void *A, int in_fmt, int a_major, int64_t lda,
                const void *B, int b_fmt, int b_major, int64_t ldb,
                const void *C, int c_fmt, int64_t ldc,
                double alpha, double beta,
                double *D, double *S, int nthreads)
{
    if (M < 0 || N < 0 || K < 0)
        return 1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int64_t i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < M; ++i) {
        double *acc = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));
        double *sab = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));
        for (int64_t k = 0; k < K; ++k) {
            double a = a_at(A, in_fmt, a_major, lda, i, k);
            for (int64_t j = 0; j < N; ++j) {
                double p = a * b_at(B, b_fmt, b_major, ldb, k, j);
                acc[j] += p;
                sab[j] += fabs(p);
            }
        }
        for (int64_t j = 0; j < N; ++j) {
            double c = (beta != 0.0 && C) ? load(C, c_fmt, i * ldc + j) : 0.0;
            D[i * N + j] = alpha * acc[j] + beta * c;
            if (S)
                S[i * N + j] = fabs(alpha) * sab[j] + fabs(beta * c);
        }
        free(acc);
        free(sab);
    }
    return 0;
}

/*
 * Selected entries only: out_D[e] and out_S[e] for (rows[e], cols[e]).
 * Each entry is the same k = 0..K-1 sum as oracle_gemm, one dot product at
 * a time, so full-size problems can be checked on a sample.
 */
int oracle_gemm_entries(int64_t M, int64_t N, int64_t K,
                        const void *A, int in_fmt, int a_major, int64_t lda,
                        const void *B, int b_fmt, int b_major, int64_t ldb,
                        const void *C, int c_fmt, int64_t ldc,
                        double alpha, double beta,
                        int64_t n_entries, const int64_t *rows, const int64_t *cols,
                        double *out_D, double *out_S, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int bad = 0;
    int64_t e;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
    for (e = 0; e < n_entries; ++e) {
        int64_t i = rows[e], j = cols[e];
        if (i < 0 || i >= M || j < 0 || j >= N) {
            bad |= 1;
            continue;
        }
        double acc = 0.0, sab = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = a_at(A, in_fmt, a_major, lda, i, k) * b_at(B, b_fmt, b_major, ldb, k, j);
            acc += p;
            sab += fabs(p);
        }
        double c = (beta != 0.0 && C) ? load(C, c_fmt, i * ldc + j) : 0.0;
        out_D[e] = alpha * acc + beta * c;
        if (out_S)
            out_S[e] = fabs(alpha) * sab + fabs(beta * c);
    }
    return bad;
}

/*
 * Block-scaled product (MXFP8, the block-scaled tcgen05 MMA of "06 Blackwell
 * Tensor Core - tcgen05 MMA": A(i,k) is scaled by SFA[i][k/32] and B(k,j) by
 * SFB[j][k/32]; the block of 32 elements and the E8M0 scale type follow the
 * OCP Microscaling (MX) definition of MXFP8 that the page names):
 *
 *   D[i][j] = alpha * sum_k (sa(i, k/32) * A(i,k)) * (sb(j, k/32) * B(k,j)) + beta * C[i][j]
 *
 * sa, sb hold E8M0 codes, row-major: sa[i * ldsa + b] for row i of A and
 * block b, sb[j * ldsb + b] for column j of B (ld >= ceil(K/32)). A code e
 * means 2^(e - 127); 255 is NaN. S is the tolerance scale as for oracle_gemm,
 * over the scaled products. Same loop order as oracle_gemm.
 */
double oracle_decode_e8m0(uint8_t e)
{
    return e == 255 ? NAN : ldexp(1.0, (int)e - 127);
}

int oracle_gemm_mx(int64_t M, int64_t N, int64_t K,
                   const void *A, int in_fmt, int a_major, int64_t lda, const uint8_t *sa, int64_t ldsa,
                   const void *B, int b_fmt, int b_major, int64_t ldb, const uint8_t *sb, int64_t ldsb,
                   const void *C, int c_fmt, int64_t ldc,
                   double alpha, double beta,
                   double *D, double *S, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || ldsa < (K + 31) / 32 || ldsb < (K + 31) / 32)
        return 1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int64_t i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < M; ++i) {
        double *acc = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));
        double *sab = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));
        for (int64_t k = 0; k < K; ++k) {
            double a = oracle_decode_e8m0(sa[i * ldsa + k / 32]) * a_at(A, in_fmt, a_major, lda, i, k);
            for (int64_t j = 0; j < N; ++j) {
                double p = a * (oracle_decode_e8m0(sb[j * ldsb + k / 32]) * b_at(B, b_fmt, b_major, ldb, k, j));
                acc[j] += p;
                sab[j] += fabs(p);
            }
        }
        for (int64_t j = 0; j < N; ++j) {
            double c = (beta != 0.0 && C) ? load(C, c_fmt, i * ldc + j) : 0.0;
            D[i * N + j] = alpha * acc[j] + beta * c;
            if (S)
                S[i * N + j] = fabs(alpha) * sab[j] + fabs(beta * c);
        }
        free(acc);
        free(sab);
    }
    return 0;
}

/* The block-scaled product at selected entries (rows[e], cols[e]) only. */
int oracle_gemm_mx_entries(int64_t M, int64_t N, int64_t K,
                           const void *A, int in_fmt, int a_major, int64_t lda, const uint8_t *sa, int64_t ldsa,
                           const void *B, int b_fmt, int b_major, int64_t ldb, const uint8_t *sb, int64_t ldsb,
                           const void *C, int c_fmt, int64_t ldc,
                           double alpha, double beta,
                           int64_t n_entries, const int64_t *rows, const int64_t *cols,
                           double *out_D, double *out_S, int nthreads)
{
    if (ldsa < (K + 31) / 32 || ldsb < (K + 31) / 32)
        return 1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int bad = 0;
    int64_t e;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
    for (e = 0; e < n_entries; ++e) {
        int64_t i = rows[e], j = cols[e];
        if (i < 0 || i >= M || j < 0 || j >= N) {
            bad |= 1;
            continue;
        }
        double acc = 0.0, sab = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = (oracle_decode_e8m0(sa[i * ldsa + k / 32]) * a_at(A, in_fmt, a_major, lda, i, k)) *
                       (oracle_decode_e8m0(sb[j * ldsb + k / 32]) * b_at(B, b_fmt, b_major, ldb, k, j));
            acc += p;
            sab += fabs(p);
        }
        double c = (beta != 0.0 && C) ? load(C, c_fmt, i * ldc + j) : 0.0;
        out_D[e] = alpha * acc + beta * c;
        if (out_S)
            out_S[e] = fabs(alpha) * sab + fabs(beta * c);
    }
    return bad;
}

/*
 * Block-scaled fp4 (NVFP4 / MXFP4, the fp4 members of the same block-scaled
 * MMA family): E2M1 elements, packed two to a byte (element 2i of a row in
 * the low nibble of byte i, 2i+1 in the high nibble), one scale per `block`
 * consecutive elements of K (16 with UE4M3 scales, 32 with E8M0):
 *
 *   D[i][j] = alpha * sum_k (sa(i, k/block) * A(i,k)) * (sb(j, k/block) * B(k,j)) + beta * C[i][j]
 *
 * A is M x K and B is stored N x K, both K-major, lda / ldb in elements
 * (even). E2M1 (OCP Microscaling): sign, 2 exponent bits (bias 1), 1
 * mantissa bit: 0, 0.5, 1, 1.5, 2, 3, 4, 6. UE4M3: the E4M3 encoding without
 * its sign bit, 2^(e-7) * (1 + m/8), e = 0 subnormal 2^-6 * m/8, 0x7F NaN.
 */
double oracle_decode_e2m1(uint8_t nibble)
{
    const int s = (nibble >> 3) & 1, e = (nibble >> 1) & 3, m = nibble & 1;
    const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

double oracle_decode_ue4m3(uint8_t code)
{
    const int e = (code >> 3) & 15, m = code & 7;
    if (code == 0x7F)
        return NAN;
    return e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
}

static double fp4_at(const uint8_t *X, int64_t ld, int64_t row, int64_t k)
{
    const uint8_t byte = X[(row * ld + k) / 2];
    return oracle_decode_e2m1((k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15));
}

static double fp4_scale(const uint8_t *s, int64_t lds, int64_t row, int64_t blk, int scale_e8m0)
{
    const uint8_t c = s[row * lds + blk];
    return scale_e8m0 ? oracle_decode_e8m0(c) : oracle_decode_ue4m3(c);
}

int oracle_gemm_fp4(int64_t M, int64_t N, int64_t K,
                    const uint8_t *A, int64_t lda, const uint8_t *sa, int64_t ldsa,
                    const uint8_t *B, int64_t ldb, const uint8_t *sb, int64_t ldsb,
                    int block, int scale_e8m0,
                    const void *C, int c_fmt, int64_t ldc,
                    double alpha, double beta,
                    double *D, double *S, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || (block != 16 && block != 32) || (lda & 1) || (ldb & 1) ||
        ldsa < (K + block - 1) / block || ldsb < (K + block - 1) / block)
        return 1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int64_t i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0, sab = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = (fp4_scale(sa, ldsa, i, k / block, scale_e8m0) * fp4_at(A, lda, i, k)) *
                           (fp4_scale(sb, ldsb, j, k / block, scale_e8m0) * fp4_at(B, ldb, j, k));
                acc += p;
                sab += fabs(p);
            }
            double c = (beta != 0.0 && C) ? load(C, c_fmt, i * ldc + j) : 0.0;
            D[i * N + j] = alpha * acc + beta * c;
            if (S)
                S[i * N + j] = fabs(alpha) * sab + fabs(beta * c);
        }
    }
    return 0;
}

/* The block-scaled fp4 product of oracle_gemm_fp4 at the listed entries only
 * (rows[e], cols[e]), for sampled checks of problems too large to evaluate
 * whole; the same sum over k in the same order. */
int oracle_gemm_fp4_entries(int64_t M, int64_t N, int64_t K,
                            const uint8_t *A, int64_t lda, const uint8_t *sa, int64_t ldsa,
                            const uint8_t *B, int64_t ldb, const uint8_t *sb, int64_t ldsb,
                            int block, int scale_e8m0,
                            const void *C, int c_fmt, int64_t ldc,
                            double alpha, double beta,
                            int64_t n_entries, const int64_t *rows, const int64_t *cols,
                            double *D, double *S, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || (block != 16 && block != 32) || (lda & 1) || (ldb & 1) ||
        ldsa < (K + block - 1) / block || ldsb < (K + block - 1) / block || n_entries < 0)
        return 1;
    for (int64_t e = 0; e < n_entries; ++e)
        if (rows[e] < 0 || rows[e] >= M || cols[e] < 0 || cols[e] >= N)
            return 1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int64_t e;
#pragma omp parallel for schedule(dynamic, 16)
    for (e = 0; e < n_entries; ++e) {
        const int64_t i = rows[e], j = cols[e];
        double acc = 0.0, sab = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = (fp4_scale(sa, ldsa, i, k / block, scale_e8m0) * fp4_at(A, lda, i, k)) *
                       (fp4_scale(sb, ldsb, j, k / block, scale_e8m0) * fp4_at(B, ldb, j, k));
            acc += p;
            sab += fabs(p);
        }
        double c = (beta != 0.0 && C) ? load(C, c_fmt, i * ldc + j) : 0.0;
        D[e] = alpha * acc + beta * c;
        if (S)
            S[e] = fabs(alpha) * sab + fabs(beta * c);
    }
    return 0;
}

/*
 * Round-to-nearest-even of x to a binary format with p significand bits
 * (hidden bit included), minimum normal exponent emin and maximum exponent
 * emax; subnormals are kept, overflow goes to infinity.
 */
static double round_rne(double x, int p, int emin, int emax)
{
    if (x == 0.0 || isnan(x) || isinf(x))
        return x;
    int e2;
    frexp(x, &e2);                 /* |x| in [2^(e2-1), 2^e2) */
    int lead = e2 - 1;
    if (lead < emin)
        lead = emin;               /* subnormal range: fixed quantum */
    int q = lead - (p - 1);        /* exponent of one unit in the last place */
    double r = nearbyint(ldexp(x, -q)) ;  /* default rounding mode: ties to even */
    double y = ldexp(r, q);
    double maxf = ldexp(ldexp(1.0, p) - 1.0, emax - (p - 1));
    if (fabs(y) > maxf)
        return x > 0 ? INFINITY : -INFINITY;
    return y;
}

double oracle_round(double x, int fmt)
{
    switch (fmt) {
    case ORC_F16: return round_rne(x, 11, -14, 15);
    case ORC_BF16: return round_rne(x, 8, -126, 127);
    default: return round_rne(x, 24, -126, 127);
    }
}

/* Round n doubles and write the output format's bit patterns. */
void oracle_round_bits(const double *x, int64_t n, int fmt, void *out)
{
    for (int64_t i = 0; i < n; ++i) {
        double y = oracle_round(x[i], fmt);
        if (fmt == ORC_F32) {
            float f = (float)y;    /* exact: y is already a binary32 value */
            uint32_t u;
            memcpy(&u, &f, sizeof u);
            ((uint32_t *)out)[i] = u;
        } else if (fmt == ORC_BF16) {
            float f = (float)y;    /* exact: bf16 values are binary32 values */
            uint32_t u;
            memcpy(&u, &f, sizeof u);
            ((uint16_t *)out)[i] = (uint16_t)(u >> 16);
        } else {
            /* encode binary16 from the exact value y */
            uint16_t s = signbit(y) ? 0x8000 : 0;
            double a = fabs(y);
            uint16_t h;
            if (isnan(y))
                h = 0x7e00;
            else if (isinf(a))
                h = 0x7c00;
            else if (a < ldexp(1.0, -14))
                h = (uint16_t)nearbyint(ldexp(a, 24));   /* exact multiple of 2^-24 */
            else {
                int e2;
                double m = frexp(a, &e2);                /* a = m * 2^e2, m in [0.5,1) */
                int e = e2 - 1 + 15;
                uint16_t f = (uint16_t)(ldexp(m, 11) - 1024.0);
                h = (uint16_t)((e << 10) | f);
            }
            ((uint16_t *)out)[i] = (uint16_t)(s | h);
        }
    }
}
