/*
 * CPU oracle for the dense matrix product  D = alpha * op(A) @ op(B) + beta * C.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load, link or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant with the
 * CUDA path; the two meet only through the seeded inputs they are handed.
 *
 * What it computes (the plain definition, written out):
 *
 *   TVM TIRx "gemm" page, opening paragraph and the "What it accepts" table
 *   (rows "dtype" and "alpha / beta"); the TIRx gemm guide, section 一
 *   ("语义定义"); Phobos "@tensorcore" page, example gemm_fp16tc_fp32acc.ph
 *   (epilogue  alpha * acc + beta * c_old):
 *
 *     D[i][j] = alpha * sum_{k=0}^{K-1} Ahat[i][k] * Bhat[k][j]  +  beta * C[i][j]
 *
 *   Ahat = A   (transA = 0, A stored M x K)  or  A^T (transA = 1, stored K x M)
 *   Bhat = B   (transB = 0, B stored K x N)  or  B^T (transB = 1, stored N x K)
 *
 *   The transpose flags only name the logical orientation; the operation is
 *   normalised to A = [M,K], B = [K,N], C = D = [M,N] (TIRx gemm guide,
 *   section 二, "维度一致性").  Storage is row-major; a leading dimension is
 *   the row stride in elements (the demonstration program on the TIRx
 *   "gemm" page indexes A_g[m, k], B_g[k, n], D_g[m, n]).
 *
 *   beta == 0 means "D zero-initialised": C is never read, so a NaN in C
 *   cannot reach D ("What it accepts" table, alpha / beta row; the
 *   "How inputs change the algorithm" table, beta row).
 *
 * Operand types: fp16 and bf16 (the TIRx "gemm" page, "What it accepts",
 * dtype row), and the 8-bit floating-point types E4M3 and E5M2 that the
 * TIRx gemm guide lists among the asynchronous (tcgen05) path's precisions
 * (section 七, "精度与指令族").  The pages do not define the 8-bit formats;
 * they are the OCP 8-bit floating-point formats the PTX ISA calls .e4m3 and
 * .e5m2 (decoders below).  A and B always have the same type.
 *
 * Precision: every fp16 / bf16 / fp8 / fp32 element is decoded exactly to a
 * double by the decoders below, products and sums are taken in double
 * (binary64), in increasing k order, one output element at a time.  The
 * sum of |products| is kept alongside, so the caller can form the
 * per-element error bound  |alpha| * sum|a*b| + |beta| * |c|.
 *
 * 4-bit operands: E2M1, the OCP 4-bit floating-point format (the guide lists
 * fp4 among gemm_async's precisions, same section), stored packed, two
 * elements per byte: element e of a row-major array (e = row * ld + col, ld
 * in elements) is the low nibble of byte e / 2 when e is even, the high
 * nibble when it is odd.  E2M1 is used block-scaled (below).
 *
 * Block-scaled 8-bit and 4-bit operands (oracle_gemm_mx*): the TIRx gemm guide lists
 * block scaling with separate A and B scale factors ("SFA/SFB") among the
 * asynchronous path's modes (section 七) without defining it.  The reading
 * taken is the OCP Microscaling (MX) one: each run of 32 consecutive K
 * elements of a row of Ahat shares one scale SFA[i][k / 32], and of a column
 * of Bhat one scale SFB[j][k / 32]; a scale is a UE8M0 byte e standing for
 * 2^(e - 127) (e = 255: NaN).  The definition becomes
 *
 *     D[i][j] = alpha * sum_k (SFA[i][k/32] * Ahat[i][k]) * (SFB[j][k/32] * Bhat[k][j])
 *               + beta * C[i][j]
 *
 * with SFA stored [M, ceil(K/32)] and SFB stored [N, ceil(K/32)], row-major
 * with row strides ld_sfa / ld_sfb, whatever transA / transB say.
 *
 * Build: a plain C99 compiler, -O2, -ffp-contract=off (no fused
 * multiply-add, no fast-math), so that x86-64 and aarch64 give the same
 * bits.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1, ORACLE_F32 = 2, ORACLE_E4M3 = 3, ORACLE_E5M2 = 4, ORACLE_E2M1 = 5 };

/* ---- exact element decoders -------------------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(1024 + f), e - 25);   /* 1.f * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE 754 binary32 (8 exponent bits, bias
 * 127, 7 fraction bits). */
double oracle_decode_bf16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);              /* subnormal: f * 2^-126 * 2^-7 */
    else if (e == 255)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(128 + f), e - 134);   /* 1.f * 2^(e-127) */
    return sign ? -v : v;
}

/* E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; no
 * infinities; S.1111.111 is NaN, so the largest finite value is
 * 1.75 * 2^8 = 448. */
double oracle_decode_e4m3(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xf;
    int f = b & 0x7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);                /* subnormal: f * 2^-6 * 2^-3 */
    else
        v = ldexp((double)(8 + f), e - 10);      /* 1.f * 2^(e-7) */
    return sign ? -v : v;
}

/* E5M2: 1 sign bit, 5 exponent bits (bias 15), 2 fraction bits, with
 * binary16's infinities and NaNs (exponent 31). */
double oracle_decode_e5m2(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 2) & 0x1f;
    int f = b & 0x3;
    double v;
    if (e == 0)
        v = ldexp((double)f, -16);               /* subnormal: f * 2^-14 * 2^-2 */
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(4 + f), e - 17);      /* 1.f * 2^(e-15) */
    return sign ? -v : v;
}

/* E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 fraction bit; no
 * infinities or NaNs, so the magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double oracle_decode_e2m1(uint8_t c)
{
    const int sign = (c >> 3) & 1, e = (c >> 1) & 3, f = c & 1;
    double v;
    if (e == 0)
        v = 0.5 * f;                              /* subnormal: 0.f * 2^0 */
    else
        v = ldexp((double)(2 + f), e - 2);       /* 1.f * 2^(e-1) */
    return sign ? -v : v;
}

/* UE8M0, the MX shared scale: 8 exponent bits (bias 127), no sign and no
 * fraction, so the value is 2^(e - 127); the all-ones pattern is NaN. */
double oracle_decode_ue8m0(uint8_t e)
{
    return e == 0xFFu ? NAN : ldexp(1.0, (int)e - 127);
}

/* K elements per MX scale block */
#define MX_BLOCK 32

/* binary32 -> binary64 is exact. */
static double decode_f32(const void* p)
{
    float x;
    memcpy(&x, p, sizeof x);
    return (double)x;
}

/* The operand decoders above are memoised in tables indexed by the bit
 * pattern, filled once by calling them on every pattern (pthread_once: the
 * tests call the oracle from several threads at a time). */
static double g_f16_table[65536];
static double g_bf16_table[65536];
static double g_e4m3_table[256];
static double g_e5m2_table[256];
static double g_e2m1_table[16];
static pthread_once_t g_tables_once = PTHREAD_ONCE_INIT;

static void fill_tables(void)
{
    for (uint32_t h = 0; h < 65536u; ++h) {
        g_f16_table[h] = oracle_decode_f16((uint16_t)h);
        g_bf16_table[h] = oracle_decode_bf16((uint16_t)h);
    }
    for (uint32_t b = 0; b < 256u; ++b) {
        g_e4m3_table[b] = oracle_decode_e4m3((uint8_t)b);
        g_e5m2_table[b] = oracle_decode_e5m2((uint8_t)b);
    }
    for (uint32_t c = 0; c < 16u; ++c) g_e2m1_table[c] = oracle_decode_e2m1((uint8_t)c);
}

static const double* table_for(int dtype)
{
    pthread_once(&g_tables_once, fill_tables);
    switch (dtype) {
    case ORACLE_F16: return g_f16_table;
    case ORACLE_BF16: return g_bf16_table;
    case ORACLE_E4M3: return g_e4m3_table;
    case ORACLE_E2M1: return g_e2m1_table;
    default: return g_e5m2_table;
    }
}

/* ---- operand access ------------------------------------------------------ */

typedef struct {
    const void* A;
    const void* B;
    const void* C;
    int64_t M, N, K, lda, ldb, ldc;
    int transA, transB;
    double alpha, beta;
    const double* in_table;   /* decoder for A and B */
    int in_bytes;             /* bytes per A / B element: 2 (fp16, bf16), 1 (fp8), 0 (packed fp4) */
    int c_dtype;
    const uint8_t* SFA;       /* MX scales of Ahat's rows, or NULL (no block scaling) */
    const uint8_t* SFB;       /* MX scales of Bhat's columns */
    int64_t ld_sfa, ld_sfb;
} problem_t;

/* The bit pattern of operand element `idx` (elements of in_bytes bytes, or
 * nibbles when in_bytes is 0: even elements in the low nibble). */
static unsigned operand_bits(const problem_t* p, const void* X, int64_t idx)
{
    if (p->in_bytes == 0) {
        const uint8_t b = ((const uint8_t*)X)[idx / 2];
        return (idx % 2 == 0) ? (b & 0xFu) : (b >> 4);
    }
    return p->in_bytes == 1 ? ((const uint8_t*)X)[idx] : ((const uint16_t*)X)[idx];
}

/* Ahat[i][k], times its block's scale when the operands are block-scaled */
static double a_hat(const problem_t* p, int64_t i, int64_t k)
{
    int64_t idx = p->transA ? k * p->lda + i : i * p->lda + k;
    double v = p->in_table[operand_bits(p, p->A, idx)];
    if (p->SFA != NULL) v *= oracle_decode_ue8m0(p->SFA[i * p->ld_sfa + k / MX_BLOCK]);
    return v;
}

/* Bhat[k][j], likewise */
static double b_hat(const problem_t* p, int64_t k, int64_t j)
{
    int64_t idx = p->transB ? j * p->ldb + k : k * p->ldb + j;
    double v = p->in_table[operand_bits(p, p->B, idx)];
    if (p->SFB != NULL) v *= oracle_decode_ue8m0(p->SFB[j * p->ld_sfb + k / MX_BLOCK]);
    return v;
}

static double c_elem(const problem_t* p, int64_t i, int64_t j)
{
    int64_t off = i * p->ldc + j;
    if (p->c_dtype == ORACLE_F32)
        return decode_f32((const char*)p->C + 4 * off);
    const uint16_t bits = ((const uint16_t*)p->C)[off];
    return p->c_dtype == ORACLE_F16 ? oracle_decode_f16(bits) : oracle_decode_bf16(bits);
}

/* One output element by the definition; *bound gets
 * |alpha| * sum_k |Ahat[i][k] * Bhat[k][j]| + |beta| * |C[i][j]|. */
static double one_element(const problem_t* p, int64_t i, int64_t j, double* bound)
{
    double s = 0.0, sa = 0.0;
    for (int64_t k = 0; k < p->K; ++k) {
        double prod = a_hat(p, i, k) * b_hat(p, k, j);
        s += prod;
        sa += fabs(prod);
    }
    double d = p->alpha * s;
    double b = fabs(p->alpha) * sa;
    if (p->beta != 0.0) {             /* beta == 0: C is not read */
        double c = c_elem(p, i, j);
        d += p->beta * c;
        b += fabs(p->beta) * fabs(c);
    }
    *bound = b;
    return d;
}

static int setup(problem_t* p, const void* A, const void* B, const void* C,
                 int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                 int transA, int transB, double alpha, double beta,
                 int in_dtype, int c_dtype)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (in_dtype != ORACLE_F16 && in_dtype != ORACLE_BF16 && in_dtype != ORACLE_E4M3 &&
        in_dtype != ORACLE_E5M2 && in_dtype != ORACLE_E2M1)
        return -1;
    if (c_dtype != ORACLE_F16 && c_dtype != ORACLE_BF16 && c_dtype != ORACLE_F32) return -1;
    if ((M > 0 && K > 0 && A == NULL) || (K > 0 && N > 0 && B == NULL)) return -1;
    if (beta != 0.0 && M > 0 && N > 0 && C == NULL) return -1;
    /* the stored row length must fit in the leading dimension */
    if (K > 0 && lda < (transA ? M : K)) return -1;
    if (K > 0 && ldb < (transB ? K : N)) return -1;
    if (beta != 0.0 && ldc < N) return -1;
    p->A = A;
    p->B = B;
    p->C = C;
    p->M = M; p->N = N; p->K = K;
    p->lda = lda; p->ldb = ldb; p->ldc = ldc;
    p->transA = transA != 0; p->transB = transB != 0;
    p->alpha = alpha; p->beta = beta;
    p->in_table = table_for(in_dtype);
    p->in_bytes = (in_dtype == ORACLE_E4M3 || in_dtype == ORACLE_E5M2) ? 1 : in_dtype == ORACLE_E2M1 ? 0 : 2;
    p->c_dtype = c_dtype;
    p->SFA = NULL;
    p->SFB = NULL;
    p->ld_sfa = p->ld_sfb = 0;
    return 0;
}

/* Block scales on top of setup(): 8-bit operands only, both scale arrays
 * present whenever they are read, rows of ceil(K/32) scales. */
static int setup_mx(problem_t* p, const void* SFA, const void* SFB, int64_t ld_sfa, int64_t ld_sfb)
{
    const int64_t kb = (p->K + MX_BLOCK - 1) / MX_BLOCK;
    if (p->in_bytes > 1) return -1;
    if ((p->M > 0 && p->K > 0 && SFA == NULL) || (p->N > 0 && p->K > 0 && SFB == NULL)) return -1;
    if (p->K > 0 && (ld_sfa < kb || ld_sfb < kb)) return -1;
    p->SFA = (const uint8_t*)SFA;
    p->SFB = (const uint8_t*)SFB;
    p->ld_sfa = ld_sfa;
    p->ld_sfb = ld_sfb;
    return 0;
}

/* Full rows [row_begin, row_end) of D into D and bound (row stride ldo). */
static int rows_of(const problem_t* p, double* D, double* bound, int64_t ldo,
                   int64_t row_begin, int64_t row_end)
{
    if (row_begin < 0 || row_end > p->M || row_begin > row_end || ldo < p->N) return -1;
    for (int64_t i = row_begin; i < row_end; ++i)
        for (int64_t j = 0; j < p->N; ++j)
            D[i * ldo + j] = one_element(p, i, j, &bound[i * ldo + j]);
    return 0;
}

/* The listed elements (rows[e], cols[e]), e < count, into D[e], bound[e]. */
static int entries_of(const problem_t* p, double* D, double* bound,
                      const int64_t* rows, const int64_t* cols, int64_t count)
{
    for (int64_t e = 0; e < count; ++e)
        if (rows[e] < 0 || rows[e] >= p->M || cols[e] < 0 || cols[e] >= p->N) return -1;
    for (int64_t e = 0; e < count; ++e)
        D[e] = one_element(p, rows[e], cols[e], &bound[e]);
    return 0;
}

/* Full rows [row_begin, row_end) of D.  D and bound are dense [M, N]
 * double arrays with row stride ldo; only the requested rows are written.
 * Returns 0, or -1 on a malformed argument. */
int oracle_gemm(double* D, double* bound, int64_t ldo,
                const void* A, const void* B, const void* C,
                int64_t M, int64_t N, int64_t K,
                int64_t lda, int64_t ldb, int64_t ldc,
                int transA, int transB, double alpha, double beta,
                int in_dtype, int c_dtype,
                int64_t row_begin, int64_t row_end)
{
    problem_t p;
    if (setup(&p, A, B, C, M, N, K, lda, ldb, ldc, transA, transB, alpha, beta,
              in_dtype, c_dtype) != 0)
        return -1;
    return rows_of(&p, D, bound, ldo, row_begin, row_end);
}

/* The listed elements (rows[e], cols[e]) only, e < count: D[e], bound[e]. */
int oracle_gemm_entries(double* D, double* bound,
                        const int64_t* rows, const int64_t* cols, int64_t count,
                        const void* A, const void* B, const void* C,
                        int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldc,
                        int transA, int transB, double alpha, double beta,
                        int in_dtype, int c_dtype)
{
    problem_t p;
    if (setup(&p, A, B, C, M, N, K, lda, ldb, ldc, transA, transB, alpha, beta,
              in_dtype, c_dtype) != 0)
        return -1;
    return entries_of(&p, D, bound, rows, cols, count);
}

/* oracle_gemm with MX block-scaled 8-bit operands (scales SFA [M, ceil(K/32)]
 * and SFB [N, ceil(K/32)], UE8M0 bytes). */
int oracle_gemm_mx(double* D, double* bound, int64_t ldo,
                   const void* A, const void* B, const void* C,
                   const void* SFA, const void* SFB,
                   int64_t M, int64_t N, int64_t K,
                   int64_t lda, int64_t ldb, int64_t ldc, int64_t ld_sfa, int64_t ld_sfb,
                   int transA, int transB, double alpha, double beta,
                   int in_dtype, int c_dtype,
                   int64_t row_begin, int64_t row_end)
{
    problem_t p;
    if (setup(&p, A, B, C, M, N, K, lda, ldb, ldc, transA, transB, alpha, beta,
              in_dtype, c_dtype) != 0 ||
        setup_mx(&p, SFA, SFB, ld_sfa, ld_sfb) != 0)
        return -1;
    return rows_of(&p, D, bound, ldo, row_begin, row_end);
}

/* oracle_gemm_entries with MX block-scaled 8-bit operands. */
int oracle_gemm_mx_entries(double* D, double* bound,
                           const int64_t* rows, const int64_t* cols, int64_t count,
                           const void* A, const void* B, const void* C,
                           const void* SFA, const void* SFB,
                           int64_t M, int64_t N, int64_t K,
                           int64_t lda, int64_t ldb, int64_t ldc, int64_t ld_sfa, int64_t ld_sfb,
                           int transA, int transB, double alpha, double beta,
                           int in_dtype, int c_dtype)
{
    problem_t p;
    if (setup(&p, A, B, C, M, N, K, lda, ldb, ldc, transA, transB, alpha, beta,
              in_dtype, c_dtype) != 0 ||
        setup_mx(&p, SFA, SFB, ld_sfa, ld_sfb) != 0)
        return -1;
    return entries_of(&p, D, bound, rows, cols, count);
}
