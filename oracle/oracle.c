/*
 * oracle.c -- plain, slow, obviously-correct CPU oracle for the dense matrix
 * product C = A.B in the three precisions of the study "Hand-Written PTX
 * Tensor-Core GEMM Kernels: A Multi-Precision Study on NVIDIA L4"
 * (Borowski & Osinski):
 *
 *   FP16 operands, products summed in FP64     (paper: FP16 family, FP32 acc.)
 *   INT8 operands, products summed in int64    (paper: INT8 family, INT32 acc.)
 *   packed INT4 operands, summed in int64      (paper: INT4 family, Listing 1
 *                                               addressing, .s32.s4.s4.s32)
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker of the GPU
 * library.  It shares no code, header, table or helper with the CUDA path and
 * must never be linked into it.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.
 *
 * What is computed (paper section I-A "Tensor Cores, WMMA, and PTX mma.sync":
 * D = A B + C, here with C = 0 and no scaling, as section VI "Scope" states):
 *
 *   C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]      in ascending k.
 *
 * Storage (the library boundary's layouts):
 *   A           row-major M x K, element (i,k) at A[i*lda + k]
 *   FP16 B      row-major K x N, element (k,j) at B[k*ldb + j]
 *   INT8/INT4 B column-major K x N ("non-transposed" B of the paper's .row.col
 *               MMA, section IV-D), element (k,j) at B[j*ldb + k]
 *   packed s4   two's-complement nibbles, element 2t of a row in bits 0..3 of
 *               byte t, element 2t+1 in bits 4..7; ld counted in elements
 *               (nibbles), so row r starts at byte r*ld/2 (Listing 1 address
 *               A_b[row*(K/2) + k/2]).
 *
 * Nothing here is blocked, fused or reordered: each output element is one
 * loop over k.  Threads only split the rows of C.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------------
 * IEEE 754-2008 binary16 decoding, from the format's definition:
 *   sign s (bit 15), biased exponent e (bits 14..10, bias 15), fraction f
 *   (bits 9..0).  e == 0: subnormal (-1)^s * f * 2^-24.  0 < e < 31: normal
 *   (-1)^s * (1024 + f) * 2^(e-25).  e == 31: infinity (f == 0) or NaN.
 * Every binary16 value is exact in binary64.
 * ------------------------------------------------------------------------- */
double oracle_f16_to_f64(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e < 31)
        v = ldexp((double)(1024 + f), e - 25);
    else
        v = (f == 0) ? INFINITY : NAN;
    return s ? -v : v;
}

/* Signed value of element k of a packed s4 row (low nibble = even k). */
int oracle_s4_get(const uint8_t *row, int64_t k)
{
    uint8_t byte = row[k >> 1];
    int nib = (k & 1) ? (byte >> 4) : (byte & 0x0f);
    return nib >= 8 ? nib - 16 : nib;
}

/* Store a signed value in [-8, 7] as element k of a packed s4 row. */
void oracle_s4_set(uint8_t *row, int64_t k, int v)
{
    uint8_t nib = (uint8_t)(v & 0x0f);
    uint8_t *b = &row[k >> 1];
    if (k & 1)
        *b = (uint8_t)((*b & 0x0f) | (nib << 4));
    else
        *b = (uint8_t)((*b & 0xf0) | nib);
}

/* Unpack `rows` packed rows (ld nibbles each) into int8 values (ldo each). */
void oracle_unpack_s4(int64_t rows, int64_t cols, const uint8_t *src, int64_t ld,
                      int8_t *dst, int64_t ldo)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            dst[r * ldo + c] = (int8_t)oracle_s4_get(src + r * (ld / 2), c);
}

/* Pack int8 values in [-8, 7] into s4 rows of `ld` nibbles (bytes zeroed first). */
void oracle_pack_s4(int64_t rows, int64_t cols, const int8_t *src, int64_t lds,
                    uint8_t *dst, int64_t ld)
{
    memset(dst, 0, (size_t)(rows * (ld / 2)));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            oracle_s4_set(dst + r * (ld / 2), c, src[r * lds + c]);
}

/* ---------------------------------------------------------------------------
 * Element kernels: one output element, one loop over k.
 * ------------------------------------------------------------------------- */
static void dot_f16(int64_t K, const uint16_t *A, int64_t lda, const uint16_t *B,
                    int64_t ldb, int64_t i, int64_t j, double *c, double *s)
{
    double acc = 0.0, sabs = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        /* an 11-bit by 11-bit significand product is exact in binary64 */
        double p = oracle_f16_to_f64(A[i * lda + k]) * oracle_f16_to_f64(B[k * ldb + j]);
        acc += p;
        sabs += fabs(p);
    }
    *c = acc;
    *s = sabs;
}

static int64_t dot_s8(int64_t K, const int8_t *A, int64_t lda, const int8_t *B,
                      int64_t ldb, int64_t i, int64_t j)
{
    int64_t acc = 0;
    for (int64_t k = 0; k < K; ++k)
        acc += (int64_t)A[i * lda + k] * (int64_t)B[j * ldb + k];
    return acc;
}

static int64_t dot_s4(int64_t K, const uint8_t *A, int64_t lda, const uint8_t *B,
                      int64_t ldb, int64_t i, int64_t j)
{
    const uint8_t *arow = A + i * (lda / 2);
    const uint8_t *bcol = B + j * (ldb / 2);
    int64_t acc = 0;
    for (int64_t k = 0; k < K; ++k)
        acc += (int64_t)oracle_s4_get(arow, k) * (int64_t)oracle_s4_get(bcol, k);
    return acc;
}

/* ---------------------------------------------------------------------------
 * Row-parallel driver.
 * ------------------------------------------------------------------------- */
enum { P_F16 = 0, P_S8 = 1, P_S4 = 2 };

typedef struct {
    int prec;
    int64_t M, N, K;
    const void *A, *B;
    int64_t lda, ldb, ldc;
    void *C;      /* double (f16) or int64 (s8/s4) */
    double *S;    /* f16 only: sum_k |A[i][k] B[k][j]|, may be NULL */
    int64_t r0, r1;
} job_t;

static void *run_rows(void *arg)
{
    job_t *jb = (job_t *)arg;
    for (int64_t i = jb->r0; i < jb->r1; ++i) {
        for (int64_t j = 0; j < jb->N; ++j) {
            int64_t o = i * jb->ldc + j;
            if (jb->prec == P_F16) {
                double c, s;
                dot_f16(jb->K, (const uint16_t *)jb->A, jb->lda,
                        (const uint16_t *)jb->B, jb->ldb, i, j, &c, &s);
                ((double *)jb->C)[o] = c;
                if (jb->S) jb->S[o] = s;
            } else if (jb->prec == P_S8) {
                ((int64_t *)jb->C)[o] = dot_s8(jb->K, (const int8_t *)jb->A, jb->lda,
                                               (const int8_t *)jb->B, jb->ldb, i, j);
            } else {
                ((int64_t *)jb->C)[o] = dot_s4(jb->K, (const uint8_t *)jb->A, jb->lda,
                                               (const uint8_t *)jb->B, jb->ldb, i, j);
            }
        }
    }
    return NULL;
}

static void run_parallel(job_t base, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > base.M) nthreads = (int)(base.M > 0 ? base.M : 1);
    job_t jobs[256];
    pthread_t tid[256];
    int created[256];
    int64_t per = (base.M + nthreads - 1) / nthreads;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].r0 = t * per;
        jobs[t].r1 = (t + 1) * per < base.M ? (t + 1) * per : base.M;
        if (jobs[t].r0 >= jobs[t].r1) break;
        created[t] = nthreads > 1 && pthread_create(&tid[t], NULL, run_rows, &jobs[t]) == 0;
        if (!created[t])
            run_rows(&jobs[t]);
        started = t + 1;
    }
    for (int t = 0; t < started; ++t)
        if (created[t]) pthread_join(tid[t], NULL);
}

/* C[i][j] (double) and S[i][j] = sum_k |A_ik B_kj| for FP16 A (M x K, row-major)
 * and FP16 B (K x N, row-major).  S may be NULL. */
void oracle_gemm_f16(int64_t M, int64_t N, int64_t K, const uint16_t *A, int64_t lda,
                     const uint16_t *B, int64_t ldb, double *C, double *S, int64_t ldc,
                     int nthreads)
{
    job_t jb = {P_F16, M, N, K, A, B, lda, ldb, ldc, C, S, 0, 0};
    run_parallel(jb, nthreads);
}

/* Exact int64 C for INT8 A (row-major) and INT8 B (column-major). */
void oracle_gemm_s8(int64_t M, int64_t N, int64_t K, const int8_t *A, int64_t lda,
                    const int8_t *B, int64_t ldb, int64_t *C, int64_t ldc, int nthreads)
{
    job_t jb = {P_S8, M, N, K, A, B, lda, ldb, ldc, C, NULL, 0, 0};
    run_parallel(jb, nthreads);
}

/* Exact int64 C for packed INT4 A (row-major) and B (column-major); lda, ldb in
 * nibbles (even). */
void oracle_gemm_s4(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda,
                    const uint8_t *B, int64_t ldb, int64_t *C, int64_t ldc, int nthreads)
{
    job_t jb = {P_S4, M, N, K, A, B, lda, ldb, ldc, C, NULL, 0, 0};
    run_parallel(jb, nthreads);
}

/* ---------------------------------------------------------------------------
 * Sampled outputs: the same element loops at listed coordinates (i[p], j[p]),
 * for checking full-size results one element at a time.
 * ------------------------------------------------------------------------- */
void oracle_gemm_f16_at(int64_t K, const uint16_t *A, int64_t lda, const uint16_t *B,
                        int64_t ldb, int64_t npts, const int64_t *ii, const int64_t *jj,
                        double *C, double *S)
{
    for (int64_t p = 0; p < npts; ++p)
        dot_f16(K, A, lda, B, ldb, ii[p], jj[p], &C[p], &S[p]);
}

void oracle_gemm_s8_at(int64_t K, const int8_t *A, int64_t lda, const int8_t *B,
                       int64_t ldb, int64_t npts, const int64_t *ii, const int64_t *jj,
                       int64_t *C)
{
    for (int64_t p = 0; p < npts; ++p)
        C[p] = dot_s8(K, A, lda, B, ldb, ii[p], jj[p]);
}

void oracle_gemm_s4_at(int64_t K, const uint8_t *A, int64_t lda, const uint8_t *B,
                       int64_t ldb, int64_t npts, const int64_t *ii, const int64_t *jj,
                       int64_t *C)
{
    for (int64_t p = 0; p < npts; ++p)
        C[p] = dot_s4(K, A, lda, B, ldb, ii[p], jj[p]);
}

/* ---------------------------------------------------------------------------
 * Scaled integer GEMM (dequantisation epilogue).  This is the form the INT8 /
 * INT4 products take in quantised inference (paper section V), which the
 * paper's own kernels leave out (section VI): per-row scales of A, per-column
 * scales of B.  Definition, per element, in IEEE binary32 with
 * round-to-nearest-even at every step and no fused multiply-add:
 *     v = acc wrapped to int32;  t = (float)v;  t = t * sa[i];  t = t * sb[j]
 * then rounded to nearest-even into the output type.
 * ------------------------------------------------------------------------- */

/* binary32 -> bfloat16 (the top 16 bits of binary32), round to nearest,
 * ties to even; NaN stays NaN. */
uint16_t oracle_f32_to_bf16(float x)
{
    uint32_t b;
    memcpy(&b, &x, 4);
    if ((b & 0x7f800000u) == 0x7f800000u && (b & 0x007fffffu))
        return (uint16_t)((b >> 16) | 0x0040u);          /* quiet NaN */
    uint32_t keep = b >> 16, rest = b & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1;                                        /* may carry into the exponent: correct */
    return (uint16_t)keep;
}

/* binary32 -> binary16, round to nearest, ties to even, from the binary16
 * definition: normal values (1 + f/1024) 2^e for -14 <= e <= 15, subnormals
 * f 2^-24, overflow to infinity. */
uint16_t oracle_f32_to_f16(float x)
{
    double v = (double)x;
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v)) return (uint16_t)(sign | 0x7e00u);
    if (isinf(v)) return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {                            /* subnormal range, quantum 2^-24 */
        double q = nearbyint(a * ldexp(1.0, 24));         /* ties to even (default mode) */
        return (uint16_t)(sign | (uint16_t)q);            /* q == 1024 is the smallest normal */
    }
    int e;
    frexp(a, &e);                                         /* a = m 2^e, 0.5 <= m < 1 */
    e -= 1;                                               /* a = (1 + f) 2^e */
    double q = nearbyint(ldexp(a, 10 - e));               /* 1024 <= q <= 2048 */
    if (q >= 2048.0) { q = 1024.0; e += 1; }
    if (e > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(q - 1024.0));
}

/* out_type 0: binary32 bit patterns (uint32); 1: bfloat16; 2: binary16
 * (uint16).  acc holds exact sums (int64), M x N with pitch lda; sa / sb may
 * be NULL (all ones). */
void oracle_dequant(int64_t M, int64_t N, const int64_t *acc, int64_t lda, const float *sa,
                    const float *sb, int out_type, void *out, int64_t ldo)
{
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            int32_t v = (int32_t)(uint32_t)(uint64_t)acc[i * lda + j];
            volatile float t = (float)v;
            t = t * (sa ? sa[i] : 1.0f);
            t = t * (sb ? sb[j] : 1.0f);
            if (out_type == 0) {
                uint32_t b;
                float tf = t;
                memcpy(&b, &tf, 4);
                ((uint32_t *)out)[i * ldo + j] = b;
            } else if (out_type == 1) {
                ((uint16_t *)out)[i * ldo + j] = oracle_f32_to_bf16(t);
            } else {
                ((uint16_t *)out)[i * ldo + j] = oracle_f32_to_f16(t);
            }
        }
    }
}

/* Two's-complement wrap of an exact sum to 32 bits (reading adopted where the
 * paper is silent on INT32 overflow: .s32 accumulation without saturation). */
int32_t oracle_wrap_s32(int64_t v)
{
    return (int32_t)(uint32_t)(uint64_t)v;
}
