/*
 * gemm_oracle.c -- the CPU oracle for the pipelined GEMM library.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant table with the
 * CUDA sources of the library.
 *
 * What it computes is the plain definition of the two products the pipelined
 * kernels reach exactly (up to rounding order):
 *
 *   s32 NN  (Croqtile tutorial ch.6, "使用 swap 的双缓冲" listing):
 *       out[m,n] = (int32)( sum_{k<K} (int64)lhs[m,k] * (int64)rhs[k,n] )  [mod 2^32]
 *     with lhs [M,K] and rhs [K,N] row-major; the kernel there accumulates
 *     with "+=" into an output that it never initialises, which is read here
 *     as a zero start.  The int64 sum is truncated to its low 32 bits (two's
 *     complement wrap), which equals the wrapping 32-bit multiply-add result.
 *
 *   f16 NT  (Croqtile tutorial ch.6, "带 event 的 1P1C 内核" listing):
 *       ref[m,n] = sum_{k<K} (double)lhs[m,k] * (double)rhs[n,k]
 *     with lhs [M,K] and rhs [N,K] row-major (the listing declares rhs as
 *     [N,K] and multiplies with mma.row.row, i.e. C = A * B^T).  Every
 *     f16 x f16 product is exact in binary64 (11+11 significant bits), so the
 *     only rounding is that of the binary64 running sum.
 *
 * Binary16 is decoded and encoded here from the IEEE 754 definition of the
 * format (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits,
 * subnormal quantum 2^-24), with round-to-nearest-even taken directly from
 * the binary64 value (no intermediate binary32 rounding).
 *
 * Loop order is the textbook one (row m, column n, then the K sum in order
 * k = 0..K-1).  Rows are split over plain pthreads only to make the large
 * cases finish; each output element is still one in-order sum.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* binary16 <-> binary64 from the IEEE 754 format definition                */
/* ------------------------------------------------------------------------ */

double oracle_f16_to_f64(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1F;
    const int frac = h & 0x3FF;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);               /* subnormal or zero   */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;                  /* inf or NaN          */
    } else {
        v = ldexp((double)(1024 + frac), expo - 25); /* (1.f) * 2^(e-15)   */
    }
    return sign ? -v : v;
}

/* Encode a value that is already exactly representable in binary16 (or is
 * >= 2^16 in magnitude, which is encoded as infinity). */
static uint16_t encode_exact(int sign, double a) {
    uint16_t s = (uint16_t)(sign ? 0x8000 : 0);
    if (a >= 65536.0) return s | 0x7C00;
    if (a == 0.0) return s;
    if (a < ldexp(1.0, -14)) {                       /* subnormal           */
        return s | (uint16_t)(a / ldexp(1.0, -24));
    }
    int e;
    frexp(a, &e);                                   /* a in [2^(e-1), 2^e) */
    const int E = e - 1;                            /* 2^E <= a < 2^(E+1)  */
    const int mant = (int)(a / ldexp(1.0, E - 10)) - 1024;
    return s | (uint16_t)(((E + 15) << 10) | mant);
}

uint16_t oracle_f64_to_f16(double x) {
    if (isnan(x)) return 0x7E00;
    const int sign = signbit(x) ? 1 : 0;
    const double a = fabs(x);
    if (isinf(a)) return (uint16_t)((sign ? 0x8000 : 0) | 0x7C00);
    if (a == 0.0) return (uint16_t)(sign ? 0x8000 : 0);
    int e;
    frexp(a, &e);
    int E = e - 1;                                  /* 2^E <= a < 2^(E+1)  */
    if (E < -14) E = -14;                           /* subnormal range     */
    /* The spacing of binary16 values near a is q = 2^(E-10); round a/q to the
     * nearest integer, ties to the even integer.  a/q is exact (q is a power
     * of two and a/q stays far from the binary64 subnormal range). */
    const double q = ldexp(1.0, E - 10);
    const double t = a / q;
    double n = floor(t);
    const double rem = t - n;
    if (rem > 0.5 || (rem == 0.5 && fmod(n, 2.0) == 1.0)) n += 1.0;
    return encode_exact(sign, n * q);
}

void oracle_f16_to_f64_array(const uint16_t* h, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f64(h[i]);
}

void oracle_f64_to_f16_array(const double* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_f16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* row-parallel driver                                                      */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t row_begin, row_end;
    void (*fn)(void* ctx, int64_t row);
    void* ctx;
} row_job;

static void* run_rows(void* p) {
    row_job* j = (row_job*)p;
    for (int64_t r = j->row_begin; r < j->row_end; ++r) j->fn(j->ctx, r);
    return NULL;
}

static void for_rows(int64_t rows, int nthreads, void (*fn)(void*, int64_t), void* ctx) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if ((int64_t)nthreads > rows) nthreads = rows > 0 ? (int)rows : 1;
    pthread_t tid[512];
    int joined[512];
    row_job jobs[512];
    const int64_t per = (rows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        const int64_t b = (int64_t)t * per;
        const int64_t e = b + per < rows ? b + per : rows;
        jobs[t].row_begin = b < rows ? b : rows;
        jobs[t].row_end = e;
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        joined[t] = 0;
    }
    /* threads 1..n-1 run concurrently; a thread that cannot start runs inline */
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, run_rows, &jobs[t]) == 0) joined[t] = 1;
        else run_rows(&jobs[t]);
    }
    run_rows(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (joined[t]) pthread_join(tid[t], NULL);
}

/* ------------------------------------------------------------------------ */
/* s32 NN: out[M,N] = lhs[M,K] . rhs[K,N], int64 sum, wrapped to int32       */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t M, N, K;
    const int32_t* lhs;
    const int32_t* rhs;
    int32_t* out;
} s32_ctx;

static void s32_row(void* p, int64_t m) {
    const s32_ctx* c = (const s32_ctx*)p;
    for (int64_t n = 0; n < c->N; ++n) {
        /* Each int32 x int32 product is exact in int64.  The sum is carried
         * modulo 2^64 (unsigned, so a long K cannot overflow into undefined
         * behaviour); its low 32 bits equal those of the exact integer sum. */
        uint64_t acc = 0;                           /* zero start           */
        for (int64_t k = 0; k < c->K; ++k)
            acc += (uint64_t)((int64_t)c->lhs[m * c->K + k] * (int64_t)c->rhs[k * c->N + n]);
        /* two's-complement truncation to the low 32 bits */
        c->out[m * c->N + n] = (int32_t)(uint32_t)acc;
    }
}

void oracle_gemm_s32_nn(int64_t M, int64_t N, int64_t K, const int32_t* lhs,
                        const int32_t* rhs, int32_t* out, int nthreads) {
    s32_ctx c = {M, N, K, lhs, rhs, out};
    for_rows(M, nthreads, s32_row, &c);
}

/* ------------------------------------------------------------------------ */
/* f16 NT: ref[M,N] = lhs[M,K] . rhs[N,K]^T summed in binary64               */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t M, N, K;
    const double* a;   /* decoded lhs [M,K] */
    const double* b;   /* decoded rhs [N,K] */
    double* out;
} f16_ctx;

static void f16_row(void* p, int64_t m) {
    const f16_ctx* c = (const f16_ctx*)p;
    const double* arow = c->a + m * c->K;
    for (int64_t n = 0; n < c->N; ++n) {
        const double* brow = c->b + n * c->K;
        double acc = 0.0;
        for (int64_t k = 0; k < c->K; ++k) acc += arow[k] * brow[k];
        c->out[m * c->N + n] = acc;
    }
}

/* Returns 0 on success, -1 if the decoded operands could not be allocated. */
int oracle_gemm_f16_nt(int64_t M, int64_t N, int64_t K, const uint16_t* lhs,
                       const uint16_t* rhs, double* out, int nthreads) {
    double* a = (double*)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    double* b = (double*)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!a || !b) { free(a); free(b); return -1; }
    oracle_f16_to_f64_array(lhs, a, M * K);
    oracle_f16_to_f64_array(rhs, b, N * K);
    f16_ctx c = {M, N, K, a, b, out};
    for_rows(M, nthreads, f16_row, &c);
    free(a);
    free(b);
    return 0;
}

/* Selected entries only: ref[i] = sum_k lhs[rows[i],k] * rhs[cols[i],k].
 * Used where the full product is too large for the CPU. */
typedef struct {
    int64_t K;
    const uint16_t* lhs;
    const uint16_t* rhs;
    const int64_t* rows;
    const int64_t* cols;
    double* out;
} f16_entry_ctx;

static void f16_entry(void* p, int64_t i) {
    const f16_entry_ctx* c = (const f16_entry_ctx*)p;
    const uint16_t* arow = c->lhs + c->rows[i] * c->K;
    const uint16_t* brow = c->rhs + c->cols[i] * c->K;
    double acc = 0.0;
    for (int64_t k = 0; k < c->K; ++k)
        acc += oracle_f16_to_f64(arow[k]) * oracle_f16_to_f64(brow[k]);
    c->out[i] = acc;
}

void oracle_gemm_f16_nt_entries(int64_t K, const uint16_t* lhs, const uint16_t* rhs,
                                const int64_t* rows, const int64_t* cols, int64_t count,
                                double* out, int nthreads) {
    f16_entry_ctx c = {K, lhs, rhs, rows, cols, out};
    for_rows(count, nthreads, f16_entry, &c);
}

typedef struct {
    int64_t N, K;
    const int32_t* lhs;
    const int32_t* rhs;
    const int64_t* rows;
    const int64_t* cols;
    int32_t* out;
} s32_entry_ctx;

static void s32_entry(void* p, int64_t i) {
    const s32_entry_ctx* c = (const s32_entry_ctx*)p;
    uint64_t acc = 0;
    for (int64_t k = 0; k < c->K; ++k)
        acc += (uint64_t)((int64_t)c->lhs[c->rows[i] * c->K + k] * (int64_t)c->rhs[k * c->N + c->cols[i]]);
    c->out[i] = (int32_t)(uint32_t)acc;
}

void oracle_gemm_s32_nn_entries(int64_t N, int64_t K, const int32_t* lhs, const int32_t* rhs,
                                const int64_t* rows, const int64_t* cols, int64_t count,
                                int32_t* out, int nthreads) {
    s32_entry_ctx c = {N, K, lhs, rhs, rows, cols, out};
    for_rows(count, nthreads, s32_entry, &c);
}
