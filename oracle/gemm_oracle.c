/*
 * gemm_oracle.c -- the CPU oracle for the dense fp16 GEMM  D = A * B^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  The CUDA library
 * never links, loads or calls it, and it shares no code with that library.
 *
 * What it computes (and where the definition comes from):
 *   "Building a Tiled GEMM" (MLC, Modern GPU Programming for MLSys),
 *   section "GEMM": A is M x K, B is N x K (the linear-layer weight layout,
 *   read as stored, never transposed), D is M x N and
 *       D[m,n] = sum_k A[m,k] * B[n,k].
 *   Same section: A, B and D are stored as fp16 and the MMA accumulates in
 *   fp32.  The oracle is the plain definition at higher precision:
 *       D[m,n] = fp16_rne( sum_{k=0}^{K-1} (double)A[m,k] * (double)B[n,k] )
 *   summed in ascending k with one fp64 accumulator, then rounded ONCE,
 *   directly from fp64 to fp16 (round to nearest, ties to even).  The
 *   product of two fp16 values has at most 22 significant bits, so every
 *   product is exact in fp64; contraction into an FMA would not change it,
 *   and the build passes -ffp-contract=off anyway.
 *
 * Readings of the pages taken here (the pages leave them open):
 *   - the rounding mode of the final fp32->fp16 cast is not stated on the
 *     pages; round-to-nearest-even (the IEEE default) is used;
 *   - a K that is not a multiple of the 64-wide K tile still contributes
 *     every k (the definition sums over all k);
 *   - NaN and infinity inputs follow IEEE arithmetic in fp64.
 *
 * Binary16 (IEEE 754-2008, section 3.6, "interchange format" with k = 16):
 *   1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 *   exponent field 0       : subnormal, value = frac * 2^-24
 *   exponent field 1..30   : normal,    value = (1024 + frac) * 2^(e - 25)
 *   exponent field 31      : infinity (frac == 0) or NaN.
 * Every finite binary16 value is an integer multiple of 2^-24; in the binade
 * [2^E, 2^(E+1)) with E >= -14 the spacing is 2^(E-10); below 2^-14 the
 * spacing is 2^-24.  The largest finite value is 65504 = 2047 * 2^5.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* binary16 decode: the value a bit pattern stands for                 */
/* ------------------------------------------------------------------ */
static double f16_decode(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1F;
    const int frac = h & 0x3FF;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);                 /* zero or subnormal */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25);  /* normal */
    }
    return sign ? -v : v;
}

/* ------------------------------------------------------------------ */
/* binary16 encode: round a double to the nearest binary16, ties even  */
/* ------------------------------------------------------------------ */
static uint16_t f16_encode(double x) {
    uint64_t bits;
    memcpy(&bits, &x, sizeof bits);
    const uint16_t sign = (uint16_t)((bits >> 48) & 0x8000u);
    const int eb = (int)((bits >> 52) & 0x7FF);          /* biased double exponent */
    const uint64_t man = bits & 0x000FFFFFFFFFFFFFull;

    if (eb == 0x7FF) {                                    /* inf or NaN */
        if (man == 0) return sign | 0x7C00u;
        return sign | 0x7E00u;                            /* a quiet NaN */
    }
    if (eb == 0) return sign;                             /* |x| < 2^-1022 rounds to zero */

    /* |x| = sig * 2^(eb - 1075), sig a 53-bit integer with its top bit set. */
    const uint64_t sig = (1ull << 52) | man;
    const int E = eb - 1023;                              /* floor(log2 |x|) */
    if (E >= 16) return sign | 0x7C00u;                   /* >= 65536: overflow */

    /* Spacing of binary16 values around |x| is 2^q. */
    const int q = (E > -14 ? E : -14) - 10;
    /* n = |x| / 2^q = sig * 2^(eb - 1075 - q); the shift is >= 42. */
    const int s = q + 1075 - eb;
    uint64_t n;
    if (s >= 64) {
        n = 0;                                            /* |x| < 2^-25 * 2^-10: far below half a step */
    } else {
        n = sig >> s;
        const uint64_t rem = sig & ((1ull << s) - 1);
        const uint64_t half = 1ull << (s - 1);
        if (rem > half || (rem == half && (n & 1))) n += 1;   /* nearest, ties to even */
    }
    /* result = n * 2^q */
    int qq = q;
    if (qq == -24 && n < 1024) return sign | (uint16_t)n;   /* subnormal (or zero) */
    if (n == 2048) { n = 1024; qq += 1; }                     /* rounded up into the next binade */
    const int expo = qq + 10 + 15;                            /* biased binary16 exponent */
    if (expo >= 31) return sign | 0x7C00u;                    /* overflow to infinity */
    return sign | (uint16_t)(expo << 10) | (uint16_t)(n - 1024);
}

/* ------------------------------------------------------------------ */
/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits --  */
/* the top half of an IEEE binary32 (the GEMM blog post, section 2.2,     */
/* lists it beside fp16: same size, binary32's exponent range).           */
/*   exponent field 0      : subnormal, value = frac * 2^-133             */
/*   exponent field 1..254 : normal,    value = (128 + frac) * 2^(e - 134)*/
/*   exponent field 255    : infinity (frac == 0) or NaN.                 */
/* In the binade [2^E, 2^(E+1)), E >= -126, values are 2^(E-7) apart;     */
/* below 2^-126 they are 2^-133 apart.  Largest finite: 255 * 2^120.      */
/* ------------------------------------------------------------------ */
static double bf16_decode(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 7) & 0xFF;
    const int frac = h & 0x7F;
    double v;
    if (expo == 0) v = ldexp((double)frac, -133);
    else if (expo == 255) v = frac ? NAN : INFINITY;
    else v = ldexp((double)(128 + frac), expo - 134);
    return sign ? -v : v;
}

static uint16_t bf16_encode(double x) {
    uint64_t bits;
    memcpy(&bits, &x, sizeof bits);
    const uint16_t sign = (uint16_t)((bits >> 48) & 0x8000u);
    const int eb = (int)((bits >> 52) & 0x7FF);
    const uint64_t man = bits & 0x000FFFFFFFFFFFFFull;
    if (eb == 0x7FF) {
        if (man == 0) return sign | 0x7F80u;
        return sign | 0x7FC0u;                            /* a quiet NaN */
    }
    if (eb == 0) return sign;                             /* below 2^-1022: rounds to zero */
    const uint64_t sig = (1ull << 52) | man;              /* |x| = sig * 2^(eb - 1075) */
    const int E = eb - 1023;
    if (E >= 128) return sign | 0x7F80u;                  /* >= 2^128: overflow */
    const int q = (E > -126 ? E : -126) - 7;              /* spacing 2^q around |x| */
    const int s = q + 1075 - eb;                          /* >= 45 */
    uint64_t n;
    if (s >= 64) {
        n = 0;
    } else {
        n = sig >> s;
        const uint64_t rem = sig & ((1ull << s) - 1);
        const uint64_t half = 1ull << (s - 1);
        if (rem > half || (rem == half && (n & 1))) n += 1;  /* nearest, ties to even */
    }
    int qq = q;
    if (qq == -133 && n < 128) return sign | (uint16_t)n;    /* subnormal or zero */
    if (n == 256) { n = 128; qq += 1; }
    const int expo = qq + 7 + 127;
    if (expo >= 255) return sign | 0x7F80u;
    return sign | (uint16_t)(expo << 7) | (uint16_t)(n - 128);
}

/* ------------------------------------------------------------------ */
/* 8-bit floating point: the GEMM blog post (section 2.2) lists FP8 in  */
/* two layouts, E4M3 and E5M2.  The encodings are those of the 8-bit    */
/* formats that the tensor cores take (the OCP 8-bit floating point     */
/* formats):                                                            */
/* E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits, no      */
/*   infinities; S.1111.111 is the only NaN.                            */
/*   exponent field 0     : subnormal, value = frac * 2^-9              */
/*   exponent field 1..15 : normal,    value = (8 + frac) * 2^(e - 10)  */
/*   Largest finite: S.1111.110 = 14 * 2^5 = 448, the bound the blog    */
/*   post's quantisation step (section 4.2) scales values to.           */
/* E5M2: 1 sign bit, 5 exponent bits (bias 15), 2 fraction bits, laid   */
/*   out like binary16 with 8 fewer fraction bits.                      */
/*   exponent field 0     : subnormal, value = frac * 2^-16             */
/*   exponent field 1..30 : normal,    value = (4 + frac) * 2^(e - 17)  */
/*   exponent field 31    : infinity (frac == 0) or NaN.                */
/*   Largest finite: 7 * 2^13 = 57344.                                  */
/* The product of two such values has at most 3 + 3 (or 2 + 2)          */
/* significant bits beyond the leading one: exact in fp64.              */
/* ------------------------------------------------------------------ */
static double e4m3_decode(uint8_t h) {
    const int sign = (h >> 7) & 1;
    const int expo = (h >> 3) & 0xF;
    const int frac = h & 0x7;
    double v;
    if (expo == 0) v = ldexp((double)frac, -9);
    else if (expo == 15 && frac == 7) v = NAN;
    else v = ldexp((double)(8 + frac), expo - 10);
    return sign ? -v : v;
}

static double e5m2_decode(uint8_t h) {
    const int sign = (h >> 7) & 1;
    const int expo = (h >> 2) & 0x1F;
    const int frac = h & 0x3;
    double v;
    if (expo == 0) v = ldexp((double)frac, -16);
    else if (expo == 31) v = frac ? NAN : INFINITY;
    else v = ldexp((double)(4 + frac), expo - 17);
    return sign ? -v : v;
}

/* Decode table built from f16_decode, so the inner loop does not re-derive
 * each value.  Built once, thread-safely. */
static double g_decode[65536];
static pthread_once_t g_decode_once = PTHREAD_ONCE_INIT;
static void build_decode_table(void) {
    for (uint32_t h = 0; h < 65536u; ++h) g_decode[h] = f16_decode((uint16_t)h);
}
static const double* decode_table(void) {
    pthread_once(&g_decode_once, build_decode_table);
    return g_decode;
}

static double g_decode_bf16[65536];
static pthread_once_t g_decode_bf16_once = PTHREAD_ONCE_INIT;
static void build_decode_bf16_table(void) {
    for (uint32_t h = 0; h < 65536u; ++h) g_decode_bf16[h] = bf16_decode((uint16_t)h);
}
static const double* decode_bf16_table(void) {
    pthread_once(&g_decode_bf16_once, build_decode_bf16_table);
    return g_decode_bf16;
}

static double g_decode_e4m3[256], g_decode_e5m2[256];
static pthread_once_t g_decode_f8_once = PTHREAD_ONCE_INIT;
static void build_decode_f8_tables(void) {
    for (uint32_t h = 0; h < 256u; ++h) {
        g_decode_e4m3[h] = e4m3_decode((uint8_t)h);
        g_decode_e5m2[h] = e5m2_decode((uint8_t)h);
    }
}
static const double* decode_e4m3_table(void) {
    pthread_once(&g_decode_f8_once, build_decode_f8_tables);
    return g_decode_e4m3;
}
static const double* decode_e5m2_table(void) {
    pthread_once(&g_decode_f8_once, build_decode_f8_tables);
    return g_decode_e5m2;
}

/* One element of the definition: ascending k, one fp64 accumulator. */
static double dot_row_row(const double* dec, const uint16_t* a_row, const uint16_t* b_row, int64_t K) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += dec[a_row[k]] * dec[b_row[k]];
    return acc;
}

/* The same for 8-bit operands. */
static double dot_row_row8(const double* dec, const uint8_t* a_row, const uint8_t* b_row, int64_t K) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += dec[a_row[k]] * dec[b_row[k]];
    return acc;
}

/* ------------------------------------------------------------------ */
/* exported: element conversions                                       */
/* ------------------------------------------------------------------ */
void oracle_f16_to_f64(const uint16_t* h, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = f16_decode(h[i]);
}

void oracle_f64_to_f16(const double* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = f16_encode(x[i]);
}

void oracle_bf16_to_f64(const uint16_t* h, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_decode(h[i]);
}

void oracle_f64_to_bf16(const double* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_encode(x[i]);
}

void oracle_e4m3_to_f64(const uint8_t* h, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_decode(h[i]);
}

void oracle_e5m2_to_f64(const uint8_t* h, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = e5m2_decode(h[i]);
}

/* ------------------------------------------------------------------ */
/* exported: GEMM over a list of (row, col) entries                    */
/* ------------------------------------------------------------------ */
typedef struct {
    const uint16_t* A;
    const uint16_t* B;
    int64_t M, N, K;
    const int64_t* rows;   /* entries mode */
    const int64_t* cols;
    int64_t count;
    int64_t row_begin;     /* rows mode */
    int64_t row_end;
    double* sums;          /* optional fp64 output */
    uint16_t* out;         /* optional fp16 output */
    int nthreads;
    int tid;
} job_t;

static void* entries_worker(void* p) {
    job_t* j = (job_t*)p;
    const double* dec = decode_table();
    for (int64_t i = j->tid; i < j->count; i += j->nthreads) {
        const int64_t m = j->rows[i], n = j->cols[i];
        const double acc = dot_row_row(dec, j->A + m * j->K, j->B + n * j->K, j->K);
        if (j->sums) j->sums[i] = acc;
        if (j->out) j->out[i] = f16_encode(acc);
    }
    return NULL;
}

static void* rows_worker(void* p) {
    job_t* j = (job_t*)p;
    const double* dec = decode_table();
    /* thread tid takes one contiguous block of the (row, col) entries */
    const int64_t total = (j->row_end - j->row_begin) * j->N;
    const int64_t lo = total * j->tid / j->nthreads;
    const int64_t hi = total * (j->tid + 1) / j->nthreads;
    for (int64_t idx = lo; idx < hi; ++idx) {
        const int64_t m = j->row_begin + idx / j->N;
        const int64_t n = idx % j->N;
        const double acc = dot_row_row(dec, j->A + m * j->K, j->B + n * j->K, j->K);
        if (j->sums) j->sums[idx] = acc;
        if (j->out) j->out[idx] = f16_encode(acc);
    }
    return NULL;
}

static int run_threads(job_t* proto, void* (*fn)(void*)) {
    int nt = proto->nthreads < 1 ? 1 : proto->nthreads;
    if (nt > 1024) nt = 1024;
    proto->nthreads = nt;
    job_t* jobs = (job_t*)malloc(sizeof(job_t) * (size_t)nt);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!jobs || !th) { free(jobs); free(th); return -1; }
    int started = 0;
    for (int t = 0; t < nt; ++t) {
        jobs[t] = *proto;
        jobs[t].tid = t;
        if (t == 0) continue;
        if (pthread_create(&th[t], NULL, fn, &jobs[t]) != 0) break;
        started = t;
    }
    /* thread 0's share runs here; shares of threads that failed to start
     * are picked up serially so the result is always complete */
    fn(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    for (int t = started + 1; t < nt; ++t) fn(&jobs[t]);
    free(jobs);
    free(th);
    return 0;
}

/* D entries at (rows[i], cols[i]); sums (fp64, unrounded) and/or out (fp16
 * bits) may be NULL.  Returns 0, or -1 on bad arguments. */
int oracle_gemm_nt_entries(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K,
                           const int64_t* rows, const int64_t* cols, int64_t count,
                           double* sums, uint16_t* out, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
    for (int64_t i = 0; i < count; ++i)
        if (rows[i] < 0 || rows[i] >= M || cols[i] < 0 || cols[i] >= N) return -1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.A = A; j.B = B; j.M = M; j.N = N; j.K = K;
    j.rows = rows; j.cols = cols; j.count = count;
    j.sums = sums; j.out = out; j.nthreads = nthreads;
    return run_threads(&j, entries_worker);
}

/* Rows [row_begin, row_end) of D, all N columns, written row-major into
 * out[(m - row_begin) * N + n] (and/or sums).  Returns 0, or -1. */
int oracle_gemm_nt_rows(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K,
                        int64_t row_begin, int64_t row_end,
                        double* sums, uint16_t* out, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || row_begin < 0 || row_end > M || row_begin > row_end) return -1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.A = A; j.B = B; j.M = M; j.N = N; j.K = K;
    j.row_begin = row_begin; j.row_end = row_end;
    j.sums = sums; j.out = out; j.nthreads = nthreads;
    return run_threads(&j, rows_worker);
}

/* ------------------------------------------------------------------ */
/* exported: GEMM with an element type and the fused output transform  */
/*   D[m,n] = round( act( alpha * s[n] * S[m,n] + beta * C[m,n]         */
/*                        + bias[n] ) )                                 */
/* with S the plain definition above (fp64, ascending k), every term in */
/* fp64 and one rounding to the output type at the end.  This is the    */
/* scaled update C = alpha A B + beta C of the GEMM blog post (section  */
/* 2.1) with the bias and ReLU fusion it recommends (section 5.4).  s[n]*/
/* is an optional fp32 scale per output column: with 8-bit operands the */
/* blog post (section 4.2) quantises weights with one scale per output  */
/* channel (a row of B) and activations with one per tensor (alpha), and*/
/* passes the scales to the kernel as fp32 numbers.                     */
/* dtype 0 = fp16 operands and output, 1 = bf16 operands and output,    */
/* 2 = E4M3 operands, 3 = E5M2 operands (both with bf16 output, C and   */
/* bias).  C, bias and s may be NULL; act 0 none, 1 relu.               */
/* ------------------------------------------------------------------ */
typedef struct {
    int dtype;
    const void* A;        /* uint16_t bit patterns, or uint8_t for dtype 2 and 3 */
    const void* B;
    int64_t M, N, K;
    const int64_t* rows;
    const int64_t* cols;
    int64_t count;
    int64_t row_begin, row_end;
    double alpha, beta;
    const uint16_t* C;
    const uint16_t* bias;
    const float* scale_n;
    int act;
    double* pre;          /* optional: the value before rounding */
    uint16_t* out;
    int nthreads;
    int tid;
    int rows_mode;
} job_ex_t;

static double element_ex(const job_ex_t* j, const double* dec_in, const double* dec_out, int64_t m, int64_t n) {
    double sum;
    if (j->dtype >= 2)
        sum = dot_row_row8(dec_in, (const uint8_t*)j->A + m * j->K, (const uint8_t*)j->B + n * j->K, j->K);
    else
        sum = dot_row_row(dec_in, (const uint16_t*)j->A + m * j->K, (const uint16_t*)j->B + n * j->K, j->K);
    const double scale = j->scale_n ? (double)j->scale_n[n] : 1.0;
    double v = j->alpha * scale * sum;
    if (j->C && j->beta != 0.0) v += j->beta * dec_out[j->C[m * j->N + n]];
    if (j->bias) v += dec_out[j->bias[n]];
    if (j->act == 1 && v < 0.0) v = 0.0;   /* relu: negative values to zero; NaN and -0 pass */
    return v;
}

static void* ex_worker(void* p) {
    job_ex_t* j = (job_ex_t*)p;
    const double* dec_in = j->dtype == 0 ? decode_table()
                         : j->dtype == 1 ? decode_bf16_table()
                         : j->dtype == 2 ? decode_e4m3_table() : decode_e5m2_table();
    const double* dec_out = j->dtype == 0 ? decode_table() : decode_bf16_table();
    const int64_t total = j->rows_mode ? (j->row_end - j->row_begin) * j->N : j->count;
    const int64_t lo = total * j->tid / j->nthreads;
    const int64_t hi = total * (j->tid + 1) / j->nthreads;
    for (int64_t i = lo; i < hi; ++i) {
        int64_t m, n;
        if (j->rows_mode) { m = j->row_begin + i / j->N; n = i % j->N; }
        else { m = j->rows[i]; n = j->cols[i]; }
        const double v = element_ex(j, dec_in, dec_out, m, n);
        if (j->pre) j->pre[i] = v;
        j->out[i] = j->dtype == 0 ? f16_encode(v) : bf16_encode(v);
    }
    return NULL;
}

static int run_ex(job_ex_t* proto) {
    int nt = proto->nthreads < 1 ? 1 : proto->nthreads;
    if (nt > 1024) nt = 1024;
    proto->nthreads = nt;
    job_ex_t* jobs = (job_ex_t*)malloc(sizeof(job_ex_t) * (size_t)nt);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!jobs || !th) { free(jobs); free(th); return -1; }
    int started = 0;
    for (int t = 0; t < nt; ++t) {
        jobs[t] = *proto;
        jobs[t].tid = t;
        if (t == 0) continue;
        if (pthread_create(&th[t], NULL, ex_worker, &jobs[t]) != 0) break;
        started = t;
    }
    ex_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    for (int t = started + 1; t < nt; ++t) ex_worker(&jobs[t]);
    free(jobs);
    free(th);
    return 0;
}

/* Entries (rows[i], cols[i]) when rows != NULL, else rows [row_begin,
 * row_end) written row-major.  Returns 0, or -1 on bad arguments. */
int oracle_gemm_nt_ex(int dtype, const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                      const int64_t* rows, const int64_t* cols, int64_t count,
                      int64_t row_begin, int64_t row_end,
                      double alpha, double beta, const uint16_t* C, const uint16_t* bias,
                      const float* scale_n, int act, double* pre, uint16_t* out, int nthreads) {
    if (dtype < 0 || dtype > 3 || M < 0 || N < 0 || K < 0 || (act != 0 && act != 1)) return -1;
    job_ex_t j;
    memset(&j, 0, sizeof j);
    if (rows) {
        if (count < 0) return -1;
        for (int64_t i = 0; i < count; ++i)
            if (rows[i] < 0 || rows[i] >= M || cols[i] < 0 || cols[i] >= N) return -1;
        j.rows = rows; j.cols = cols; j.count = count;
    } else {
        if (row_begin < 0 || row_end > M || row_begin > row_end) return -1;
        j.rows_mode = 1; j.row_begin = row_begin; j.row_end = row_end;
    }
    j.dtype = dtype; j.A = A; j.B = B; j.M = M; j.N = N; j.K = K;
    j.alpha = alpha; j.beta = beta; j.C = C; j.bias = bias; j.scale_n = scale_n; j.act = act;
    j.pre = pre; j.out = out; j.nthreads = nthreads;
    return run_ex(&j);
}
