/*
 * gemm_oracle.c -- the CPU oracle for the tiled GEMM K-loop library.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant with
 * the CUDA kernels: the only include beyond the C library is <stdint.h>.
 *
 * What it computes is the plain definition of a matrix product, the form
 * printed in "Part 4 -- Pipelining and Occupancy", section 4.3 "Register
 * reuse": the triple loop over i, j, k whose inner sum is kept in a local
 * variable and stored once per output element.  The software pipeline that the
 * library implements ("CUDA Kernel Study: Pipelining", Case 1 and Case 2;
 * "pipeline-gpu-kernel", Step 5 item 4) only reorders loads, so this
 * definition is the exact result the pipelined kernels must reach.
 *
 *  - INT8 x INT8 -> INT32: the products are formed in 32-bit integers and
 *    summed with two's-complement wrap-around, which is the wrap that the
 *    uint32_t triple loop at the end of section 4.3 has.  Exact; the order of
 *    summation cannot matter.
 *  - FP16 / BF16 / FP32 inputs: each stored element is converted exactly to
 *    double (the conversions below are written from the IEEE-754 binary16
 *    and the bfloat16 bit layouts), the products are exact in double and the
 *    sum is kept in a double.  The result C_ref is returned in double; the
 *    caller rounds it to the output type with the round-to-nearest-even
 *    routines below when it wants the stored form.
 *  - A float-sum triple loop (the section 4.3 code with T = float) is also
 *    provided, as an information line only.
 *
 * Element addressing is by strides so that one routine serves every layout:
 * A[i][k] = A[i*a_si + k*a_sk], B[k][j] = B[k*b_sk + j*b_sj].
 * Rows may be restricted to a list so that very large problems can be
 * checked on a subset; outputs for listed rows are written densely,
 * C[r*N + j] for the r-th listed row.
 *
 * The only concession to speed is an OpenMP "parallel for" over output rows
 * (each row is computed by exactly the same loop as without it).
 */
#include <stdint.h>
#include <math.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* threads                                                                    */
/* ------------------------------------------------------------------------- */

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_has_openmp(void) {
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}

/* ------------------------------------------------------------------------- */
/* IEEE-754 binary16 and bfloat16 <-> double                                  */
/* ------------------------------------------------------------------------- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/2^10) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_f64(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);                /* subnormal: f * 2^-133 */
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + f), e - 134);     /* (1 + f/2^7) * 2^(e-127) */
    }
    return sign ? -v : v;
}

/* Round a non-negative double holding a value below 2^52 to the nearest
 * integer, ties to even. */
static double round_half_even(double r) {
    double fl = floor(r);
    double d = r - fl;                  /* exact for r < 2^52 */
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* Generic round-to-nearest-even of |x| into a binary format with `mant` fraction
 * bits, exponent bias `bias` and all-ones exponent reserved for inf/NaN.
 * Returns the magnitude bits (without the sign). */
static uint32_t round_magnitude(double a, int mant, int bias, int ebits) {
    const int emax = (1 << ebits) - 2 - bias;          /* largest normal exponent */
    const int emin = 1 - bias;                         /* smallest normal exponent */
    const uint32_t inf_bits = (uint32_t)((1 << ebits) - 1) << mant;
    if (a == 0.0) return 0;
    if (isinf(a)) return inf_bits;
    int ex;
    frexp(a, &ex);                                     /* a = m * 2^ex, m in [0.5,1) */
    int E = ex - 1;                                    /* a = (2m) * 2^E */
    if (E < emin) {
        /* subnormal range: multiples of 2^(emin - mant) */
        double q = round_half_even(ldexp(a, mant - emin));
        return (uint32_t)q;                            /* q == 2^mant encodes the smallest normal */
    }
    double s = round_half_even(ldexp(a, mant - E));    /* in [2^mant, 2^(mant+1)] */
    if (s >= ldexp(1.0, mant + 1)) { s = ldexp(1.0, mant); E += 1; }
    if (E > emax) return inf_bits;
    return ((uint32_t)(E + bias) << mant) | ((uint32_t)s - (1u << mant));
}

uint16_t oracle_f64_to_f16_rn(double x) {
    if (isnan(x)) return 0x7e00;
    uint16_t s = signbit(x) ? 0x8000 : 0;
    return (uint16_t)(s | round_magnitude(fabs(x), 10, 15, 5));
}

uint16_t oracle_f64_to_bf16_rn(double x) {
    if (isnan(x)) return 0x7fc0;
    uint16_t s = signbit(x) ? 0x8000 : 0;
    return (uint16_t)(s | round_magnitude(fabs(x), 7, 127, 8));
}

void oracle_decode_f16(const uint16_t* x, double* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_f16_to_f64(x[i]);
}

void oracle_decode_bf16(const uint16_t* x, double* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_bf16_to_f64(x[i]);
}

void oracle_round_f16(const double* x, uint16_t* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_f64_to_f16_rn(x[i]);
}

void oracle_round_bf16(const double* x, uint16_t* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_f64_to_bf16_rn(x[i]);
}

/* ------------------------------------------------------------------------- */
/* INT8 x INT8 -> INT32 (wrap)                                                */
/* ------------------------------------------------------------------------- */

/* rows == NULL means every row 0..M-1 (nrows must then be M). */
void oracle_gemm_i8_i32(const int8_t* A, const int8_t* B, int32_t* C,
                        int64_t M, int64_t N, int64_t K,
                        int64_t a_si, int64_t a_sk, int64_t b_sk, int64_t b_sj,
                        const int64_t* rows, int64_t nrows) {
    (void)M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        for (int64_t j = 0; j < N; ++j) {
            uint32_t sum = 0;                          /* wraps modulo 2^32 */
            for (int64_t k = 0; k < K; ++k) {
                int32_t a = A[i * a_si + k * a_sk];
                int32_t b = B[k * b_sk + j * b_sj];
                sum += (uint32_t)(a * b);              /* |a*b| <= 2^14: no overflow */
            }
            int32_t out;
            memcpy(&out, &sum, sizeof out);            /* two's-complement reading */
            C[r * N + j] = out;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* FP16 / BF16 / FP32 inputs, products and sum in double                      */
/* ------------------------------------------------------------------------- */

enum { ORACLE_IN_F16 = 0, ORACLE_IN_BF16 = 1, ORACLE_IN_F32 = 2 };

static double decode(int in_type, const void* base, int64_t idx, const double* lut) {
    if (in_type == ORACLE_IN_F32) return (double)((const float*)base)[idx];
    return lut[((const uint16_t*)base)[idx]];
}

/* lut: caller-free scratch of 65536 doubles (may be NULL for f32). */
static void build_lut(int in_type, double* lut) {
    for (uint32_t b = 0; b < 65536u; ++b)
        lut[b] = (in_type == ORACLE_IN_F16) ? oracle_f16_to_f64((uint16_t)b)
                                            : oracle_bf16_to_f64((uint16_t)b);
}

static double g_lut_f16[65536];
static double g_lut_bf16[65536];
static int g_lut_ready = 0;

static const double* lut_for(int in_type) {
    if (!g_lut_ready) {
        build_lut(ORACLE_IN_F16, g_lut_f16);
        build_lut(ORACLE_IN_BF16, g_lut_bf16);
        g_lut_ready = 1;
    }
    if (in_type == ORACLE_IN_F16) return g_lut_f16;
    if (in_type == ORACLE_IN_BF16) return g_lut_bf16;
    return 0;
}

int oracle_gemm_f64(int in_type, const void* A, const void* B, double* C,
                    int64_t M, int64_t N, int64_t K,
                    int64_t a_si, int64_t a_sk, int64_t b_sk, int64_t b_sj,
                    const int64_t* rows, int64_t nrows) {
    (void)M;
    if (in_type < 0 || in_type > 2) return -1;
    const double* lut = lut_for(in_type);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        for (int64_t j = 0; j < N; ++j) {
            double sum = 0.0;
            for (int64_t k = 0; k < K; ++k)
                sum += decode(in_type, A, i * a_si + k * a_sk, lut) *
                       decode(in_type, B, k * b_sk + j * b_sj, lut);
            C[r * N + j] = sum;
        }
    }
    return 0;
}

/* Sampled points: C[p] = sum_k A[rows[p]][k] * B[k][cols[p]]. */
void oracle_points_i8_i32(const int8_t* A, const int8_t* B, int32_t* C, int64_t K,
                          int64_t a_si, int64_t a_sk, int64_t b_sk, int64_t b_sj,
                          const int64_t* rows, const int64_t* cols, int64_t npts) {
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < npts; ++p) {
        uint32_t sum = 0;
        for (int64_t k = 0; k < K; ++k) {
            int32_t a = A[rows[p] * a_si + k * a_sk];
            int32_t b = B[k * b_sk + cols[p] * b_sj];
            sum += (uint32_t)(a * b);
        }
        int32_t out;
        memcpy(&out, &sum, sizeof out);
        C[p] = out;
    }
}

int oracle_points_f64(int in_type, const void* A, const void* B, double* C, int64_t K,
                      int64_t a_si, int64_t a_sk, int64_t b_sk, int64_t b_sj,
                      const int64_t* rows, const int64_t* cols, int64_t npts) {
    if (in_type < 0 || in_type > 2) return -1;
    const double* lut = lut_for(in_type);
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < npts; ++p) {
        double sum = 0.0;
        for (int64_t k = 0; k < K; ++k)
            sum += decode(in_type, A, rows[p] * a_si + k * a_sk, lut) *
                   decode(in_type, B, k * b_sk + cols[p] * b_sj, lut);
        C[p] = sum;
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* The section 4.3 triple loop with T = float (information only)             */
/* ------------------------------------------------------------------------- */

void oracle_gemm_f32_loop(const float* A, const float* B, float* C,
                          int64_t M, int64_t N, int64_t K,
                          int64_t a_si, int64_t a_sk, int64_t b_sk, int64_t b_sj,
                          const int64_t* rows, int64_t nrows) {
    (void)M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        for (int64_t j = 0; j < N; ++j) {
            float sum = 0.0f;
            for (int64_t k = 0; k < K; ++k)
                sum += A[i * a_si + k * a_sk] * B[k * b_sk + j * b_sj];
            C[r * N + j] = sum;
        }
    }
}
