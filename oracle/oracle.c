/*
 * ORACLE -- test infrastructure only.
 *
 * A plain, slow, obviously correct CPU restatement of what the ONNX MatMul
 * operator computes, used to check the CUDA library.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load this code; the
 * product library never links, loads or calls it, and it shares no code,
 * header or table with the product.
 *
 * What it computes (MatMul Kernel Design, sections "Shape and plan model" and
 * "Types and algorithm selection"; Gemm and MatMul Performance Roadmap,
 * section "Scope and type matrix", the type/accumulation table):
 *
 *   Y[i, j] = sum over k = 0 .. K-1 of A[i, k] * B[k, j]
 *
 *   float32  inputs: float32 accumulator, k ascending, one rounding per product
 *                    and one per addition (no fused multiply-add);
 *   float64  inputs: float64 accumulator, same order;
 *   float16 / bfloat16 inputs: every element widened exactly to float32, the
 *                    products accumulated in float32 with k ascending, and the
 *                    finished sum narrowed once to the input type with
 *                    round-to-nearest-even ("FP32 accumulation and final
 *                    narrowing").
 *
 * It also returns S[i, j] = sum_k |A[i, k]| * |B[k, j]| in float64: the scale
 * that the parity tolerance |y - ref| <= tol * S is stated against.
 *
 * The batch loop, rank-one promotion and broadcasting live in the Python half
 * of the oracle (oracle/__init__.py); this file holds only the 2-D product and
 * the binary16 / bfloat16 encode and decode.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC.
 * -ffp-contract=off keeps every product and every sum separately rounded, so
 * the compiler cannot turn the accumulation into FMAs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Number of host threads the oracle's parallel loops use.                  */
int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Set the number of host threads (n >= 1) for the following calls; used
 * to time the oracle on one core.  The results do not depend on it: every
 * output row is computed by one thread in the same k order. */
void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 -> binary32 (exact).  Fields: 1 sign bit, 5 exponent bits
 * (bias 15), 10 fraction bits.  exponent 0 = zero / subnormal (value =
 * fraction * 2^-24), exponent 31 = infinity (fraction 0) or NaN. */
float oracle_f16_to_f32(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    float v;
    if (e == 0) {
        v = ldexpf((float)f, -24);
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        /* (1024 + f) * 2^(e - 15 - 10) */
        v = ldexpf((float)(f | 0x400), e - 25);
    }
    return sign ? -v : v;
}

/* bfloat16 is, by definition, the upper half of a binary32 encoding. */
float oracle_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float v;
    memcpy(&v, &u, sizeof v);
    return v;
}

/* Round a non-negative double to the nearest integer, ties to even. */
static double round_half_even(double n) {
    double fl = floor(n);
    double d = n - fl;
    if (d > 0.5 || (d == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    return fl;
}

/*
 * Narrow a binary32 value to a binary format with p significand bits
 * (implicit bit included), exponent bias `bias` (so normal exponents run from
 * 1 - bias to bias) and round-to-nearest-even.  Returns the 16-bit encoding:
 * sign | biased exponent << (p - 1) | fraction.
 *
 * The value is written as n * q with q the spacing of the format at |x|
 * (2^(E - p + 1) for a normal binade 2^E, 2^(1 - bias - p + 1) below the
 * smallest normal), n is rounded half-to-even, and the encoding is formed by
 * adding n into the exponent field so a carry out of the fraction moves to the
 * next binade -- and past the largest binade to infinity.  NaN becomes the
 * quiet NaN with the input's sign.
 */
static uint16_t narrow_rne(float f, int p, int bias) {
    const int frac_bits = p - 1;
    const int exp_all_ones = 2 * bias + 1;
    uint16_t sign = signbit(f) ? (uint16_t)(1u << 15) : 0;
    if (isnan(f)) {
        return sign | (uint16_t)(exp_all_ones << frac_bits) | (uint16_t)(1u << (frac_bits - 1));
    }
    double x = fabs((double)f);
    if (isinf(f)) return sign | (uint16_t)(exp_all_ones << frac_bits);
    if (x == 0.0) return sign;
    int e2;
    frexp(x, &e2);            /* x = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;           /* x in [2^E, 2^(E+1)) */
    const int emin = 1 - bias;
    if (E > bias) return sign | (uint16_t)(exp_all_ones << frac_bits); /* beyond the largest binade */
    int qexp = (E < emin ? emin : E) - frac_bits;   /* exponent of the spacing q */
    double n = round_half_even(ldexp(x, -qexp));    /* exact scaling by a power of two */
    uint32_t bits;
    if (E < emin) {
        /* subnormal: exponent field 0, fraction n; n == 2^frac_bits lands on the
           smallest normal encoding by itself */
        bits = (uint32_t)n;
    } else {
        bits = ((uint32_t)(E + bias) << frac_bits) + ((uint32_t)n - (1u << frac_bits));
    }
    if (bits >= (uint32_t)(exp_all_ones << frac_bits)) bits = (uint32_t)(exp_all_ones << frac_bits);
    return sign | (uint16_t)bits;
}

uint16_t oracle_f32_to_f16(float f) { return narrow_rne(f, 11, 15); }
uint16_t oracle_f32_to_bf16(float f) { return narrow_rne(f, 8, 127); }

void oracle_decode_f16(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f32(in[i]);
}
void oracle_decode_bf16(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f32(in[i]);
}
void oracle_encode_f16(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16(in[i]);
}
void oracle_encode_bf16(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(in[i]);
}

/* ------------------------------------------------------------------------ */
/*
 * The 2-D product over a chosen set of output rows.
 *
 * A is row-major [M, K], B row-major [K, N].  `rows` lists nrows row indices
 * of Y to compute (NULL = all M rows, nrows = M).  Y and S are [nrows, N]:
 * output row r holds row rows[r] of the product.
 *
 * Loop order per output row: k outer, j inner, with one accumulator per
 * column.  Every Y[i, j] therefore sums its K terms in ascending k, exactly
 * the order of the definition; the j loop only runs independent sums side by
 * side.  K == 0 leaves Y = 0 and S = 0 (the empty sum).
 */
#define ROW_INDEX(r) (rows ? rows[(r)] : (r))

void oracle_gemm_f32(int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                     const int64_t* rows, int64_t nrows, float* Y, double* S) {
    (void)M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = ROW_INDEX(r);
        float* acc = Y + r * N;
        double* s = S + r * N;
        for (int64_t j = 0; j < N; ++j) { acc[j] = 0.0f; s[j] = 0.0; }
        for (int64_t k = 0; k < K; ++k) {
            const float a = A[i * K + k];
            const float* brow = B + k * N;
            for (int64_t j = 0; j < N; ++j) {
                float prod = a * brow[j];
                acc[j] = acc[j] + prod;
                s[j] += fabs((double)a) * fabs((double)brow[j]);
            }
        }
    }
}

void oracle_gemm_f64(int64_t M, int64_t N, int64_t K, const double* A, const double* B,
                     const int64_t* rows, int64_t nrows, double* Y, double* S) {
    (void)M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = ROW_INDEX(r);
        double* acc = Y + r * N;
        double* s = S + r * N;
        for (int64_t j = 0; j < N; ++j) { acc[j] = 0.0; s[j] = 0.0; }
        for (int64_t k = 0; k < K; ++k) {
            const double a = A[i * K + k];
            const double* brow = B + k * N;
            for (int64_t j = 0; j < N; ++j) {
                double prod = a * brow[j];
                acc[j] = acc[j] + prod;
                s[j] += fabs(a) * fabs(brow[j]);
            }
        }
    }
}

/* Shared body of the two 16-bit products: widen, accumulate in float32,
 * narrow once.  `kind` 0 = binary16, 1 = bfloat16.  With Y == NULL the
 * float32 accumulators are returned in Yacc instead (not narrowed), for the
 * Gemm operator, which narrows only after its alpha/beta epilogue. */
static void gemm_half(int kind, int64_t N, int64_t K, const uint16_t* A, const uint16_t* B,
                      const int64_t* rows, int64_t nrows, uint16_t* Y, double* S, float* Yacc) {
    float (*widen)(uint16_t) = kind ? oracle_bf16_to_f32 : oracle_f16_to_f32;
    uint16_t (*narrow)(float) = kind ? oracle_f32_to_bf16 : oracle_f32_to_f16;
    /* B widened once; widening is exact, so this is the same B. */
    float* Bw = (float*)malloc(sizeof(float) * (size_t)(K * N > 0 ? K * N : 1));
    for (int64_t t = 0; t < K * N; ++t) Bw[t] = widen(B[t]);
#pragma omp parallel
    {
        float* acc = (float*)malloc(sizeof(float) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t i = ROW_INDEX(r);
            double* s = S + r * N;
            for (int64_t j = 0; j < N; ++j) { acc[j] = 0.0f; s[j] = 0.0; }
            for (int64_t k = 0; k < K; ++k) {
                const float a = widen(A[i * K + k]);
                const float* brow = Bw + k * N;
                for (int64_t j = 0; j < N; ++j) {
                    float prod = a * brow[j]; /* exact: 11- or 8-bit significands */
                    acc[j] = acc[j] + prod;
                    s[j] += fabs((double)a) * fabs((double)brow[j]);
                }
            }
            for (int64_t j = 0; j < N; ++j) {
                if (Y) Y[r * N + j] = narrow(acc[j]);
                else Yacc[r * N + j] = acc[j];
            }
        }
        free(acc);
    }
    free(Bw);
}

void oracle_gemm_f16(int64_t M, int64_t N, int64_t K, const uint16_t* A, const uint16_t* B,
                     const int64_t* rows, int64_t nrows, uint16_t* Y, double* S) {
    (void)M;
    gemm_half(0, N, K, A, B, rows, nrows, Y, S, NULL);
}

void oracle_gemm_bf16(int64_t M, int64_t N, int64_t K, const uint16_t* A, const uint16_t* B,
                      const int64_t* rows, int64_t nrows, uint16_t* Y, double* S) {
    (void)M;
    gemm_half(1, N, K, A, B, rows, nrows, Y, S, NULL);
}

/* The 16-bit products' float32 accumulators, not narrowed (Gemm epilogue). */
void oracle_gemm_f16_acc(int64_t M, int64_t N, int64_t K, const uint16_t* A, const uint16_t* B,
                         const int64_t* rows, int64_t nrows, float* Yacc, double* S) {
    (void)M;
    gemm_half(0, N, K, A, B, rows, nrows, NULL, S, Yacc);
}

void oracle_gemm_bf16_acc(int64_t M, int64_t N, int64_t K, const uint16_t* A, const uint16_t* B,
                          const int64_t* rows, int64_t nrows, float* Yacc, double* S) {
    (void)M;
    gemm_half(1, N, K, A, B, rows, nrows, NULL, S, Yacc);
}
