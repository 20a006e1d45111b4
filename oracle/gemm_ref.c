/*
 * Oracle for the tiled GEMM  D = alpha * A * B + beta * C  (TEST INFRASTRUCTURE ONLY).
 *
 * This file is the plain, slow, obviously correct CPU definition that the GPU path is
 * checked against.  Only tests/, the smoke check and the bench's CPU-baseline leg may
 * load it; the product library never does.  It shares no code, header, table or helper
 * with the CUDA path.
 *
 * What it computes, and where that is defined:
 *   - "CUTLASS, in depth", section "The problem CUTLASS solves": D = alpha*A*B + beta*C,
 *     A of shape M x K, B of shape K x N.
 *   - "Day 84: CUTLASS and CuTe layouts", section "Two programs": the CPU reference reads
 *     the same half values the GPU read and sums the products in double precision.
 *   So every output is   acc(i,j)  = sum_k  double(A(i,k)) * double(B(k,j))
 *                        ref(i,j)  = alpha*acc + (beta != 0 ? beta*double(C(i,j)) : 0)
 *   with no blocking, no reordering and no fusion: k runs 0..K-1 in order.
 *
 * Operand addressing follows the layout convention of "Layouts as Algebra: CUTLASS &
 * CuTe", section "One notation, and no more transposes" (a matrix is named by its
 * stride-1 mode):
 *   A is M x K.  K-major: A(i,k) = A[i*lda + k].   M-major: A(i,k) = A[i + k*lda].
 *   B is K x N.  K-major: B(k,j) = B[j*ldb + k].   N-major: B(k,j) = B[k*ldb + j].
 *   C is M x N row-major: C(i,j) = C[i*ldc + j].
 *
 * The 16-bit formats are decoded from their IEEE-754 definitions (binary16: 1/5/10,
 * bfloat16: 1/8/7) and results are rounded back with round-to-nearest-even written
 * from the definition of that rounding (nearest representable value, ties to the even
 * significand).  Decoding is exact in double.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1, ORACLE_E4M3 = 2, ORACLE_E5M2 = 3 };
enum { ORACLE_K_MAJOR = 0, ORACLE_MN_MAJOR = 1 };

/* binary16: sign 1 bit, exponent 5 bits (bias 15), fraction 10 bits. */
static double decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^(1-15-10) */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f + 1024), e - 25);     /* (1 + f/2^10) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: sign 1 bit, exponent 8 bits (bias 127), fraction 7 bits. */
static double decode_bf16(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);                /* subnormal: f * 2^(1-127-7) */
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f + 128), e - 134);     /* (1 + f/2^7) * 2^(e-127) */
    }
    return sign ? -v : v;
}

/* FP8 E4M3 (the "fn" variant: 1/4/3, bias 7, no infinities; S.1111.111 is NaN, the
   largest finite value is 448). */
static double decode_e4m3(uint16_t bits) {
    int sign = (bits >> 7) & 1;
    int e = (bits >> 3) & 0xf;
    int f = bits & 0x7;
    double v;
    if (e == 15 && f == 7) {
        v = NAN;
    } else if (e == 0) {
        v = ldexp((double)f, -9);                  /* f * 2^(1-7-3) */
    } else {
        v = ldexp((double)(f + 8), e - 10);        /* (1 + f/8) * 2^(e-7) */
    }
    return sign ? -v : v;
}

/* FP8 E5M2 (1/5/2, bias 15, IEEE-style infinities and NaNs; largest finite 57344). */
static double decode_e5m2(uint16_t bits) {
    int sign = (bits >> 7) & 1;
    int e = (bits >> 2) & 0x1f;
    int f = bits & 0x3;
    double v;
    if (e == 31) {
        v = f ? NAN : INFINITY;
    } else if (e == 0) {
        v = ldexp((double)f, -16);                 /* f * 2^(1-15-2) */
    } else {
        v = ldexp((double)(f + 4), e - 17);        /* (1 + f/4) * 2^(e-15) */
    }
    return sign ? -v : v;
}

static double decode(int dtype, uint16_t bits) {
    switch (dtype) {
        case ORACLE_BF16: return decode_bf16(bits);
        case ORACLE_E4M3: return decode_e4m3(bits);
        case ORACLE_E5M2: return decode_e5m2(bits);
        default: return decode_f16(bits);
    }
}

/*
 * Round a double to the nearest value of a binary format with `p` significand bits
 * (including the implicit one), minimum normal exponent `emin` and maximum finite
 * value `maxfin`; ties go to the even significand.  `rint` under the default rounding
 * mode is round-half-even on an exactly scaled value, so the only work here is to pick
 * the scale (the spacing of the format at |x|).
 */
static uint16_t encode_rne(double x, int p, int emin, int exp_bits, double maxfin) {
    int frac_bits = p - 1;
    int bias = (1 << (exp_bits - 1)) - 1;
    uint16_t sign = (uint16_t)(signbit(x) ? 1u << 15 : 0u);
    uint16_t exp_all_ones = (uint16_t)(((1u << exp_bits) - 1u) << frac_bits);
    if (isnan(x)) return (uint16_t)(exp_all_ones | (1u << (frac_bits - 1)));
    double a = fabs(x);
    /* Halfway between the largest finite value and the next power of two: at or above
       it the nearest-even result is infinity (the largest finite significand is odd). */
    double overflow_at = maxfin + ldexp(1.0, (int)floor(log2(maxfin)) - frac_bits - 1);
    if (a >= overflow_at) return (uint16_t)(sign | exp_all_ones);
    if (a < ldexp(1.0, emin)) {
        /* subnormal range: spacing 2^(emin - frac_bits) */
        double q = rint(ldexp(a, frac_bits - emin));
        /* q == 2^frac_bits lands exactly on the smallest normal, whose encoding is the
           same integer (exponent field 1, fraction 0). */
        return (uint16_t)(sign | (uint16_t)q);
    }
    int E;
    double fr = frexp(a, &E);          /* a = fr * 2^E, fr in [0.5, 1) */
    int unbiased = E - 1;              /* a in [2^unbiased, 2^(unbiased+1)) */
    double q = rint(ldexp(fr, p));     /* significand scaled to [2^(p-1), 2^p] */
    if (q == ldexp(1.0, p)) {          /* rounded up into the next binade */
        q = ldexp(1.0, p - 1);
        unbiased += 1;
    }
    uint32_t field = (uint32_t)(unbiased + bias);
    uint32_t frac = (uint32_t)q - (1u << frac_bits);
    return (uint16_t)(sign | (field << frac_bits) | frac);
}

/*
 * Round to FP8 with saturation to the largest finite value (the conversion a scaled FP8
 * output uses): round to nearest, ties to even, on the format's grid; magnitudes beyond
 * the largest finite value become that value; NaN stays NaN.
 */
static uint16_t encode_fp8_sat(int dtype, double x) {
    int frac_bits = dtype == ORACLE_E4M3 ? 3 : 2;
    int bias = dtype == ORACLE_E4M3 ? 7 : 15;
    int emin = 1 - bias;
    double maxfin = dtype == ORACLE_E4M3 ? 448.0 : 57344.0;
    uint16_t sign = (uint16_t)(signbit(x) ? 0x80u : 0u);
    if (isnan(x)) return (uint16_t)(dtype == ORACLE_E4M3 ? 0x7f : 0x7e);
    double a = fabs(x);
    if (a >= maxfin) a = maxfin;
    double q;
    int unbiased;
    if (a < ldexp(1.0, emin)) {
        q = rint(ldexp(a, frac_bits - emin));              /* subnormal grid 2^(emin-frac) */
        return (uint16_t)(sign | (uint16_t)q);             /* q == 2^frac is the smallest normal */
    }
    int E;
    double fr = frexp(a, &E);
    unbiased = E - 1;
    q = rint(ldexp(fr, frac_bits + 1));
    if (q == ldexp(1.0, frac_bits + 1)) {
        q = ldexp(1.0, frac_bits);
        unbiased += 1;
    }
    uint32_t bits = ((uint32_t)(unbiased + bias) << frac_bits) | ((uint32_t)q - (1u << frac_bits));
    /* rounding up past the largest finite value saturates */
    double back = ldexp(q, unbiased - frac_bits);
    if (back > maxfin) return (uint16_t)(sign | (dtype == ORACLE_E4M3 ? 0x7e : 0x7b));
    return (uint16_t)(sign | bits);
}

static uint16_t encode(int dtype, double x) {
    if (dtype == ORACLE_BF16)
        return encode_rne(x, 8, -126, 8, ldexp(255.0, 120));   /* (2 - 2^-7) * 2^127 */
    if (dtype == ORACLE_E4M3 || dtype == ORACLE_E5M2) return encode_fp8_sat(dtype, x);
    return encode_rne(x, 11, -14, 5, 65504.0);                  /* (2 - 2^-10) * 2^15 */
}

void oracle_decode(int dtype, const uint16_t* in, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = decode(dtype, in[i]);
}

void oracle_round(int dtype, const double* in, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = encode(dtype, in[i]);
}

static uint16_t a_at(const uint16_t* A, int64_t lda, int majorA, int64_t i, int64_t k) {
    return majorA == ORACLE_K_MAJOR ? A[i * lda + k] : A[i + k * lda];
}

static uint16_t b_at(const uint16_t* B, int64_t ldb, int majorB, int64_t k, int64_t j) {
    return majorB == ORACLE_K_MAJOR ? B[j * ldb + k] : B[k * ldb + j];
}

/*
 * Reference values for a set of output entries, each operand in its own format.
 *   dtA, dtB, dtC: ORACLE_F16 / ORACLE_BF16 / ORACLE_E4M3 / ORACLE_E5M2 codes, one per
 *              operand (FP8 operands are one-byte codes widened to 16 bits).  The tensor
 *              cores take FP8 operands with a 16-bit C and D ("CUTLASS, in depth", sections
 *              "Epilogue fusion" and "Numerics"); the definition of D does not change.
 *   rows/cols: n entries (i, j).  When rows == NULL the entries are all M*N outputs in
 *              row-major order (n is then ignored).
 *   ref[e]   : alpha * sum_k a(i,k) b(k,j) + beta * c(i,j)   (beta*c skipped if beta == 0)
 *   sumabs[e]: sum_k |a(i,k) * b(k,j)|  (input to the acceptance bound), may be NULL.
 *   C may be NULL when beta == 0.
 * Returns 0, or -1 on an invalid argument.
 */
int oracle_gemm_typed(int64_t M, int64_t N, int64_t K, double alpha,
                      const uint16_t* A, int64_t lda, int majorA, int dtA,
                      const uint16_t* B, int64_t ldb, int majorB, int dtB,
                      double beta, const uint16_t* C, int64_t ldc, int dtC,
                      const int64_t* rows, const int64_t* cols, int64_t n,
                      double* ref, double* sumabs, int nthreads) {
    if (M < 0 || N < 0 || K < 0) return -1;
    if (beta != 0.0 && C == NULL) return -1;
    int64_t total = rows ? n : M * N;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t e = 0; e < total; ++e) {
        int64_t i = rows ? rows[e] : e / (N ? N : 1);
        int64_t j = rows ? cols[e] : e % (N ? N : 1);
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double prod = decode(dtA, a_at(A, lda, majorA, i, k)) *
                          decode(dtB, b_at(B, ldb, majorB, k, j));
            acc += prod;
            mag += fabs(prod);
        }
        double r = alpha * acc;
        if (beta != 0.0) r += beta * decode(dtC, C[i * ldc + j]);
        ref[e] = r;
        if (sumabs) sumabs[e] = mag;
    }
    return 0;
}

/* All three operands in one format `dtype`. */
int oracle_gemm(int64_t M, int64_t N, int64_t K, double alpha,
                const uint16_t* A, int64_t lda, int majorA,
                const uint16_t* B, int64_t ldb, int majorB,
                double beta, const uint16_t* C, int64_t ldc, int dtype,
                const int64_t* rows, const int64_t* cols, int64_t n,
                double* ref, double* sumabs, int nthreads) {
    return oracle_gemm_typed(M, N, K, alpha, A, lda, majorA, dtype, B, ldb, majorB, dtype,
                             beta, C, ldc, dtype, rows, cols, n, ref, sumabs, nthreads);
}

/* E8M0 scale (OCP Microscaling): an 8-bit biased exponent, value 2^(e - 127); 0xFF is NaN. */
static double decode_e8m0(uint8_t e) {
    return e == 0xFF ? NAN : ldexp(1.0, (int)e - 127);
}

/*
 * Block-scaled ("MX") GEMM: every 32 consecutive K elements of a row of A, and of a column
 * of B, share one E8M0 scale ("CUTLASS, in depth", "Epilogue fusion": FP8 operands carry
 * per-tensor or per-block scale factors).  The operands are the FP8 codes A, B (as for
 * oracle_gemm_typed, K-major) and the scales
 *   SFA[i * ld_sfa + k / 32]  (M rows of ceil(K/32) scales),
 *   SFB[j * ld_sfb + k / 32]  (N rows of ceil(K/32) scales),
 * so that
 *   acc(i,j) = sum_k  (2^(sfa(i,k/32)-127) a(i,k)) * (2^(sfb(j,k/32)-127) b(k,j))
 *   ref(i,j) = alpha*acc + beta*c(i,j)
 * with k in order and every product and sum in double.  sumabs as for oracle_gemm_typed,
 * of the scaled products.
 */
int oracle_gemm_mx(int64_t M, int64_t N, int64_t K, double alpha,
                   const uint16_t* A, int64_t lda, int dtA, const uint8_t* SFA, int64_t ld_sfa,
                   const uint16_t* B, int64_t ldb, int dtB, const uint8_t* SFB, int64_t ld_sfb,
                   double beta, const uint16_t* C, int64_t ldc, int dtC,
                   const int64_t* rows, const int64_t* cols, int64_t n,
                   double* ref, double* sumabs, int nthreads) {
    if (M < 0 || N < 0 || K < 0) return -1;
    if (beta != 0.0 && C == NULL) return -1;
    if (K > 0 && (SFA == NULL || SFB == NULL)) return -1;
    int64_t total = rows ? n : M * N;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t e = 0; e < total; ++e) {
        int64_t i = rows ? rows[e] : e / (N ? N : 1);
        int64_t j = rows ? cols[e] : e % (N ? N : 1);
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = decode_e8m0(SFA[i * ld_sfa + k / 32]) * decode(dtA, A[i * lda + k]);
            double b = decode_e8m0(SFB[j * ld_sfb + k / 32]) * decode(dtB, B[j * ldb + k]);
            double prod = a * b;
            acc += prod;
            mag += fabs(prod);
        }
        double r = alpha * acc;
        if (beta != 0.0) r += beta * decode(dtC, C[i * ldc + j]);
        ref[e] = r;
        if (sumabs) sumabs[e] = mag;
    }
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
