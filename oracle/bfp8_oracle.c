/*
 * Blockwise-scaled FP8 oracle: a plain, slow, CPU-only restatement of what the
 * blockwise FP8 dense-training path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code, header, table or
 * constant with the CUDA path; it is compiled with plain gcc
 * (-O2 -ffp-contract=off, no fast-math) so that every float operation below is
 * one IEEE-754 operation rounded to nearest-even.
 *
 * Sources (pytorch/ao pull-request pages):
 *   [P1] "Mask a_s/b_s scale loads in blockwise FP8 training GEMM kernels",
 *        Summary and Fix: the two GEMMs (1x128 x 128x128, 1x128 x 128x1),
 *        per-tile a_s/b_s scales, every load and the output store masked to
 *        offs_m < M / offs_n < N.
 *   [P2] "Enable blockwise FP8 dense training kernels on ROCm": the three
 *        quantizations act_quant_lhs (1x128), act_quant_rhs (128x1) and
 *        weight_quant_rhs (128x128) with block_size=128 (correctness table);
 *        FP8_MAX = 448 for float8_e4m3fn (summary); the lhs scale tensor is
 *        column-major and its store must be masked to m < M (root-cause
 *        comment); GEMM SQNR against a BF16 matmul (GEMM correctness table).
 *   Method statement used for the formulas: scale s = amax / 448,
 *   q = round-to-nearest-even-to-e4m3(clamp(x / s, -448, 448)); GEMM output
 *   C = sum over 128-wide K-blocks of (a_s * b_s) * (FP8 partial product),
 *   accumulated per K-block.
 *
 * Readings taken where the pages are silent (each one is listed in the design
 * notes of the repository):
 *   R1  the stored scale is the dequantisation multiplier s = fl32(amax/448),
 *       computed by one division; quantisation divides by s (one division).
 *   R2  an all-zero group would give s = 0 and 0/0; amax is floored at 1e-12
 *       first, so such a group stores s = fl32(1e-12/448) and codes 0x00/0x80.
 *   R3  a tail group (K, M or N not a multiple of 128) takes its amax over its
 *       in-range elements only; nothing outside the logical tensor is written.
 *   R4  the e4m3 rounding keeps the sign of zero: a negative value that rounds
 *       to zero gives 0x80.
 *   R5  the GEMM result is kept in double: per K-block partial sums are exact
 *       double sums of exact e4m3 products, then scaled by (double)a_s*b_s.
 *   R14 MXFP8 ([P3] "Fixes accuracy error for mxfp8 linear": the mxfp8 linear,
 *       its dim1 cast kernel and ScaleCalculationMode.FLOOR) follows the OCP
 *       Microscaling Formats v1.0 definition, which the page does not spell
 *       out: blocks of 32 elements, one E8M0 scale 2^e per block with
 *       e = floor(log2(amax)) - 8 (8 = the exponent of 448, E4M3's largest
 *       normal), clamped to [-127, 127] (e = -127 for an all-zero block),
 *       stored biased as e + 127; codes RNE_e4m3(clamp(fl32(x * 2^-e), +-448)).
 *       The dim0 cast groups 32 consecutive elements of a row; the dim1 cast
 *       groups 32 consecutive elements of a column and writes codes and
 *       scales transposed (the dim0 cast of the transpose).
 *
 * Parity pins (tests/test_oracle_pins.py) tie every function here to facts the
 * pages or the mathematics fix; no function is "parity unpinned".
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_BLOCK 128           /* group / tile edge, block_size=128 [P2] */
#define ORA_E4M3_MAX 448.0f     /* FP8_MAX of float8_e4m3fn [P2 summary] */
#define ORA_AMAX_FLOOR 1e-12f   /* reading R2 */

static int64_t ora_ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* ---------------------------------------------------------------------- */
/* Number formats                                                          */
/* ---------------------------------------------------------------------- */

/* bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits. */
float ora_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * Exact value of an OCP FP8 E4M3 ("e4m3fn") code: 1 sign bit, 4 exponent bits
 * (bias 7), 3 mantissa bits, no infinities, S.1111.111 is NaN.
 * Normal: (1 + m/8) * 2^(e-7) for e >= 1; subnormal: (m/8) * 2^-6 for e == 0.
 */
double ora_e4m3_value(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/*
 * Round an fp32 value to e4m3fn, ties to even, after clamping to [-448, 448]
 * (the method's q = RNE(clamp(x/s, +-448))).  Written from the format's
 * definition: find the binade of |r|, the spacing (quantum) of e4m3 values in
 * it, and round |r|/quantum to the nearest integer with ties to even.  All
 * arithmetic is exact in double (|r| has 24 significant bits and the quantum
 * is a power of two).
 */
uint8_t ora_e4m3_rne(float r) {
    uint32_t bits;
    memcpy(&bits, &r, sizeof bits);
    uint8_t sign = (uint8_t)((bits >> 31) << 7);       /* R4: keep the sign of 0 */
    double a = fabs((double)r);
    if (a > (double)ORA_E4M3_MAX) a = (double)ORA_E4M3_MAX; /* the clamp */

    int e;           /* binade exponent: 2^e <= a < 2^(e+1), e >= -6 */
    double quantum;  /* spacing of e4m3 values in that binade */
    if (a < ldexp(1.0, -6)) {
        e = -6;                        /* subnormal binade shares exponent -6 */
        quantum = ldexp(1.0, -9);      /* min subnormal 2^-9 */
    } else {
        e = (int)floor(log2(a));
        if (ldexp(1.0, e) > a) e -= 1;       /* guard log2 rounding */
        if (ldexp(1.0, e + 1) <= a) e += 1;
        quantum = ldexp(1.0, e - 3);   /* 3 mantissa bits */
    }
    double n = a / quantum;            /* exact: power-of-two division */
    double fl = floor(n);
    double frac = n - fl;
    double k = fl;
    if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0)) k = fl + 1.0;
    /* k counts quanta: magnitude = k * quantum */
    int ki = (int)k;
    uint8_t mag;
    if (a < ldexp(1.0, -6)) {
        /* subnormal: code = k (k == 8 is exactly the smallest normal 0x08) */
        mag = (uint8_t)ki;
    } else {
        if (ki == 16) { e += 1; ki = 8; }  /* rounded up into the next binade */
        mag = (uint8_t)(((e + 7) << 3) | (ki - 8));
    }
    return (uint8_t)(sign | mag);
}

/*
 * Independent check of ora_e4m3_rne: brute-force nearest finite e4m3 value of
 * the same sign, ties broken toward the code with an even mantissa.
 * Shares nothing with ora_e4m3_rne except ora_e4m3_value.
 */
uint8_t ora_e4m3_nearest(float r) {
    uint32_t bits;
    memcpy(&bits, &r, sizeof bits);
    uint8_t sign = (uint8_t)((bits >> 31) << 7);
    double a = fabs((double)r);
    if (a > 448.0) a = 448.0;
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(ora_e4m3_value((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best_d = d;
            best = c;
        }
    }
    return (uint8_t)(sign | best);
}

/* Sorted magnitudes of the 127 non-negative finite codes, for a fast but still
 * independent nearest search used by the exhaustive sweep. */
static double ora_mag_table[127];
static void ora_build_mag_table(void) {
    for (int c = 0; c <= 0x7E; ++c) ora_mag_table[c] = ora_e4m3_value((uint8_t)c);
}

static uint8_t ora_nearest_bsearch(float r) {
    uint32_t bits;
    memcpy(&bits, &r, sizeof bits);
    uint8_t sign = (uint8_t)((bits >> 31) << 7);
    double a = fabs((double)r);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    /* largest c with table[c] <= a (codes are monotone in magnitude) */
    int lo = 0, hi = 0x7E;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (ora_mag_table[mid] <= a) lo = mid; else hi = mid - 1;
    }
    int c = lo;
    if (ora_mag_table[c] == a) return (uint8_t)(sign | c);
    double dlo = a - ora_mag_table[c];
    double dhi = ora_mag_table[c + 1] - a;
    int pick = (dlo < dhi) ? c : (dhi < dlo) ? c + 1 : ((c & 1) == 0 ? c : c + 1);
    return (uint8_t)(sign | pick);
}

/* ---------------------------------------------------------------------- */
/* Exhaustive cast sweep (pins ora_e4m3_rne against the nearest search)     */
/* ---------------------------------------------------------------------- */

typedef struct {
    uint64_t lo, hi;      /* fp32 bit patterns [lo, hi) */
    uint64_t mismatches;
    uint64_t first_bad;
} ora_sweep_job;

static void *ora_sweep_worker(void *arg) {
    ora_sweep_job *j = (ora_sweep_job *)arg;
    for (uint64_t b = j->lo; b < j->hi; ++b) {
        uint32_t u = (uint32_t)b;
        float r;
        memcpy(&r, &u, sizeof r);
        if (r != r) continue; /* NaN inputs are outside the method's domain */
        uint8_t x = ora_e4m3_rne(r), y = ora_nearest_bsearch(r);
        if (x != y) {
            if (j->mismatches == 0) j->first_bad = b;
            j->mismatches++;
        }
    }
    return NULL;
}

/* Compare ora_e4m3_rne with the nearest-code search on every fp32 bit pattern
 * in [lo, hi), with `stride` between patterns.  Returns the mismatch count and
 * writes the first mismatching pattern to *first_bad. */
uint64_t ora_sweep_cast(uint64_t lo, uint64_t hi, int nthreads, uint64_t *first_bad) {
    ora_build_mag_table();
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    ora_sweep_job jobs[256];
    uint64_t span = hi - lo, per = (span + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].lo = lo + per * t < hi ? lo + per * t : hi;
        jobs[t].hi = lo + per * (t + 1) < hi ? lo + per * (t + 1) : hi;
        jobs[t].mismatches = 0;
        jobs[t].first_bad = 0;
        pthread_create(&th[t], NULL, ora_sweep_worker, &jobs[t]);
    }
    uint64_t total = 0;
    *first_bad = 0;
    for (int t = 0; t < nthreads; ++t) {
        pthread_join(th[t], NULL);
        if (jobs[t].mismatches && total == 0) *first_bad = jobs[t].first_bad;
        total += jobs[t].mismatches;
    }
    return total;
}

/* Elementwise cast of n fp32 values (used to compare the device's rounding
 * step against this definition over large sweeps). */
typedef struct { const float *x; uint8_t *q; int64_t lo, hi; } ora_cast_job;
static void *ora_cast_worker(void *arg) {
    ora_cast_job *j = (ora_cast_job *)arg;
    for (int64_t i = j->lo; i < j->hi; ++i) j->q[i] = ora_e4m3_rne(j->x[i]);
    return NULL;
}
void ora_cast_e4m3(const float *x, int64_t n, uint8_t *q, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    ora_cast_job jobs[256];
    int64_t per = (n + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].x = x; jobs[t].q = q;
        jobs[t].lo = per * t < n ? per * t : n;
        jobs[t].hi = per * (t + 1) < n ? per * (t + 1) : n;
        pthread_create(&th[t], NULL, ora_cast_worker, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* Compare a caller-supplied byte array (e.g. produced by another
 * implementation) with ora_e4m3_rne over the fp32 bit patterns
 * start, start+1, ..., start+n-1.  Returns the mismatch count (NaN patterns
 * are skipped) and the first mismatching pattern in *first_bad. */
typedef struct { uint64_t start; const uint8_t *got; int64_t lo, hi; uint64_t bad, first; } ora_cmp_job;
static void *ora_cmp_worker(void *arg) {
    ora_cmp_job *j = (ora_cmp_job *)arg;
    for (int64_t i = j->lo; i < j->hi; ++i) {
        uint32_t u = (uint32_t)(j->start + (uint64_t)i);
        float r;
        memcpy(&r, &u, sizeof r);
        if (r != r) continue;
        if (j->got[i] != ora_e4m3_rne(r)) {
            if (j->bad == 0) j->first = (uint64_t)u;
            j->bad++;
        }
    }
    return NULL;
}
uint64_t ora_check_cast_range(uint64_t start, int64_t n, const uint8_t *got, int nthreads,
                              uint64_t *first_bad) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    ora_cmp_job jobs[256];
    int64_t per = (n + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].start = start; jobs[t].got = got; jobs[t].bad = 0; jobs[t].first = 0;
        jobs[t].lo = per * t < n ? per * t : n;
        jobs[t].hi = per * (t + 1) < n ? per * (t + 1) : n;
        pthread_create(&th[t], NULL, ora_cmp_worker, &jobs[t]);
    }
    uint64_t total = 0;
    *first_bad = 0;
    for (int t = 0; t < nthreads; ++t) {
        pthread_join(th[t], NULL);
        if (jobs[t].bad && total == 0) *first_bad = jobs[t].first;
        total += jobs[t].bad;
    }
    return total;
}

/* ---------------------------------------------------------------------- */
/* Quantisation                                                            */
/* ---------------------------------------------------------------------- */

/* s = fl32(max(amax, 1e-12) / 448)  (method formula, readings R1 and R2) */
float ora_group_scale(float amax) {
    float a = amax;
    if (a < ORA_AMAX_FLOOR) a = ORA_AMAX_FLOOR;
    return a / ORA_E4M3_MAX;
}

/* q = RNE_e4m3(clamp(fl32(x / s), +-448)) */
uint8_t ora_quantize_one(float x, float s) {
    float r = x / s;
    return ora_e4m3_rne(r);
}

/* ---------------------------------------------------------------------- */
/* MXFP8 casts (reading R14)                                               */
/* ---------------------------------------------------------------------- */

#define ORA_MX_BLOCK 32

/* e = floor(log2(amax)) - 8 clamped to [-127, 127]; -127 for amax == 0.
 * frexpf gives amax = f * 2^ex with f in [0.5, 1), so floor(log2(amax)) = ex - 1
 * for every positive finite amax, subnormals included. */
int ora_mx_exponent(float amax) {
    if (!(amax > 0.0f)) return -127;
    int ex;
    (void)frexpf(amax, &ex);
    int e = (ex - 1) - 8;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* q = RNE_e4m3(clamp(fl32(x * 2^-e), +-448)): one fp32 multiplication by a
 * power of two (exact unless the product falls below the normal range). */
uint8_t ora_mx_quantize_one(float x, int e) {
    return ora_e4m3_rne(x * ldexpf(1.0f, -e));
}

/*
 * MXFP8 cast of x [M,K] (bf16, row stride ldx).
 *   dim0 (q0 != NULL): blocks of 32 along K; q0[m * ldq0 + k], biased
 *        exponents e0[m * lde0 + k / 32] (lde0 >= ceil(K/32)).
 *   dim1 (q1 != NULL): blocks of 32 along M, written transposed:
 *        q1[k * ldq1 + m], e1[k * lde1 + m / 32] (lde1 >= ceil(M/32)).
 * A tail block takes its amax over its in-range elements; nothing else is written.
 */
void ora_mx_cast(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                 uint8_t *q0, int64_t ldq0, uint8_t *e0, int64_t lde0,
                 uint8_t *q1, int64_t ldq1, uint8_t *e1, int64_t lde1) {
    if (q0) {
        for (int64_t m = 0; m < M; ++m)
            for (int64_t k0 = 0; k0 < K; k0 += ORA_MX_BLOCK) {
                int64_t k1 = k0 + ORA_MX_BLOCK < K ? k0 + ORA_MX_BLOCK : K;
                float amax = 0.0f;
                for (int64_t k = k0; k < k1; ++k) {
                    float v = fabsf(ora_bf16_to_f32(x[m * ldx + k]));
                    if (v > amax) amax = v;
                }
                int e = ora_mx_exponent(amax);
                e0[m * lde0 + k0 / ORA_MX_BLOCK] = (uint8_t)(e + 127);
                for (int64_t k = k0; k < k1; ++k)
                    q0[m * ldq0 + k] = ora_mx_quantize_one(ora_bf16_to_f32(x[m * ldx + k]), e);
            }
    }
    if (q1) {
        for (int64_t k = 0; k < K; ++k)
            for (int64_t m0 = 0; m0 < M; m0 += ORA_MX_BLOCK) {
                int64_t m1 = m0 + ORA_MX_BLOCK < M ? m0 + ORA_MX_BLOCK : M;
                float amax = 0.0f;
                for (int64_t m = m0; m < m1; ++m) {
                    float v = fabsf(ora_bf16_to_f32(x[m * ldx + k]));
                    if (v > amax) amax = v;
                }
                int e = ora_mx_exponent(amax);
                e1[k * lde1 + m0 / ORA_MX_BLOCK] = (uint8_t)(e + 127);
                for (int64_t m = m0; m < m1; ++m)
                    q1[k * ldq1 + m] = ora_mx_quantize_one(ora_bf16_to_f32(x[m * ldx + k]), e);
            }
    }
}

/*
 * act_quant_lhs [P2]: A[M,K] is quantised in 1x128 groups along K (one group =
 * one row m and 128 consecutive k).  Scales are stored column-major
 * s[kb * lds + m], lds >= M [P2 root-cause comment]; only rows m < M are
 * written [P2 fix].
 *   transposed == 0: A[m,k] = x[m * ldx + k]  (x is [M,K] row-major)
 *   transposed == 1: A[m,k] = x[k * ldx + m]  (x is [K,M] row-major; this is
 *                    the dY^T operand of the weight-gradient GEMM)
 * q[m * ldq + k] for k < K; bytes k in [K, ldq) are not written.
 */
void ora_quant_lhs(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int transposed,
                   uint8_t *q, int64_t ldq, float *s, int64_t lds) {
    int64_t Kb = ora_ceil_div(K, ORA_BLOCK);
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < Kb; ++kb) {
            int64_t k0 = kb * ORA_BLOCK;
            int64_t k1 = k0 + ORA_BLOCK < K ? k0 + ORA_BLOCK : K;
            float amax = 0.0f;
            for (int64_t k = k0; k < k1; ++k) {
                float v = ora_bf16_to_f32(transposed ? x[k * ldx + m] : x[m * ldx + k]);
                if (fabsf(v) > amax) amax = fabsf(v);
            }
            float sc = ora_group_scale(amax);
            s[kb * lds + m] = sc;
            for (int64_t k = k0; k < k1; ++k) {
                float v = ora_bf16_to_f32(transposed ? x[k * ldx + m] : x[m * ldx + k]);
                q[m * ldq + k] = ora_quantize_one(v, sc);
            }
        }
    }
}

/*
 * act_quant_rhs [P2]: X[K,N] (K = the reduction dimension of the GEMM that
 * consumes it) is quantised in 128x1 groups: one column n and 128 consecutive
 * rows k.  The bytes are written transposed, qT[n * ldq + k], so that the GEMM
 * reads them K-major; scales are s[kb * lds + n] (row-major [Kb, N], lds >= N).
 */
void ora_quant_rhs(const uint16_t *x, int64_t K, int64_t N, int64_t ldx,
                   uint8_t *qT, int64_t ldq, float *s, int64_t lds) {
    int64_t Kb = ora_ceil_div(K, ORA_BLOCK);
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t kb = 0; kb < Kb; ++kb) {
            int64_t k0 = kb * ORA_BLOCK;
            int64_t k1 = k0 + ORA_BLOCK < K ? k0 + ORA_BLOCK : K;
            float amax = 0.0f;
            for (int64_t k = k0; k < k1; ++k) {
                float v = ora_bf16_to_f32(x[k * ldx + n]);
                if (fabsf(v) > amax) amax = fabsf(v);
            }
            float sc = ora_group_scale(amax);
            s[kb * lds + n] = sc;
            for (int64_t k = k0; k < k1; ++k)
                qT[n * ldq + k] = ora_quantize_one(ora_bf16_to_f32(x[k * ldx + n]), sc);
        }
    }
}

/*
 * weight_quant_rhs [P2]: W[N,K] is quantised in 128x128 tiles, one scale per
 * tile, s[nb * lds + kb] (row-major [Nb, Kb], lds >= Kb).  q[n * ldq + k];
 * if qt is not NULL the same bytes are also written transposed,
 * qt[k * ldqt + n], for the input-gradient GEMM.
 */
void ora_quant_weight(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                      uint8_t *q, int64_t ldq, uint8_t *qt, int64_t ldqt,
                      float *s, int64_t lds) {
    int64_t Nb = ora_ceil_div(N, ORA_BLOCK), Kb = ora_ceil_div(K, ORA_BLOCK);
    for (int64_t nb = 0; nb < Nb; ++nb) {
        for (int64_t kb = 0; kb < Kb; ++kb) {
            int64_t n0 = nb * ORA_BLOCK, n1 = n0 + ORA_BLOCK < N ? n0 + ORA_BLOCK : N;
            int64_t k0 = kb * ORA_BLOCK, k1 = k0 + ORA_BLOCK < K ? k0 + ORA_BLOCK : K;
            float amax = 0.0f;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = k0; k < k1; ++k) {
                    float v = ora_bf16_to_f32(w[n * ldw + k]);
                    if (fabsf(v) > amax) amax = fabsf(v);
                }
            float sc = ora_group_scale(amax);
            s[nb * lds + kb] = sc;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = k0; k < k1; ++k) {
                    uint8_t c = ora_quantize_one(ora_bf16_to_f32(w[n * ldw + k]), sc);
                    q[n * ldq + k] = c;
                    if (qt) qt[k * ldqt + n] = c;
                }
        }
    }
}

/* ---------------------------------------------------------------------- */
/* GEMM                                                                    */
/* ---------------------------------------------------------------------- */

/* How the B-side scale of output column n and K-block kb is addressed. */
enum {
    ORA_SB_TILE = 0,      /* 128x128 weight tiles, sb[(n/128) * ldsb + kb]  */
    ORA_SB_TILE_T = 1,    /* the same tiles read transposed, sb[kb * ldsb + n/128] */
    ORA_SB_COL = 2        /* 128x1 groups, sb[kb * ldsb + n]                 */
};

typedef struct {
    const uint8_t *qa; int64_t lda; const float *sa; int64_t ldsa;
    const uint8_t *qb; int64_t ldb; const float *sb; int64_t ldsb; int sb_mode;
    int64_t K;
    const int64_t *rows; int64_t nrows; const int64_t *cols; int64_t ncols;
    double *out;
    int64_t r_lo, r_hi;
    const double *deq;
} ora_gemm_job;

static void *ora_gemm_worker(void *arg) {
    ora_gemm_job *j = (ora_gemm_job *)arg;
    int64_t Kb = ora_ceil_div(j->K, ORA_BLOCK);
    for (int64_t ri = j->r_lo; ri < j->r_hi; ++ri) {
        int64_t m = j->rows[ri];
        const uint8_t *arow = j->qa + m * j->lda;
        for (int64_t ci = 0; ci < j->ncols; ++ci) {
            int64_t n = j->cols[ci];
            const uint8_t *brow = j->qb + n * j->ldb;
            double c = 0.0;
            for (int64_t kb = 0; kb < Kb; ++kb) {
                int64_t k0 = kb * ORA_BLOCK;
                int64_t k1 = k0 + ORA_BLOCK < j->K ? k0 + ORA_BLOCK : j->K;
                double partial = 0.0; /* the K-block's FP8 partial product */
                for (int64_t k = k0; k < k1; ++k) partial += j->deq[arow[k]] * j->deq[brow[k]];
                double a_s = (double)j->sa[kb * j->ldsa + m];
                double b_s;
                if (j->sb_mode == ORA_SB_TILE) b_s = (double)j->sb[(n / ORA_BLOCK) * j->ldsb + kb];
                else if (j->sb_mode == ORA_SB_TILE_T) b_s = (double)j->sb[kb * j->ldsb + n / ORA_BLOCK];
                else b_s = (double)j->sb[kb * j->ldsb + n];
                c += (a_s * b_s) * partial; /* promotion of the K-block */
            }
            j->out[ri * j->ncols + ci] = c;
        }
    }
    return NULL;
}

/*
 * Blockwise-scaled FP8 GEMM [P1 Summary]: for output C[M,N] = A[M,K] B[K,N]
 *   C[m,n] = sum_kb a_s[m,kb] * b_s(n,kb) * sum_{k in kb, k < K} A[m,k] B[k,n]
 * with A = deq(qa[m * lda + k]), B[k,n] = deq(qb[n * ldb + k]) (B given as
 * [N,K], K contiguous), a_s column-major sa[kb * ldsa + m] (1x128 groups) and
 * b_s addressed per sb_mode (128x128 tiles, or 128x1 groups).
 * Computes C only at rows[0..nrows) x cols[0..ncols) into
 * out[ri * ncols + ci], in double (reading R5).
 */
void ora_gemm(const uint8_t *qa, int64_t lda, const float *sa, int64_t ldsa,
              const uint8_t *qb, int64_t ldb, const float *sb, int64_t ldsb, int sb_mode,
              int64_t K, const int64_t *rows, int64_t nrows, const int64_t *cols, int64_t ncols,
              double *out, int nthreads) {
    double deq[256];
    for (int c = 0; c < 256; ++c) deq[c] = ora_e4m3_value((uint8_t)c);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > nrows) nthreads = nrows > 0 ? (int)nrows : 1;
    pthread_t th[256];
    ora_gemm_job jobs[256];
    int64_t per = (nrows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        ora_gemm_job *j = &jobs[t];
        j->qa = qa; j->lda = lda; j->sa = sa; j->ldsa = ldsa;
        j->qb = qb; j->ldb = ldb; j->sb = sb; j->ldsb = ldsb; j->sb_mode = sb_mode;
        j->K = K; j->rows = rows; j->nrows = nrows; j->cols = cols; j->ncols = ncols;
        j->out = out; j->deq = deq;
        j->r_lo = per * t < nrows ? per * t : nrows;
        j->r_hi = per * (t + 1) < nrows ? per * (t + 1) : nrows;
        pthread_create(&th[t], NULL, ora_gemm_worker, j);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* SQNR = 20 log10(||ref|| / ||ref - out||)  [P2 GEMM correctness table] */
double ora_sqnr_db(const double *ref, const double *out, int64_t n) {
    double num = 0.0, den = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        num += ref[i] * ref[i];
        double d = ref[i] - out[i];
        den += d * d;
    }
    return 10.0 * log10(num / den);
}

/* Plain fp64 matmul of bf16 inputs, C = X W^T with X [M,K], W [N,K]: the
 * high-precision reference the SQNR is measured against. */
void ora_matmul_bf16_f64(const uint16_t *x, int64_t ldx, const uint16_t *w, int64_t ldw,
                         int64_t M, int64_t N, int64_t K, double *out) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double c = 0.0;
            for (int64_t k = 0; k < K; ++k)
                c += (double)ora_bf16_to_f32(x[m * ldx + k]) * (double)ora_bf16_to_f32(w[n * ldw + k]);
            out[m * N + n] = c;
        }
}
