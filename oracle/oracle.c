/*
 * Plain CPU oracle for the block-scaled MXFP4 GEMM (and its MXFP8 form).
 *
 *     D[M,N] (bf16) = alpha * A[M,K] (mxfp4) * B[N,K]^T (mxfp4) + beta * C[M,N]
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * CPU-baseline leg of the benchmark may load this file.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * It is written from the page "asm_f4gemm -- driving aiter's gfx950 MXFP4
 * GEMM code objects":
 *   - the GEMM formula at the top of the page;
 *   - section "Data layouts": A/B are [rows, K/2] bytes, element 2i in the low
 *     nibble and 2i+1 in the high nibble, E2M1 magnitudes {0,.5,1,1.5,2,3,4,6}
 *     with the sign in bit 3; E8M0 value = 2^(e-127), one scale per 32 K;
 *   - section "Verification": the reference accumulates in double over the
 *     dequantised operands, and the only error left is the bf16 rounding.
 * And from the page "CDNA4 dense MFMA builtins", section "Mixed-precision with
 * scaling": each per-block scale is applied to the inputs before they are
 * accumulated.
 *
 * Steps, in the order the definition gives them:
 *   1. unpack the nibble of element k (low nibble for even k);
 *   2. decode it with the page's value list and sign bit;
 *   3. decode the block's E8M0 scale as 2^(e-127);
 *   4. accumulate a(m,k) * b(n,k) in double, in k order;
 *   5. y = alpha * acc + beta * C[m][n] in double;
 *   6. round y once, straight from double, to bf16 (nearest, ties to even).
 *
 * Exactness: every product is an integer multiple of 2^(ea+eb-256) (E2M1
 * values are multiples of 1/2), so the double sum is exact, in any order,
 * whenever sum|a*b| / min-granule < 2^52.  The oracle checks that bound for
 * every output and checks with an exact product/sum test that step 5 did not
 * round; outputs that fail either check are counted and reported.
 *
 * MXFP8 / MXFP6 form (oracle_gemm8): the same steps with one 8-bit E4M3 or
 * E5M2 element per byte, or E2M3 / E3M2 elements in the padded 6-bit form
 * (oracle_fp8_value_q and oracle_fp6_value_q give the encodings read from
 * the MFMA page).  A product's granule is 2^(qa + qb + ea + eb - 254), where
 * qa, qb are the elements' ulp exponents, and the same 2^52 bound applies.
 *
 * NVFP4 form (oracle_gemm_nv): packed E2M1 elements as in MXFP4 with one
 * UE4M3 scale per 16 K (oracle_ue4m3_value_q).  The pages do not cover this
 * format; it follows the E4M3 encoding already read for MXFP8 elements.  A
 * product's granule is 2^(qa + qb + sa_q + sb_q) with the scales' ulp
 * exponents, under the same 2^52 bound.
 *
 * Readings where the pages are silent or at odds:
 *   - E8M0 code 0: the page writes both 2^(e-127) and "0 -> 2^-126"; the
 *     formula is taken (code 0 -> 2^-127).  Code 255 decodes to NaN.
 *   - D is rounded to nearest, ties to even (the MFMA page's rounding mode).
 *   - C is bf16.  C is not read when beta == 0 (it may be NULL).
 *   - FP8 / BF8 biases and special codes: the OCP 8-bit formats (the page
 *     gives the field widths only); see oracle_fp8_value_q.  FP6 likewise:
 *     the OCP 6-bit formats (oracle_fp6_value_q), stored 16 codes per 16
 *     bytes (oracle_fp6_code).
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* Step 2: the E2M1 magnitudes in the order the page lists them, indexed by
 * bits 2..0 of the code; bit 3 is the sign. */
static const double kE2M1Magnitude[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_value(unsigned code)
{
    double mag = kE2M1Magnitude[code & 7u];
    return (code & 8u) ? -mag : mag;
}

/* Step 3: E8M0 is a bare biased exponent. */
double oracle_e8m0_value(unsigned code)
{
    code &= 0xFFu;
    if (code == 0xFFu)
        return NAN;
    return ldexp(1.0, (int)code - 127);
}

/*
 * MXFP8 elements (page "CDNA4 dense MFMA builtins", section "FP8 and BF8
 * matrix inputs": FP8 is E4M3 = 1 sign, 4 exponent, 3 mantissa bits; BF8 is
 * E5M2 = 1, 5, 2; section "Mixed-precision with scaling": the scaled
 * builtins take either with one scale per block).  The pages give the field
 * widths only; the encodings read here are the OCP 8-bit formats those
 * builtins use: E4M3 with bias 7, no infinities and NaN at S.1111.111
 * (largest 448); E5M2 with bias 15, infinities at S.11111.00 and NaN at
 * S.11111.{01,10,11} (largest 57344).  Exponent field 0 is subnormal:
 * (m / 2^mbits) * 2^(1 - bias).
 *
 * fmt: 1 = E4M3, 2 = E5M2.  *ulp_exp (optional) receives q such that the value
 * is an integer multiple of 2^q (the spacing of its binade).
 */
double oracle_fp8_value_q(unsigned code, int fmt, int *ulp_exp)
{
    const int ebits = fmt == 1 ? 4 : 5, mbits = fmt == 1 ? 3 : 2, bias = fmt == 1 ? 7 : 15;
    const unsigned s = (code >> 7) & 1u;
    const unsigned e = (code >> mbits) & ((1u << ebits) - 1u);
    const unsigned m = code & ((1u << mbits) - 1u);
    const unsigned emax = (1u << ebits) - 1u;
    double v;
    if (fmt == 1 && e == emax && m == (1u << mbits) - 1u)
        v = NAN;
    else if (fmt == 2 && e == emax)
        v = m == 0 ? INFINITY : NAN;
    else {
        const int ee = e == 0 ? 1 : (int)e;
        const double frac = (e == 0 ? 0.0 : 1.0) + ldexp((double)m, -mbits);
        v = ldexp(frac, ee - bias);
    }
    if (ulp_exp)
        *ulp_exp = (e == 0 ? 1 : (int)e) - bias - mbits;
    return s ? -v : v;
}

double oracle_fp8_value(unsigned code, int fmt)
{
    return oracle_fp8_value_q(code, fmt, NULL);
}

/*
 * NVFP4 block scales (a member of the block-scaled family beyond the pages:
 * packed E2M1 elements as in the MXFP4 GEMM, one scale per 16 consecutive K
 * elements instead of 32).  The scale byte is unsigned E4M3 ("UE4M3"): the
 * E4M3 encoding of the MXFP8 elements above with the sign bit 0, so
 * (1 + m/8) * 2^(e-7), exponent field 0 subnormal (m/8) * 2^-6, and 0x7F
 * NaN.  A byte with bit 7 set is not a UE4M3 code: NaN here, and the GEMM
 * entry points below reject it.  *ulp_exp as for oracle_fp8_value_q.
 */
double oracle_ue4m3_value_q(unsigned code, int *ulp_exp)
{
    code &= 0xFFu;
    if (code & 0x80u) {
        if (ulp_exp)
            *ulp_exp = 0;
        return NAN;
    }
    return oracle_fp8_value_q(code, 1, ulp_exp);
}

double oracle_ue4m3_value(unsigned code)
{
    return oracle_ue4m3_value_q(code, NULL);
}

/*
 * MXFP6 elements (page "CDNA4 dense MFMA builtins", section "Mixed-precision
 * with scaling": FP6 is E2M3 or E3M2, 6 bits per element, scaled per block
 * like the others).  The pages give the field widths only; the encodings
 * read here are the OCP 6-bit formats: E2M3 with bias 1 (largest 7.5), E3M2
 * with bias 3 (largest 28), no infinities or NaNs, exponent field 0
 * subnormal: (m / 2^mbits) * 2^(1 - bias).  Bit 5 is the sign.
 *
 * fmt: 3 = E2M3, 4 = E3M2.  *ulp_exp as for oracle_fp8_value_q.
 */
double oracle_fp6_value_q(unsigned code, int fmt, int *ulp_exp)
{
    const int ebits = fmt == 3 ? 2 : 3, mbits = fmt == 3 ? 3 : 2, bias = fmt == 3 ? 1 : 3;
    const unsigned s = (code >> 5) & 1u;
    const unsigned e = (code >> mbits) & ((1u << ebits) - 1u);
    const unsigned m = code & ((1u << mbits) - 1u);
    /* Integer significand (the implicit 1 only for a non-zero exponent
     * field) times the binade's spacing. */
    const unsigned sig = e == 0 ? m : (m | (1u << mbits));
    const int q = (e == 0 ? 1 : (int)e) - bias - mbits;
    const double v = ldexp((double)sig, q);
    if (ulp_exp)
        *ulp_exp = q;
    return s ? -v : v;
}

double oracle_fp6_value(unsigned code, int fmt)
{
    return oracle_fp6_value_q(code, fmt, NULL);
}

/*
 * FP6 storage: the rows hold K bytes, 16 bytes per 16 consecutive elements:
 * the 16 codes packed little-endian (element i of the group in bits 6i ..
 * 6i+5 of the first 12 bytes) and 4 bytes of padding that are not read.
 * This is the operand form the scaled tensor-core instruction reads, so the
 * GEMM loads it as bytes; the pages' own FP6 operands are packed 6-bit
 * register fragments.
 */
unsigned oracle_fp6_code(const uint8_t *row, int64_t k)
{
    const uint8_t *g = row + (k >> 4) * 16;
    const int bit = 6 * (int)(k & 15);
    const unsigned two = (unsigned)g[bit >> 3] | ((unsigned)g[(bit >> 3) + 1] << 8);
    return (two >> (bit & 7)) & 63u;
}

/*
 * E2M1 in the same padded form (fmt 5): every 16 elements take 16 bytes, the
 * first 8 holding two codes each -- element 2i of the group in the low
 * nibble of byte i, element 2i+1 in its high nibble, the order of the packed
 * MXFP4 rows -- and 8 padding bytes that are not read.  This lets E2M1 be
 * mixed with the 8- and 6-bit formats, which the page's scaled builtins
 * allow (A and B formats chosen independently).
 */
unsigned oracle_fp4_padded_code(const uint8_t *row, int64_t k)
{
    const unsigned pair = row[(k >> 4) * 16 + ((k & 15) >> 1)];
    return (k & 1) ? pair >> 4 : pair & 15u;
}

/* Any element format of the one-byte-footprint forms (fmt 1-5). */
static double byte_form_value(const uint8_t *row, int64_t k, int fmt, int *q)
{
    if (fmt == 5) {
        *q = -1;                       /* E2M1 values are multiples of 1/2 */
        return oracle_e2m1_value(oracle_fp4_padded_code(row, k));
    }
    if (fmt >= 3)
        return oracle_fp6_value_q(oracle_fp6_code(row, k), fmt, q);
    return oracle_fp8_value_q(row[k], fmt, q);
}

/* Step 1: element k of a packed row. */
static unsigned nibble(const uint8_t *row, int64_t k)
{
    uint8_t byte = row[k >> 1];
    return (k & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 0xFu);
}

/* Exported for the nibble-order check: the code of element k of a row. */
unsigned oracle_fp4_code(const uint8_t *row, int64_t k)
{
    return nibble(row, k);
}

/* bf16 bits -> double (exact). */
double oracle_bf16_to_double(uint16_t bits)
{
    int sign = bits >> 15;
    int e = (bits >> 7) & 0xFF;
    int f = bits & 0x7F;
    double v;
    if (e == 0xFF)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -133);
    else
        v = ldexp((double)(128 + f), e - 134);
    return sign ? -v : v;
}

/*
 * Step 6: round a double to the nearest bf16, ties to even, in one step.
 * bf16 has 8 significand bits and exponents down to 2^-126 (subnormals below
 * that, spaced 2^-133).  With q the exponent of the spacing at |x|, the
 * result is n * 2^q for the nearest-even integer n to |x| / 2^q, and its bit
 * pattern is (q + 133) * 128 + n (this also carries n = 256 into the next
 * binade and overflows into the infinity pattern 0x7F80).
 */
uint16_t oracle_bf16_rne(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x))
        return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a) || a >= 0x1p128)
        return (uint16_t)(sign | 0x7F80u);
    int E;
    frexp(a, &E);                       /* a = f * 2^E, f in [0.5, 1) */
    int q = (E - 1 > -126 ? E - 1 : -126) - 7;
    double r = ldexp(a, -q);            /* exact: scaling by a power of two */
    double n = floor(r);
    double frac = r - n;                /* exact */
    if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0))
        n += 1.0;
    long bits = (long)(q + 133) * 128L + (long)n;
    if (bits >= 0x7F80L)
        return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | (uint16_t)bits);
}

/* Exact-arithmetic checks used for step 5. */
static int two_sum_exact(double a, double b, double s)
{
    double bb = s - a;
    double err = (a - (s - bb)) + (b - bb);
    return err == 0.0;
}

struct gemm_job {
    int M, N, K;
    int fmt_a, fmt_b;  /* 0: E2M1 packed two per byte; 1: E4M3, 2: E5M2 bytes;
                          3: E2M3, 4: E3M2, 5: E2M1 in the padded
                          16-per-16-bytes forms */
    int nv;            /* 1: UE4M3 scales, one per 16 K (NVFP4); 0: E8M0 per 32 */
    const uint8_t *A; int64_t lda_bytes;
    const uint8_t *B; int64_t ldb_bytes;
    const uint8_t *SA; int64_t ldsa;
    const uint8_t *SB; int64_t ldsb;
    double alpha, beta;
    const uint16_t *C; int64_t ldc;
    uint16_t *D; int64_t ldd;
    double *acc_out;   /* [M*N] or NULL */
    double *abs_out;   /* [M*N] or NULL */
    const int64_t *pairs; int64_t npairs;   /* sampled mode: (m, n) pairs */
    int64_t next;      /* work counter */
    pthread_mutex_t lock;
    int64_t inexact;   /* outputs that failed an exactness check */
};

/* Steps 1-6 for one output element. */
static int one_output(struct gemm_job *j, int m, int n, uint16_t *d,
                      double *acc_o, double *abs_o)
{
    const uint8_t *arow = j->A + (int64_t)m * j->lda_bytes;
    const uint8_t *brow = j->B + (int64_t)n * j->ldb_bytes;
    const uint8_t *sarow = j->SA + (int64_t)m * j->ldsa;
    const uint8_t *sbrow = j->SB + (int64_t)n * j->ldsb;
    double acc = 0.0, sabs = 0.0;
    int min_g = 1 << 30;               /* min over products of their granule exponent */
    for (int64_t k = 0; k < j->K; ++k) {
        /* E2M1 values are multiples of 2^-1; FP8 values of 2^(ulp exponent). */
        int qa = -1, qb = -1;
        double va, vb;
        if (j->fmt_a == 0)
            va = oracle_e2m1_value(nibble(arow, k));
        else
            va = byte_form_value(arow, k, j->fmt_a, &qa);
        if (j->fmt_b == 0)
            vb = oracle_e2m1_value(nibble(brow, k));
        else
            vb = byte_form_value(brow, k, j->fmt_b, &qb);
        if (j->nv) {
            /* Step 3, NVFP4: the scale of the 16-element block holding k. */
            int sa_q, sb_q;
            double an = va * oracle_ue4m3_value_q(sarow[k / 16], &sa_q);
            double bn = vb * oracle_ue4m3_value_q(sbrow[k / 16], &sb_q);
            double pn = an * bn;
            acc += pn;
            sabs += fabs(pn);
            if (pn != 0.0 && qa + qb + sa_q + sb_q < min_g)
                min_g = qa + qb + sa_q + sb_q;
            continue;
        }
        unsigned ea = sarow[k / 32], eb = sbrow[k / 32];
        double a = va * oracle_e8m0_value(ea);
        double b = vb * oracle_e8m0_value(eb);
        double p = a * b;
        acc += p;
        sabs += fabs(p);
        if (p != 0.0) {
            int g = qa + qb + (int)ea + (int)eb - 254;
            if (g < min_g)
                min_g = g;
        }
    }
    int exact = 1;
    if (sabs != 0.0 && !(isfinite(sabs) && sabs < ldexp(1.0, 52 + min_g)))
        exact = 0;
    double y;
    if (j->beta != 0.0) {
        double c = oracle_bf16_to_double(j->C[(int64_t)m * j->ldc + n]);
        double p1 = j->alpha * acc;
        double p2 = j->beta * c;
        if (fma(j->alpha, acc, -p1) != 0.0 || fma(j->beta, c, -p2) != 0.0)
            exact = 0;
        y = p1 + p2;
        if (!two_sum_exact(p1, p2, y))
            exact = 0;
    } else {
        y = j->alpha * acc;
        if (fma(j->alpha, acc, -y) != 0.0)
            exact = 0;
    }
    *d = oracle_bf16_rne(y);
    if (acc_o)
        *acc_o = acc;
    if (abs_o)
        *abs_o = sabs;
    return exact;
}

static void *worker(void *arg)
{
    struct gemm_job *j = (struct gemm_job *)arg;
    int64_t total = j->pairs ? j->npairs : (int64_t)j->M;
    int64_t local_inexact = 0;
    for (;;) {
        pthread_mutex_lock(&j->lock);
        int64_t i = j->next++;
        pthread_mutex_unlock(&j->lock);
        if (i >= total)
            break;
        if (j->pairs) {
            int m = (int)j->pairs[2 * i], n = (int)j->pairs[2 * i + 1];
            if (!one_output(j, m, n, &j->D[i], j->acc_out ? &j->acc_out[i] : NULL,
                            j->abs_out ? &j->abs_out[i] : NULL))
                ++local_inexact;
        } else {
            int m = (int)i;
            for (int n = 0; n < j->N; ++n) {
                int64_t o = (int64_t)m * j->N + n;
                if (!one_output(j, m, n, &j->D[(int64_t)m * j->ldd + n],
                                j->acc_out ? &j->acc_out[o] : NULL,
                                j->abs_out ? &j->abs_out[o] : NULL))
                    ++local_inexact;
            }
        }
    }
    pthread_mutex_lock(&j->lock);
    j->inexact += local_inexact;
    pthread_mutex_unlock(&j->lock);
    return NULL;
}

/* Threads this process may run on (its CPU affinity set). */
int oracle_host_cores(void)
{
    cpu_set_t set;
    if (sched_getaffinity(0, sizeof(set), &set) == 0)
        return CPU_COUNT(&set);
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int64_t run(struct gemm_job *j, int nthreads)
{
    if (nthreads <= 0)
        nthreads = oracle_host_cores();
    pthread_mutex_init(&j->lock, NULL);
    j->next = 0;
    j->inexact = 0;
    pthread_t *t = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    int started = 0;
    for (int i = 0; i < nthreads; ++i)
        if (pthread_create(&t[i], NULL, worker, j) == 0)
            ++started;
    if (started == 0)
        worker(j);
    for (int i = 0; i < started; ++i)
        pthread_join(t[i], NULL);
    free(t);
    pthread_mutex_destroy(&j->lock);
    return j->inexact;
}

/*
 * Full GEMM.  A: uint8 [M, lda/2] (lda in fp4 elements, as the page's
 * kernarg block counts A/B strides), B likewise, SA/SB: uint8 E8M0 with row
 * strides in bytes, C: bf16 bits [M, ldc] (ignored when beta == 0), D: bf16
 * bits [M, ldd].  acc_out / abs_out (optional, [M*N] dense) receive the
 * exact double sum and sum|a*b| per output.  Returns the number of outputs
 * whose exactness checks failed (0 means every D is the correctly rounded
 * exact result), or -1 on bad arguments.
 */
int64_t oracle_gemm(int M, int N, int K,
                    const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                    const uint8_t *SA, int64_t ldsa, const uint8_t *SB, int64_t ldsb,
                    double alpha, double beta, const uint16_t *C, int64_t ldc,
                    uint16_t *D, int64_t ldd, double *acc_out, double *abs_out,
                    int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || K % 32 != 0 || (lda & 1) || (ldb & 1))
        return -1;
    if (beta != 0.0 && C == NULL)
        return -1;
    struct gemm_job j;
    memset(&j, 0, sizeof(j));
    j.M = M; j.N = N; j.K = K;
    j.A = A; j.lda_bytes = lda / 2; j.B = B; j.ldb_bytes = ldb / 2;
    j.SA = SA; j.ldsa = ldsa; j.SB = SB; j.ldsb = ldsb;
    j.alpha = alpha; j.beta = beta; j.C = C; j.ldc = ldc;
    j.D = D; j.ldd = ldd; j.acc_out = acc_out; j.abs_out = abs_out;
    return run(&j, nthreads);
}

/*
 * Sampled GEMM: the same computation at npairs (m, n) positions given as
 * pairs[2*i], pairs[2*i+1].  D, acc_out and abs_out are indexed by i.
 */
int64_t oracle_gemm_sampled(int M, int N, int K,
                            const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                            const uint8_t *SA, int64_t ldsa, const uint8_t *SB, int64_t ldsb,
                            double alpha, double beta, const uint16_t *C, int64_t ldc,
                            const int64_t *pairs, int64_t npairs,
                            uint16_t *D, double *acc_out, double *abs_out, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || K % 32 != 0 || (lda & 1) || (ldb & 1))
        return -1;
    if (beta != 0.0 && C == NULL)
        return -1;
    for (int64_t i = 0; i < npairs; ++i)
        if (pairs[2 * i] < 0 || pairs[2 * i] >= M || pairs[2 * i + 1] < 0 ||
            pairs[2 * i + 1] >= N)
            return -1;
    struct gemm_job j;
    memset(&j, 0, sizeof(j));
    j.M = M; j.N = N; j.K = K;
    j.A = A; j.lda_bytes = lda / 2; j.B = B; j.ldb_bytes = ldb / 2;
    j.SA = SA; j.ldsa = ldsa; j.SB = SB; j.ldsb = ldsb;
    j.alpha = alpha; j.beta = beta; j.C = C; j.ldc = ldc;
    j.D = D; j.ldd = 0; j.acc_out = acc_out; j.abs_out = abs_out;
    j.pairs = pairs; j.npairs = npairs;
    return run(&j, nthreads);
}

/*
 * NVFP4 forms of oracle_gemm / oracle_gemm_sampled: A and B as there (packed
 * E2M1, lda / ldb in elements), SA / SB one UE4M3 byte per 16 K (row strides
 * in bytes, at least K / 16).  K % 32 == 0 as for the MXFP4 GEMM.  Returns -1
 * for bad arguments, including a scale byte with bit 7 set.
 */
static int nv_args_ok(int M, int N, int K, int64_t lda, int64_t ldb,
                      const uint8_t *SA, int64_t ldsa, const uint8_t *SB, int64_t ldsb,
                      double beta, const uint16_t *C)
{
    if (M < 0 || N < 0 || K < 0 || K % 32 != 0 || (lda & 1) || (ldb & 1))
        return 0;
    if (ldsa < K / 16 || ldsb < K / 16 || (beta != 0.0 && C == NULL))
        return 0;
    for (int64_t r = 0; r < M; ++r)
        for (int64_t b = 0; b < K / 16; ++b)
            if (SA[r * ldsa + b] & 0x80u)
                return 0;
    for (int64_t r = 0; r < N; ++r)
        for (int64_t b = 0; b < K / 16; ++b)
            if (SB[r * ldsb + b] & 0x80u)
                return 0;
    return 1;
}

int64_t oracle_gemm_nv(int M, int N, int K,
                       const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                       const uint8_t *SA, int64_t ldsa, const uint8_t *SB, int64_t ldsb,
                       double alpha, double beta, const uint16_t *C, int64_t ldc,
                       uint16_t *D, int64_t ldd, double *acc_out, double *abs_out,
                       int nthreads)
{
    if (!nv_args_ok(M, N, K, lda, ldb, SA, ldsa, SB, ldsb, beta, C))
        return -1;
    struct gemm_job j;
    memset(&j, 0, sizeof(j));
    j.M = M; j.N = N; j.K = K; j.nv = 1;
    j.A = A; j.lda_bytes = lda / 2; j.B = B; j.ldb_bytes = ldb / 2;
    j.SA = SA; j.ldsa = ldsa; j.SB = SB; j.ldsb = ldsb;
    j.alpha = alpha; j.beta = beta; j.C = C; j.ldc = ldc;
    j.D = D; j.ldd = ldd; j.acc_out = acc_out; j.abs_out = abs_out;
    return run(&j, nthreads);
}

int64_t oracle_gemm_nv_sampled(int M, int N, int K,
                               const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                               const uint8_t *SA, int64_t ldsa, const uint8_t *SB, int64_t ldsb,
                               double alpha, double beta, const uint16_t *C, int64_t ldc,
                               const int64_t *pairs, int64_t npairs,
                               uint16_t *D, double *acc_out, double *abs_out, int nthreads)
{
    if (!nv_args_ok(M, N, K, lda, ldb, SA, ldsa, SB, ldsb, beta, C))
        return -1;
    for (int64_t i = 0; i < npairs; ++i)
        if (pairs[2 * i] < 0 || pairs[2 * i] >= M || pairs[2 * i + 1] < 0 ||
            pairs[2 * i + 1] >= N)
            return -1;
    struct gemm_job j;
    memset(&j, 0, sizeof(j));
    j.M = M; j.N = N; j.K = K; j.nv = 1;
    j.A = A; j.lda_bytes = lda / 2; j.B = B; j.ldb_bytes = ldb / 2;
    j.SA = SA; j.ldsa = ldsa; j.SB = SB; j.ldsb = ldsb;
    j.alpha = alpha; j.beta = beta; j.C = C; j.ldc = ldc;
    j.D = D; j.ldd = 0; j.acc_out = acc_out; j.abs_out = abs_out;
    j.pairs = pairs; j.npairs = npairs;
    return run(&j, nthreads);
}

/*
 * MXFP8 / MXFP6 forms of oracle_gemm / oracle_gemm_sampled: A and B hold one
 * 8-bit element per byte, or 6-bit elements in the padded form above (one
 * byte of footprint per element either way: lda, ldb in elements = bytes);
 * fmt_a / fmt_b = 1 (E4M3), 2 (E5M2), 3 (E2M3), 4 (E3M2) or 5 (E2M1,
 * padded), one E8M0 scale per 32 K as before.  Same steps 2-6, with the
 * element decoded by oracle_fp8_value_q, oracle_fp6_value_q or
 * oracle_e2m1_value.
 */
static int fp8_args_ok(int M, int N, int K, int fmt_a, int fmt_b, double beta, const uint16_t *C)
{
    if (M < 0 || N < 0 || K < 0 || K % 32 != 0)
        return 0;
    if (fmt_a < 1 || fmt_a > 5 || fmt_b < 1 || fmt_b > 5)
        return 0;
    if ((fmt_a >= 3 || fmt_b >= 3) && K % 16 != 0)
        return 0;
    return !(beta != 0.0 && C == NULL);
}

int64_t oracle_gemm8(int M, int N, int K, int fmt_a, int fmt_b,
                     const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                     const uint8_t *SA, int64_t ldsa, const uint8_t *SB, int64_t ldsb,
                     double alpha, double beta, const uint16_t *C, int64_t ldc,
                     uint16_t *D, int64_t ldd, double *acc_out, double *abs_out,
                     int nthreads)
{
    if (!fp8_args_ok(M, N, K, fmt_a, fmt_b, beta, C))
        return -1;
    struct gemm_job j;
    memset(&j, 0, sizeof(j));
    j.M = M; j.N = N; j.K = K; j.fmt_a = fmt_a; j.fmt_b = fmt_b;
    j.A = A; j.lda_bytes = lda; j.B = B; j.ldb_bytes = ldb;
    j.SA = SA; j.ldsa = ldsa; j.SB = SB; j.ldsb = ldsb;
    j.alpha = alpha; j.beta = beta; j.C = C; j.ldc = ldc;
    j.D = D; j.ldd = ldd; j.acc_out = acc_out; j.abs_out = abs_out;
    return run(&j, nthreads);
}

int64_t oracle_gemm8_sampled(int M, int N, int K, int fmt_a, int fmt_b,
                             const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                             const uint8_t *SA, int64_t ldsa, const uint8_t *SB, int64_t ldsb,
                             double alpha, double beta, const uint16_t *C, int64_t ldc,
                             const int64_t *pairs, int64_t npairs,
                             uint16_t *D, double *acc_out, double *abs_out, int nthreads)
{
    if (!fp8_args_ok(M, N, K, fmt_a, fmt_b, beta, C))
        return -1;
    for (int64_t i = 0; i < npairs; ++i)
        if (pairs[2 * i] < 0 || pairs[2 * i] >= M || pairs[2 * i + 1] < 0 ||
            pairs[2 * i + 1] >= N)
            return -1;
    struct gemm_job j;
    memset(&j, 0, sizeof(j));
    j.M = M; j.N = N; j.K = K; j.fmt_a = fmt_a; j.fmt_b = fmt_b;
    j.A = A; j.lda_bytes = lda; j.B = B; j.ldb_bytes = ldb;
    j.SA = SA; j.ldsa = ldsa; j.SB = SB; j.ldsb = ldsb;
    j.alpha = alpha; j.beta = beta; j.C = C; j.ldc = ldc;
    j.D = D; j.ldd = 0; j.acc_out = acc_out; j.abs_out = abs_out;
    j.pairs = pairs; j.npairs = npairs;
    return run(&j, nthreads);
}


/* ------------------------------------------------------------------------
 * MXFP4 quantisation of bf16 rows: the step before the GEMM that produces its
 * operands (the asm_f4gemm page lists operand generation among its reference
 * helpers, section "Files", without stating the rule; the rule here is the
 * one the benchmark workloads are built with).  For each 1x32 block of a row:
 *   1. amax = largest |x| of the block (bf16 values, exact in double);
 *   2. s = floor(log2(amax / 6)) -- the largest integer with 6 * 2^s <= amax
 *      (s = 0 when amax == 0), clamped to [-127, 127]; scale code = s + 127;
 *   3. y = |x| / 2^s (exact), rounded to the nearest E2M1 magnitude
 *      {0, .5, 1, 1.5, 2, 3, 4, 6} (section "Data layouts"), ties to the
 *      magnitude with an even code, y >= 6 saturating to 6;
 *   4. the sign bit (bit 3) copies the sign of x, so a negative x that
 *      rounds to 0 gives code 8 (-0);
 *   5. codes are packed two per byte, element 2i in the low nibble.
 * Readings where the rule is silent: the rounding mode (nearest, ties to
 * even, as the MFMA page states for its conversions), saturation at 6, and
 * the sign of zero.  Inputs are finite.
 * ------------------------------------------------------------------------ */

/* Step 2: the largest s with 6 * 2^s <= amax, found by exact comparisons. */
static int quant_exponent(double amax)
{
    if (amax == 0.0)
        return 0;
    int e = 0;
    frexp(amax, &e);
    int s = e - 3;
    while (ldexp(6.0, s) > amax)
        --s;
    while (ldexp(6.0, s + 1) <= amax)
        ++s;
    if (s < -127)
        s = -127;
    if (s > 127)
        s = 127;
    return s;
}

/* Step 3: nearest magnitude code 0..7, ties to the even code. */
static unsigned quant_magnitude_code(double y)
{
    if (y >= 6.0)
        return 7u;
    unsigned best = 0u;
    double best_d = y;   /* distance to magnitude 0 */
    for (unsigned c = 1u; c < 8u; ++c) {
        const double d = fabs(y - kE2M1Magnitude[c]);
        if (d < best_d || (d == best_d && (c & 1u) == 0u)) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

/* Quantise rows [rows, K] of bf16 bits (row stride ldx elements) into packed
 * codes Q (row stride ldq bytes) and scale codes S (row stride lds bytes).
 * Returns 0, or -1 for bad sizes. */
int oracle_quantize(int rows, int K, const uint16_t *X, int64_t ldx, uint8_t *Q, int64_t ldq,
                    uint8_t *S, int64_t lds)
{
    if (rows < 0 || K < 0 || (K % 32) != 0 || ldx < K || ldq < K / 2 || lds < K / 32)
        return -1;
    for (int r = 0; r < rows; ++r) {
        const uint16_t *x = X + (int64_t)r * ldx;
        for (int b = 0; b < K / 32; ++b) {
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                const double v = fabs(oracle_bf16_to_double(x[b * 32 + i]));
                if (v > amax)
                    amax = v;
            }
            const int s = quant_exponent(amax);
            S[(int64_t)r * lds + b] = (uint8_t)(s + 127);
            for (int i = 0; i < 32; i += 2) {
                unsigned code[2];
                for (int h = 0; h < 2; ++h) {
                    const double v = oracle_bf16_to_double(x[b * 32 + i + h]);
                    code[h] = quant_magnitude_code(ldexp(fabs(v), -s));
                    if (signbit(v))
                        code[h] |= 8u;
                }
                Q[(int64_t)r * ldq + (b * 32 + i) / 2] = (uint8_t)(code[0] | (code[1] << 4));
            }
        }
    }
    return 0;
}

/*
 * MXFP8 quantiser, the counterpart of oracle_quantize for 8-bit elements
 * (fmt 1 = E4M3, 2 = E5M2, decoded by oracle_fp8_value_q), and for the
 * padded 6- and 4-bit forms (fmt 3 = E2M3, 4 = E3M2, 5 = E2M1; emax 2, 4
 * and 2).  Per 1x32 block:
 *   1. amax = the largest magnitude of the block's 32 bf16 values;
 *   2. s = the largest integer with 2^(s + emax) <= amax, where emax is the
 *      exponent of the format's largest binade (8 for E4M3, whose largest
 *      value is 448; 15 for E5M2, 57344) -- the OCP MX scale rule, the plain
 *      reading where the pages only say the scaled builtins take one scale
 *      per block; s = 0 for an all-zero block; clamped to [-127, 127];
 *      scale code s + 127;
 *   3. each element: |x| / 2^s rounded to the nearest finite value of the
 *      format, ties to the even code (round-half-even), saturating at the
 *      largest finite value, with the sign of x.
 * Q holds one code per byte (row stride ldq bytes), or for fmt 3-5 the
 * padded form the GEMM reads, with zero padding bytes.
 */
static int quant8_exponent(double amax, int emax)
{
    if (amax == 0.0)
        return 0;
    int e = 0;
    frexp(amax, &e);
    int s = e - 1 - emax;
    while (ldexp(1.0, s + emax) > amax)
        --s;
    while (ldexp(1.0, s + emax + 1) <= amax)
        ++s;
    if (s < -127)
        s = -127;
    if (s > 127)
        s = 127;
    return s;
}

static double quant8_value(unsigned code, int fmt)
{
    if (fmt == 5)
        return oracle_e2m1_value(code);
    if (fmt >= 3)
        return oracle_fp6_value(code, fmt);
    return oracle_fp8_value(code, fmt);
}

static unsigned quant8_magnitude_code(double y, int fmt)
{
    static const unsigned kTop[6] = {0u, 0x7Eu, 0x7Bu, 0x1Fu, 0x1Fu, 0x7u};
    const unsigned top = kTop[fmt];                   /* largest finite code */
    if (y >= quant8_value(top, fmt))
        return top;
    unsigned best = 0u;
    double best_d = y;                                /* distance to code 0 (= 0.0) */
    for (unsigned c = 1u; c <= top; ++c) {
        const double d = fabs(y - quant8_value(c, fmt));
        if (d < best_d || (d == best_d && !(c & 1u))) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

/* Write element k's code into a row of the format's storage form. */
static void quant8_store(uint8_t *row, int64_t k, unsigned code, int fmt)
{
    if (fmt <= 2) {
        row[k] = (uint8_t)code;
        return;
    }
    uint8_t *g = row + (k >> 4) * 16;
    if ((k & 15) == 0)
        memset(g, 0, 16);                             /* codes and padding */
    if (fmt == 5) {
        g[(k & 15) >> 1] |= (uint8_t)((k & 1) ? code << 4 : code);
        return;
    }
    const int at = (int)(k & 15) * 6;                 /* first bit of the code */
    g[at / 8] |= (uint8_t)(code << (at % 8));
    if (at % 8 > 2)                                   /* it runs into the next byte */
        g[at / 8 + 1] |= (uint8_t)(code >> (8 - at % 8));
}

int oracle_quantize8(int rows, int K, int fmt, const uint16_t *X, int64_t ldx, uint8_t *Q,
                     int64_t ldq, uint8_t *S, int64_t lds)
{
    if (rows < 0 || K < 0 || (K % 32) != 0 || ldx < K || ldq < K || lds < K / 32 ||
        fmt < 1 || fmt > 5)
        return -1;
    static const int kEmax[6] = {0, 8, 15, 2, 4, 2};
    static const unsigned kSign[6] = {0u, 0x80u, 0x80u, 0x20u, 0x20u, 0x8u};
    const int emax = kEmax[fmt];
    for (int r = 0; r < rows; ++r) {
        const uint16_t *x = X + (int64_t)r * ldx;
        for (int b = 0; b < K / 32; ++b) {
            double amax = 0.0;                        /* step 1 */
            for (int i = 0; i < 32; ++i)
                amax = fmax(amax, fabs(oracle_bf16_to_double(x[b * 32 + i])));
            const int s = quant8_exponent(amax, emax);
            S[(int64_t)r * lds + b] = (uint8_t)(127 + s);
            for (int i = 0; i < 32; ++i) {
                const double v = oracle_bf16_to_double(x[b * 32 + i]);
                unsigned code = quant8_magnitude_code(ldexp(fabs(v), -s), fmt);
                if (signbit(v) != 0)
                    code |= kSign[fmt];
                quant8_store(Q + (int64_t)r * ldq, b * 32 + i, code, fmt);
            }
        }
    }
    return 0;
}
