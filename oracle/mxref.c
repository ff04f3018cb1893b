/*
 * mxref.c -- CPU oracle for the MX block-scaled NT GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, table or header with the CUDA path.
 *
 * What it computes (the plain definition, written out):
 *
 *   C[m,n] = sum_{j=0}^{K/32-1} 2^(SA[m,j]-127) * 2^(SB[n,j]-127)
 *                               * sum_{t=0}^{31} dec(A[m,32j+t]) * dec(B[n,32j+t])
 *
 *   S[m,n] = the same sum with every product replaced by its absolute value
 *            (the scale of the rounding-error bound used by the parity tests).
 *
 * Sources:
 *  - "Accelerating PyTorch on AMD GPUs with FlyDSL" (English digest), section
 *    "API compatibility is not universal input coverage": MXFP scaled GEMM takes
 *    one E8M0 scale per 32 values along K, and K divisible by 128.
 *  - AI-compiler daily digest of 2026-10-22, item 1 (FlyDSL): MXFP8/MXFP4 scaled
 *    GEMM uses scale blocks of 1 x 32 values, E8M0 scales and FP32 accumulation.
 *  - Same digest, item 2 ("Deciding Scale Placement in MXFP4 Dot Products"):
 *    applying the scale before or after the dot product can round differently.
 *    This oracle evaluates each 32-block's inner sum exactly (see below), so both
 *    placements give the same value here and no placement choice is made.
 *  - The element formats (OCP MX): E4M3 for MXFP8, E2M1 (two codes per byte)
 *    for MXFP4, E8M0 scales with code 0xFF = NaN.  The pages name only "MXFP8"
 *    and "MXFP4"; these encodings are the reading this build takes.
 *
 * Exactness: an E4M3 product has at most 8 significant bits and lies in
 * [2^-18, 448^2]; an E2M1 product is a multiple of 1/4 of magnitude <= 36.  Any
 * 32-term sum of such products is exact in binary64, and so is its scaling by a
 * power of two in [2^-254, 2^254].  The only rounding left is the binary64
 * accumulation across blocks, in increasing j (relative error <= (K/32)*2^-53
 * of S, far below the 1e-5*S tolerance the parity tests use).
 *
 * Element order inside an MXFP4 byte: element 2i is the low nibble, element
 * 2i+1 the high nibble.  Decoding is by table (16 entries for E2M1, 256 for
 * E4M3 and E8M0); NaN codes decode to NaN and propagate through the sums.
 *
 * Built with: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (by build() in oracle/mxref.py).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define MXREF_FMT_MXFP8 1
#define MXREF_FMT_MXFP4 2

static double tab_e2m1[16];
static double tab_e4m3[256];
static double tab_e8m0[256];
static int tables_ready = 0;

/* E2M1 (OCP FP4): sign bit 3, exponent bits 2..1, mantissa bit 0, bias 1.
 * The eight magnitudes are listed outright: 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 * No infinities and no NaN; code 0x8 is -0. */
static void fill_e2m1(void)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    for (int c = 0; c < 16; ++c)
        tab_e2m1[c] = (c & 8) ? -mag[c & 7] : mag[c & 7];
}

/* E4M3 (OCP FP8 "E4M3FN"): sign bit 7, exponent bits 6..3 (bias 7), mantissa
 * bits 2..0.  Exponent field 0 is subnormal: m/8 * 2^-6.  Otherwise
 * (1 + m/8) * 2^(e-7).  e=15,m=7 (0x7F / 0xFF) is NaN; there is no infinity,
 * so 0x7E = 448 is the largest finite value. */
static void fill_e4m3(void)
{
    for (int c = 0; c < 256; ++c) {
        int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
        double v;
        if (e == 15 && m == 7)
            v = NAN;
        else if (e == 0)
            v = ldexp((double)m, -9);          /* m/8 * 2^-6 */
        else
            v = ldexp(8.0 + m, e - 10);        /* (8+m)/8 * 2^(e-7) */
        tab_e4m3[c] = s ? -v : v;
    }
}

/* E8M0: unsigned power-of-two exponent, value 2^(c-127) for c in 0..254;
 * c = 255 is NaN.  There is no zero and no sign. */
static void fill_e8m0(void)
{
    for (int c = 0; c < 255; ++c)
        tab_e8m0[c] = ldexp(1.0, c - 127);
    tab_e8m0[255] = NAN;
}

void mxref_init(void)
{
    if (tables_ready)
        return;
    fill_e2m1();
    fill_e4m3();
    fill_e8m0();
    tables_ready = 1;
}

/* Copy a decode table out (which: 1 = E4M3, 2 = E2M1, 3 = E8M0).
 * Returns the number of entries written, or -1 for an unknown table. */
int mxref_decode_table(int which, double *out)
{
    mxref_init();
    switch (which) {
    case 1: memcpy(out, tab_e4m3, sizeof tab_e4m3); return 256;
    case 2: memcpy(out, tab_e2m1, sizeof tab_e2m1); return 16;
    case 3: memcpy(out, tab_e8m0, sizeof tab_e8m0); return 256;
    default: return -1;
    }
}

/* Decode one packed operand row (codes only, no scale) into K doubles. */
static void decode_row(int fmt, const uint8_t *row, int64_t K, double *dst)
{
    if (fmt == MXREF_FMT_MXFP8) {
        for (int64_t k = 0; k < K; ++k)
            dst[k] = tab_e4m3[row[k]];
    } else {
        for (int64_t k = 0; k < K; k += 2) {
            uint8_t byte = row[k >> 1];
            dst[k] = tab_e2m1[byte & 15];
            dst[k + 1] = tab_e2m1[byte >> 4];
        }
    }
}

/*
 * Reference GEMM over a set of output rows and columns.
 *
 *   fmt          1 = MXFP8 (E4M3, one byte per code), 2 = MXFP4 (E2M1, two codes/byte)
 *   A, SA        M x K codes (row-major, K or K/2 bytes per row) and M x K/32 scales
 *   B, SB        N x K codes and N x K/32 scales (B is the "T" operand: C = A * B^T)
 *   rows, nrows  which rows of C to compute (NULL: all M, in order)
 *   cols, ncols  which columns of C to compute (NULL: all N, in order)
 *   C, S         nrows x ncols binary64 outputs (S may be NULL)
 *   nthreads     OpenMP threads (<= 0: the runtime default)
 *
 * Returns 0, or -1 for bad arguments (K not a positive multiple of 32, unknown
 * fmt, out-of-range row or column index).
 */
int mxref_gemm(int fmt, int64_t M, int64_t N, int64_t K,
               const uint8_t *A, const uint8_t *SA,
               const uint8_t *B, const uint8_t *SB,
               const int64_t *rows, int64_t nrows,
               const int64_t *cols, int64_t ncols,
               double *C, double *S, int nthreads)
{
    mxref_init();
    if ((fmt != MXREF_FMT_MXFP8 && fmt != MXREF_FMT_MXFP4) || K <= 0 || K % 32 != 0 ||
        M < 0 || N < 0)
        return -1;
    if (rows == NULL) nrows = M;
    if (cols == NULL) ncols = N;
    for (int64_t i = 0; i < (rows ? nrows : 0); ++i)
        if (rows[i] < 0 || rows[i] >= M) return -1;
    for (int64_t i = 0; i < (cols ? ncols : 0); ++i)
        if (cols[i] < 0 || cols[i] >= N) return -1;

    const int64_t row_bytes = (fmt == MXREF_FMT_MXFP8) ? K : K / 2;
    const int64_t nblk = K / 32;
    int err = 0;

#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

#pragma omp parallel
    {
        double *a = (double *)malloc(sizeof(double) * (size_t)K);
        double *b = (double *)malloc(sizeof(double) * (size_t)K);
        if (!a || !b) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            if (!a || !b) continue;
            const int64_t m = rows ? rows[i] : i;
            decode_row(fmt, A + m * row_bytes, K, a);
            for (int64_t jcol = 0; jcol < ncols; ++jcol) {
                const int64_t n = cols ? cols[jcol] : jcol;
                decode_row(fmt, B + n * row_bytes, K, b);
                double acc = 0.0, acc_abs = 0.0;
                for (int64_t j = 0; j < nblk; ++j) {
                    double inner = 0.0, inner_abs = 0.0;
                    for (int64_t t = 0; t < 32; ++t) {
                        const double p = a[32 * j + t] * b[32 * j + t];
                        inner += p;
                        inner_abs += fabs(p);
                    }
                    const double sc = tab_e8m0[SA[m * nblk + j]] * tab_e8m0[SB[n * nblk + j]];
                    acc += sc * inner;
                    acc_abs += sc * inner_abs;
                }
                C[i * ncols + jcol] = acc;
                if (S) S[i * ncols + jcol] = acc_abs;
            }
        }
        free(a);
        free(b);
    }
    return err ? -1 : 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int mxref_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------- */
/* Reference MX quantiser (the step before the GEMM).                         */
/*                                                                            */
/* The FlyDSL page (English digest, "Performance numbers need their           */
/* baselines") times the scaled GEMMs from already-quantised inputs and       */
/* prints no quantisation formula; the recipe below is this repository's      */
/* reading.  Per row and 32-value block along K:                              */
/*   amax = max |x| over the block;                                           */
/*   E = floor(log2 amax), taken exactly from the binary exponent (frexp);    */
/*   s = max(E - e_max, -127), e_max = 8 (E4M3: 448 = 1.75 * 2^8) or          */
/*       2 (E2M1: 6 = 1.5 * 2^2); s cannot exceed 125 for finite input;       */
/*   an all-zero block takes s = 0;                                           */
/*   scale code = s + 127;                                                    */
/*   element = x / 2^s rounded to the nearest value of the element grid,      */
/*   ties to even, magnitudes past the largest finite value saturate (448 or  */
/*   6); the sign of a zero result is the sign of x.                          */
/*   A block holding a NaN or an infinity gets scale code 0xFF (NaN) and all  */
/*   element codes 0: in MX a NaN scale makes the whole block NaN, and E2M1   */
/*   has no NaN of its own, so this is the one encoding both formats share.   */
/* Arithmetic in binary64: x / 2^s is exact, so rounding happens once.        */
/* ------------------------------------------------------------------------- */

/* Round v (exact binary64) to the nearest value of the grid with `mbits`
 * fraction bits and smallest normal exponent `emin`, ties to even, then
 * saturate to vmax. */
static double grid_round(double v, int emin, int mbits, double vmax)
{
    double mag = fabs(v);
    if (mag == 0.0)
        return v;
    int e;
    frexp(mag, &e); /* mag = f * 2^e, f in [0.5, 1): floor(log2 mag) = e - 1 */
    int q = (e - 1 > emin ? e - 1 : emin) - mbits;  /* grid spacing 2^q */
    double t = ldexp(mag, -q);                      /* exact */
    double fl = floor(t);
    double fr = t - fl;
    double r;
    if (fr > 0.5)
        r = fl + 1.0;
    else if (fr < 0.5)
        r = fl;
    else
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    r = ldexp(r, q);
    if (r > vmax)
        r = vmax;
    return v < 0 ? -r : r;  /* a negative v that rounds to zero gives -0 */
}

/* Code of an E4M3 grid value (|r| <= 448, never NaN here). */
static uint8_t encode_e4m3(double r)
{
    uint8_t sign = signbit(r) ? 0x80 : 0;
    double mag = fabs(r);
    if (mag == 0.0)
        return sign;
    if (mag < ldexp(1.0, -6))                    /* subnormal: m * 2^-9 */
        return sign | (uint8_t)(mag * 512.0);
    int e;
    double f = frexp(mag, &e);                   /* mag = f * 2^e */
    int ef = e + 6;                              /* biased exponent (bias 7) */
    int mf = (int)((2.0 * f - 1.0) * 8.0 + 0.5); /* exact: r is on the grid */
    return sign | (uint8_t)(ef << 3) | (uint8_t)mf;
}

/* Code of an E2M1 grid value (|r| <= 6). */
static uint8_t encode_e2m1(double r)
{
    static const double mag_of[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    uint8_t sign = signbit(r) ? 8 : 0;
    double mag = fabs(r);
    for (uint8_t c = 0; c < 8; ++c)
        if (mag_of[c] == mag)
            return sign | c;
    return 0; /* unreachable after grid_round */
}

/*
 * in_dtype: 1 = FP32, 2 = BF16 (raw 16-bit patterns).  x: rows x K, row-major.
 * codes: rows x K bytes (MXFP8) or rows x K/2 bytes (MXFP4, element 2i in the
 * low nibble); scales: rows x K/32 bytes, row-major.  Returns 0, or -1 for
 * bad arguments (unknown fmt or in_dtype, K not a positive multiple of 32).
 */
int mxref_quantize(int fmt, int in_dtype, int64_t rows, int64_t K, const void *x,
                   uint8_t *codes, uint8_t *scales)
{
    if ((fmt != MXREF_FMT_MXFP8 && fmt != MXREF_FMT_MXFP4) || (in_dtype != 1 && in_dtype != 2) ||
        rows < 0 || K <= 0 || K % 32 != 0)
        return -1;
    const int e_max = fmt == MXREF_FMT_MXFP8 ? 8 : 2;
    const int emin = fmt == MXREF_FMT_MXFP8 ? -6 : 0;
    const int mbits = fmt == MXREF_FMT_MXFP8 ? 3 : 1;
    const double vmax = fmt == MXREF_FMT_MXFP8 ? 448.0 : 6.0;
    const int64_t row_bytes = fmt == MXREF_FMT_MXFP8 ? K : K / 2;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        uint8_t *code_row = codes + r * row_bytes;
        for (int64_t j = 0; j < K / 32; ++j) {
            double v[32];
            double amax = 0.0;
            int nonfinite = 0;
            for (int t = 0; t < 32; ++t) {
                const int64_t k = 32 * j + t;
                if (in_dtype == 1) {
                    v[t] = (double)((const float *)x)[r * K + k];
                } else {
                    uint32_t bits = (uint32_t)((const uint16_t *)x)[r * K + k] << 16;
                    float f;
                    memcpy(&f, &bits, sizeof f);
                    v[t] = (double)f;
                }
                if (!isfinite(v[t]))
                    nonfinite = 1;
                else if (fabs(v[t]) > amax)
                    amax = fabs(v[t]);
            }
            if (nonfinite) {
                scales[r * (K / 32) + j] = 0xFF;
                memset(code_row + j * (row_bytes / (K / 32)), 0, (size_t)(row_bytes / (K / 32)));
                continue;
            }
            int s = 0;
            if (amax > 0.0) {
                int e;
                frexp(amax, &e);
                s = (e - 1) - e_max;
                if (s < -127)
                    s = -127;
            }
            scales[r * (K / 32) + j] = (uint8_t)(s + 127);
            for (int t = 0; t < 32; ++t) {
                const int64_t k = 32 * j + t;
                const double q = grid_round(ldexp(v[t], -s), emin, mbits, vmax);
                if (fmt == MXREF_FMT_MXFP8) {
                    code_row[k] = encode_e4m3(q);
                } else {
                    const uint8_t c = encode_e2m1(q);
                    uint8_t *b = &code_row[k / 2];
                    *b = (k & 1) ? (uint8_t)((*b & 0x0F) | (c << 4)) : (uint8_t)((*b & 0xF0) | c);
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Scale placement in MXFP4 dot products (reference checker).                 */
/*                                                                            */
/* AI-compiler daily digest of 2026-10-22, item 2 ("Deciding Scale Placement  */
/* in MXFP4 Dot Products with Integer Arithmetic"): lowering an MXFP4 dot     */
/* product may apply the shared power-of-two scales before the products       */
/* ("pre") or after the sum ("post"); in binary32 the two can round           */
/* differently (overflow, NaN, subnormals), and the study bounds the sum of   */
/* scale exponents for which they agree under a fixed binary reduction tree.  */
/* The bound is not printed on the page.  Readings taken here:                */
/*   k elements a_i, b_i (E2M1), scales sa, sb (E8M0 codes 0..254),           */
/*   f_a = 2^(sa-127), f_b = 2^(sb-127) as binary32 values (exact, also when  */
/*   subnormal);                                                              */
/*   pre  = tree_sum(  (a_i * f_a) * (b_i * f_b) ),                           */
/*   post = (tree_sum( a_i * b_i ) * f_a) * f_b,                              */
/*   every operation one binary32 operation rounded to nearest-even, no fused */
/*   multiply-add; tree_sum over n terms = tree_sum(first ceil(n/2)) +        */
/*   tree_sum(rest);                                                          */
/*   exact = sum a_i b_i * 2^(sa+sb-254), and rn_exact its binary32 rounding; */
/*   two results are "equal" when both are NaN or they are equal values       */
/*   (+0 == -0: the sign of a zero sum is not a placement question).          */
/* Tuples are numbered t = sum_i a_i << 4i + sum_i b_i << 4(k+i) over the     */
/* 4-bit codes, 16^(2k) of them.                                              */
/* ------------------------------------------------------------------------- */

static float tree_sum_f(const float *v, int n)
{
    if (n == 1)
        return v[0];
    const int h = (n + 1) / 2;
    volatile float l = tree_sum_f(v, h);
    volatile float r = tree_sum_f(v + h, n - h);
    volatile float s = l + r;
    return s;
}

static int same_f(float x, float y)
{
    if (isnan(x) || isnan(y))
        return isnan(x) && isnan(y);
    return x == y;
}

/* The three values of tuple t under scales fa = 2^(sa-127), fb = 2^(sb-127). */
static void placement_eval(int k, int sa, int sb, float fa, float fb, long long t, float *pre, float *post,
                           float *rn)
{
    float prod_pre[4], prod_post[4];
    double exact_sum = 0.0;
    for (int i = 0; i < k; ++i) {
        const double a = tab_e2m1[(t >> (4 * i)) & 15];
        const double b = tab_e2m1[(t >> (4 * (k + i))) & 15];
        volatile float as = (float)a * fa;
        volatile float bs = (float)b * fb;
        volatile float pp = as * bs;
        prod_pre[i] = pp;
        volatile float q = (float)a * (float)b;  /* exact: a multiple of 1/4, |.| <= 36 */
        prod_post[i] = q;
        exact_sum += a * b;                         /* exact */
    }
    *pre = tree_sum_f(prod_pre, k);
    volatile float post1 = tree_sum_f(prod_post, k) * fa;
    volatile float post2 = post1 * fb;
    *post = post2;
    *rn = (float)ldexp(exact_sum, sa + sb - 254);  /* one rounding of an exact value */
}

/* pre, post and rn of one tuple (out[0..2]).  Returns 0, or -1 for bad arguments. */
int mxref_placement_eval(int k, int sa, int sb, long long t, float *out)
{
    mxref_init();
    if (k < 1 || k > 4 || sa < 0 || sa > 254 || sb < 0 || sb > 254 || t < 0 || t >= (1ll << (8 * k)))
        return -1;
    placement_eval(k, sa, sb, (float)ldexp(1.0, sa - 127), (float)ldexp(1.0, sb - 127), t, &out[0], &out[1],
                   &out[2]);
    return 0;
}

/*
 * For each of the npairs scale pairs (sa[p], sb[p]), enumerate every tuple of a
 * k-element (1 <= k <= 4) MXFP4 dot product and write
 *   counts[3p+0] = tuples with pre != post,
 *   counts[3p+1] = tuples with pre == rn,
 *   counts[3p+2] = tuples with post == rn,
 *   first_diff[p] = the smallest tuple number with pre != post, or -1.
 * Returns 0, or -1 for bad arguments.
 */
int mxref_placement_scan(int k, const int *sa, const int *sb, int npairs, long long *counts, long long *first_diff)
{
    mxref_init();
    if (k < 1 || k > 4 || npairs < 0)
        return -1;
    for (int p = 0; p < npairs; ++p)
        if (sa[p] < 0 || sa[p] > 254 || sb[p] < 0 || sb[p] > 254)
            return -1;
    const long long ntup = 1ll << (8 * k);
    for (int p = 0; p < npairs; ++p) {
        const float fa = (float)ldexp(1.0, sa[p] - 127), fb = (float)ldexp(1.0, sb[p] - 127);
        long long n_diff = 0, n_pre = 0, n_post = 0, first = ntup;
#pragma omp parallel for schedule(static) reduction(+ : n_diff, n_pre, n_post) reduction(min : first)
        for (long long t = 0; t < ntup; ++t) {
            float pre, post, rn;
            placement_eval(k, sa[p], sb[p], fa, fb, t, &pre, &post, &rn);
            const int d = !same_f(pre, post);
            n_diff += d;
            n_pre += same_f(pre, rn);
            n_post += same_f(post, rn);
            if (d && t < first)
                first = t;
        }
        counts[3 * p] = n_diff;
        counts[3 * p + 1] = n_pre;
        counts[3 * p + 2] = n_post;
        first_diff[p] = n_diff ? first : -1;
    }
    return 0;
}

/* pre, post and rn of every tuple of one scale pair: out[3t+0..2]
 * (16^(2k) x 3 floats).  Returns 0, or -1 for bad arguments. */
int mxref_placement_values(int k, int sa, int sb, float *out)
{
    mxref_init();
    if (k < 1 || k > 3 || sa < 0 || sa > 254 || sb < 0 || sb > 254)
        return -1;
    const long long ntup = 1ll << (8 * k);
    const float fa = (float)ldexp(1.0, sa - 127), fb = (float)ldexp(1.0, sb - 127);
#pragma omp parallel for schedule(static)
    for (long long t = 0; t < ntup; ++t)
        placement_eval(k, sa, sb, fa, fb, t, &out[3 * t], &out[3 * t + 1], &out[3 * t + 2]);
    return 0;
}
