/*
 * CPU oracle for the GEMV library -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg use
 * this file.  The library's product path never links, loads or calls it, and
 * it shares no code, header or table with the CUDA sources.
 *
 * What it computes (double precision, plain loops, column index ascending):
 *
 *   y[i] = sum_{j=0}^{N-1} w(i,j) * x(j)
 *
 *   "Making GEMV Fast", section "Algorithm": every output is the dot product of
 *   one row of A with x; "Row-major indexing refresher": A(r,c) = A[r*N + c].
 *   "llama.cpp GEMV CUDA": y_i = sum_j W_ij x_j with W [M, d] row-major.
 *
 *   f32: w = A[i*N+j],                 x = x[j]           (FP32 storage)
 *   f16: w = dec16(A[i*N+j]),          x = dec16(x[j])    (binary16 storage)
 *   q8 : w = dec16(S[i*g + j/128]) * (int8)A[i*N+j]
 *   q4 : byte b = A[i*(N/2) + j/2]; nibble = low 4 bits for even j, high 4
 *        bits for odd j, read as 4-bit two's complement in [-8, 7];
 *        w = dec16(S[i*g + j/128]) * nibble
 *        with g = ceil(N/128) FP16 scales per row ("membound", section
 *        "dequant GEMV": weights dequantised in register as q times the
 *        group scale; the reference there is computed on q*s exactly).
 *   f16 weights with FP32 x: w = dec16(A[i*N+j]), x = x[j] (FP32 storage)
 *        ("llama.cpp GEMV CUDA", implementation note: FP32 hidden state).
 *   q8 with one scale per row: w = dec16(S[i]) * (int8)A[i*N+j] ("membound",
 *        section "dequant GEMV": the page's kernel keeps one scale per row).
 *
 * Alongside y it returns den[i] = sum_j |w(i,j)| * |x(j)|, the normaliser of
 * the parity metric |y_gpu - y_ref| / den.
 *
 * dec16 is written from the IEEE 754 binary16 definition: 1 sign bit, 5
 * exponent bits with bias 15, 10 fraction bits; exponent 0 encodes zero and
 * subnormals (fraction * 2^-24), exponent 31 encodes inf / NaN.
 *
 * Rows may be requested one by one (a list of row indices) so that a parity
 * check at full size can sample outputs.  Rows are split across threads with
 * OpenMP; each row is still summed by one thread in column order, so the
 * result does not depend on the thread count.
 *
 * Counting model ("Making GEMV Fast", sections "Memory Access" and
 * "Computation"): FLOPs = M(2N-1) = 2MN - M; FP32 bytes = 4(MN + N + M),
 * generalised per storage type as bytes(A) + bytes(scales) + bytes(x) + 4M.
 *
 * The file also holds the row softmax of the same pages' second memory-bound
 * decode kernel (see oracle_softmax_f16) and the symmetric weight quantiser
 * that produces the INT8 / INT4 operands (see oracle_quantize).
 *
 * Built with ORACLE_MUTANT=k (k > 0) it contains one deliberate mistake; the
 * test-suite builds those variants to show that its pins catch each one.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define ORACLE_GROUP 128

/* ---- IEEE 754 binary16 -> double ---------------------------------------- */

double oracle_dec16(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1F;
    const int frac = h & 0x3FF;
    double mag;
    if (expo == 0) {
#if ORACLE_MUTANT == 5
        mag = ldexp(1.0 + frac / 1024.0, -15); /* subnormals treated as normals */
#else
        mag = ldexp((double)frac, -24);        /* zero and subnormals */
#endif
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp(1024.0 + frac, expo - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -mag : mag;
}

void oracle_dec16_array(const uint16_t *h, double *out, int64_t n)
{
    for (int64_t k = 0; k < n; ++k) out[k] = oracle_dec16(h[k]);
}

/* ---- weight of element (i, j) per storage type ---------------------------- */

static int64_t n_groups(int64_t N) { return (N + ORACLE_GROUP - 1) / ORACLE_GROUP; }

static double w_f32(const float *A, int64_t M, int64_t N, int64_t i, int64_t j)
{
#if ORACLE_MUTANT == 4
    (void)N;
    return (double)A[j * M + i]; /* transposed operand (column-major read) */
#else
    (void)M;
    return (double)A[i * N + j];
#endif
}

static double w_f16(const uint16_t *A, int64_t N, int64_t i, int64_t j)
{
    return oracle_dec16(A[i * N + j]);
}

static double scale_of(const uint16_t *S, int64_t N, int64_t i, int64_t j)
{
#if ORACLE_MUTANT == 3
    return oracle_dec16(S[i * n_groups(N) + j / 64]); /* wrong group width */
#elif ORACLE_MUTANT == 7
    return oracle_dec16(S[i * (N / ORACLE_GROUP) + j / ORACLE_GROUP]); /* floor(N/128) pitch */
#else
    return oracle_dec16(S[i * n_groups(N) + j / ORACLE_GROUP]);
#endif
}

static double w_q8(const int8_t *A, const uint16_t *S, int64_t N, int64_t i, int64_t j)
{
    return scale_of(S, N, i, j) * (double)A[i * N + j];
}

static int q4_code(const uint8_t *A, int64_t N, int64_t i, int64_t j)
{
    const uint8_t b = A[i * (N / 2) + j / 2];
#if ORACLE_MUTANT == 1
    const int nib = (j & 1) ? (b & 0xF) : (b >> 4); /* nibble order swapped */
#else
    const int nib = (j & 1) ? (b >> 4) : (b & 0xF);
#endif
#if ORACLE_MUTANT == 2
    return nib - 8; /* offset-8 instead of two's complement */
#else
    return nib >= 8 ? nib - 16 : nib;
#endif
}

static double w_q4(const uint8_t *A, const uint16_t *S, int64_t N, int64_t i, int64_t j)
{
    return scale_of(S, N, i, j) * (double)q4_code(A, N, i, j);
}

/* ---- one row ------------------------------------------------------------- */

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_Q8 = 2, ORACLE_Q4 = 3, ORACLE_F16X32 = 4,
       ORACLE_Q8ROW = 5 };

/* one FP16 scale per row: S[i] */
static double w_q8row(const int8_t *A, const uint16_t *S, int64_t N, int64_t i, int64_t j)
{
#if ORACLE_MUTANT == 11
    const double s = oracle_dec16(S[0]); /* every row scaled by row 0's scale */
#else
    const double s = oracle_dec16(S[i]);
#endif
    return s * (double)A[i * N + j];
}

static double x_of(int kind, const void *x, int64_t j)
{
#if ORACLE_MUTANT == 12
    if (kind == ORACLE_F32) return (double)((const float *)x)[j]; /* FP32 x read as binary16 */
#else
    if (kind == ORACLE_F32 || kind == ORACLE_F16X32) return (double)((const float *)x)[j];
#endif
    return oracle_dec16(((const uint16_t *)x)[j]);
}

static double w_of(int kind, const void *A, const uint16_t *S, int64_t M, int64_t N, int64_t i,
                   int64_t j)
{
    switch (kind) {
    case ORACLE_F32: return w_f32((const float *)A, M, N, i, j);
    case ORACLE_F16:
    case ORACLE_F16X32: return w_f16((const uint16_t *)A, N, i, j);
    case ORACLE_Q8: return w_q8((const int8_t *)A, S, N, i, j);
    case ORACLE_Q8ROW: return w_q8row((const int8_t *)A, S, N, i, j);
    default: return w_q4((const uint8_t *)A, S, N, i, j);
    }
}

static void one_row(int kind, const void *A, const void *x, const uint16_t *S, int64_t M,
                    int64_t N, int64_t i, double *y, double *den)
{
    double acc = 0.0, mag = 0.0;
#if ORACLE_MUTANT == 6
    const int64_t jend = N > 0 ? N - 1 : 0; /* last column dropped */
#else
    const int64_t jend = N;
#endif
    for (int64_t j = 0; j < jend; ++j) {
        const double w = w_of(kind, A, S, M, N, i, j);
        const double v = x_of(kind, x, j);
        acc += w * v;
        mag += fabs(w) * fabs(v);
    }
    *y = acc;
    *den = mag;
}

static int run_rows(int kind, const void *A, const void *x, const uint16_t *S, int64_t M,
                    int64_t N, const int64_t *rows, int64_t nrows, double *y, double *den,
                    int threads)
{
    if (M < 0 || N < 0 || nrows < 0 || !y || !den) return -1;
    if ((M > 0 && N > 0) && (!A || !x)) return -1;
    if ((kind == ORACLE_Q8 || kind == ORACLE_Q4 || kind == ORACLE_Q8ROW) && M > 0 && N > 0 && !S)
        return -1;
    if (kind == ORACLE_Q4 && (N % 2)) return -1;
    if (!rows) nrows = M;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= M) return -1;
    }
    if (threads < 1) threads = 1;
#pragma omp parallel for num_threads(threads) schedule(dynamic, 16)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        one_row(kind, A, x, S, M, N, i, &y[r], &den[r]);
    }
    return 0;
}

int oracle_gemv_f32(const float *A, const float *x, int64_t M, int64_t N, const int64_t *rows,
                    int64_t nrows, double *y, double *den, int threads)
{
    return run_rows(ORACLE_F32, A, x, NULL, M, N, rows, nrows, y, den, threads);
}

int oracle_gemv_f16(const uint16_t *A, const uint16_t *x, int64_t M, int64_t N,
                    const int64_t *rows, int64_t nrows, double *y, double *den, int threads)
{
    return run_rows(ORACLE_F16, A, x, NULL, M, N, rows, nrows, y, den, threads);
}

int oracle_gemv_q8(const int8_t *A, const uint16_t *x, const uint16_t *S, int64_t M, int64_t N,
                   const int64_t *rows, int64_t nrows, double *y, double *den, int threads)
{
    return run_rows(ORACLE_Q8, A, x, S, M, N, rows, nrows, y, den, threads);
}

int oracle_gemv_q4(const uint8_t *A, const uint16_t *x, const uint16_t *S, int64_t M, int64_t N,
                   const int64_t *rows, int64_t nrows, double *y, double *den, int threads)
{
    return run_rows(ORACLE_Q4, A, x, S, M, N, rows, nrows, y, den, threads);
}

int oracle_gemv_f16_xf32(const uint16_t *A, const float *x, int64_t M, int64_t N,
                         const int64_t *rows, int64_t nrows, double *y, double *den, int threads)
{
    return run_rows(ORACLE_F16X32, A, x, NULL, M, N, rows, nrows, y, den, threads);
}

int oracle_gemv_q8_rowscale(const int8_t *A, const uint16_t *x, const uint16_t *S, int64_t M,
                            int64_t N, const int64_t *rows, int64_t nrows, double *y, double *den,
                            int threads)
{
    return run_rows(ORACLE_Q8ROW, A, x, S, M, N, rows, nrows, y, den, threads);
}

/* ---- dequantised weights (the q*s the reference is computed on) --------- */

int oracle_dequant_q8(const int8_t *A, const uint16_t *S, int64_t M, int64_t N, double *W)
{
    if (M < 0 || N < 0 || ((M > 0 && N > 0) && (!A || !S || !W))) return -1;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) W[i * N + j] = w_q8(A, S, N, i, j);
    return 0;
}

int oracle_dequant_q4(const uint8_t *A, const uint16_t *S, int64_t M, int64_t N, double *W)
{
    if (M < 0 || N < 0 || (N % 2) || ((M > 0 && N > 0) && (!A || !S || !W))) return -1;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) W[i * N + j] = w_q4(A, S, N, i, j);
    return 0;
}

/* ---- counting model ------------------------------------------------------ */

double oracle_flops(int64_t M, int64_t N)
{
    if (M <= 0 || N <= 0) return 0.0;
    return (double)M * (double)(2 * N - 1);
}

/* bytes read (A, scales, x) plus bytes written (y, FP32) for one call */
double oracle_bytes(int kind, int64_t M, int64_t N)
{
    const double m = (double)M, n = (double)N;
    switch (kind) {
    case ORACLE_F32: return 4.0 * (m * n + n + m);
    case ORACLE_F16: return 2.0 * m * n + 2.0 * n + 4.0 * m;
    case ORACLE_Q8: return m * n + 2.0 * m * (double)n_groups(N) + 2.0 * n + 4.0 * m;
    case ORACLE_Q4: return m * n / 2.0 + 2.0 * m * (double)n_groups(N) + 2.0 * n + 4.0 * m;
    case ORACLE_F16X32: return 2.0 * m * n + 4.0 * n + 4.0 * m;
    case ORACLE_Q8ROW: return m * n + 2.0 * m + 2.0 * n + 4.0 * m;
    default: return -1.0;
    }
}

/* ---- row softmax ----------------------------------------------------------
 *
 * "membound", section "Bonus kernel: online softmax": each row of an FP16
 * matrix is mapped to exp(x_j - m) / sum_k exp(x_k - m) with m the row
 * maximum.  The page computes it with the online update of the running
 * maximum and sum; the oracle is the plain definition (the online form reaches
 * the same value up to rounding), in double precision, columns ascending.
 * y receives nrows rows of N doubles.
 */
int oracle_softmax_f16(const uint16_t *x, int64_t M, int64_t N, const int64_t *rows, int64_t nrows,
                       double *y, int threads)
{
    if (M < 0 || N < 0 || nrows < 0 || (M > 0 && N > 0 && (!x || !y))) return -1;
    if (!rows) nrows = M;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= M) return -1;
    }
    if (threads < 1) threads = 1;
#pragma omp parallel for num_threads(threads) schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        const uint16_t *xi = x + i * N;
        double *yi = y + r * N;
        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j) {
            const double v = oracle_dec16(xi[j]);
            if (v > m || j == 0) m = v;
        }
#if ORACLE_MUTANT == 8
        m = 0.0; /* maximum not subtracted */
#endif
        double sum = 0.0;
#if ORACLE_MUTANT == 9
        const int64_t jend = N > 0 ? N - 1 : 0; /* last term left out of the sum */
#else
        const int64_t jend = N;
#endif
        for (int64_t j = 0; j < jend; ++j) sum += exp(oracle_dec16(xi[j]) - m);
#if ORACLE_MUTANT == 10
        sum = (double)N; /* normalised by the length instead of the sum */
#endif
        for (int64_t j = 0; j < N; ++j) yi[j] = exp(oracle_dec16(xi[j]) - m) / sum;
    }
    return 0;
}

/* ---- symmetric weight quantisation -----------------------------------------
 *
 * "membound", section "The kernel decode actually runs: dequant GEMV": INT8
 * weights with a symmetric scale per row, INT4 with a symmetric scale per
 * group of 128 columns, and the quantisation RMSE of U[-1,1] weights reported
 * next to the kernels (about 2.3e-3 for INT8, 4.1e-2 for INT4).  Those two
 * figures fix the scale as max|w| / 127 and max|w| / 7: rounding to the
 * nearest code leaves a uniform error of RMS s / sqrt(12), i.e.
 * (1/127)/sqrt(12) = 2.27e-3 and (0.992/7)/sqrt(12) = 4.09e-2 (0.992 being the
 * expected maximum of 128 uniform magnitudes).
 *
 * The page does not state the arithmetic; it is read as FP32 throughout, one
 * group at a time:
 *   a   = max |w| over the group                 (exact)
 *   s   = a / qmax                               (binary32 division, nearest even)
 *   s16 = binary16(s), nearest even; an overflow to +inf is replaced by 65504
 *   q   = clamp(rint(w / s16), -qmax, qmax)      (binary32 division; rint ties to even)
 *         and q = 0 where s16 == 0 or w is NaN
 * A group is 128 columns of a row (the last one may be shorter) or a whole
 * row (per_row).  Codes are stored as the GEMV reads them: int8 [M][N], or
 * int4 two per byte with the even column in the low nibble ([M][N/2]).
 * scales: binary16 bits [M][groups].  *sq_err = sum over all weights of
 * (w - s16 * q)^2, in double.
 */

/* binary32 -> binary16 bit pattern, round to nearest, ties to even, written
 * from the IEEE 754 definition (10 fraction bits, exponent bias 15,
 * subnormals with unit 2^-24). */
uint16_t oracle_enc16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)(sign | 0x7E00u); /* NaN */
    if ((u & 0x7FFFFFFFu) == 0x7F800000u) return (uint16_t)(sign | 0x7C00u); /* inf */
    const double v = fabs((double)f);
    if (v < ldexp(1.0, -14)) {
        /* subnormal range: integer multiple of 2^-24 (1024 becomes the
         * smallest normal, whose pattern is the same integer) */
#if ORACLE_MUTANT == 16
        const double t = floor(ldexp(v, 24)); /* truncation instead of rounding */
#else
        const double t = nearbyint(ldexp(v, 24));
#endif
        return (uint16_t)(sign | (uint16_t)t);
    }
    int e;
    frexp(v, &e);       /* v = m * 2^e, m in [0.5, 1) */
    e -= 1;             /* v = (1.f) * 2^e */
#if ORACLE_MUTANT == 16
    double t = floor(ldexp(v, 10 - e));
#else
    double t = nearbyint(ldexp(v, 10 - e)); /* in [1024, 2048] */
#endif
    if (t >= 2048.0) {
        t = 1024.0;
        e += 1;
    }
    if (e > 15) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(t - 1024.0));
}

void oracle_enc16_array(const float *f, uint16_t *out, int64_t n)
{
    for (int64_t k = 0; k < n; ++k) out[k] = oracle_enc16(f[k]);
}

/* w_kind: 0 = FP32 weights, 1 = binary16 bit patterns (widened exactly). */
static float w_in(int w_kind, const void *W, int64_t k)
{
    if (w_kind == 0) return ((const float *)W)[k];
    return (float)oracle_dec16(((const uint16_t *)W)[k]);
}

int oracle_quantize(int bits, int per_row, int w_kind, const void *W, int64_t M, int64_t N,
                    void *A, uint16_t *scales, double *sq_err)
{
    if ((bits != 8 && bits != 4) || (w_kind != 0 && w_kind != 1) || M < 0 || N < 0) return -1;
    if (bits == 4 && (per_row || N % 2)) return -1;
    if (M > 0 && N > 0 && (!W || !A || !scales)) return -1;
#if ORACLE_MUTANT == 13
    const float qmax = bits == 8 ? 127.0f : 8.0f; /* INT4 scale by 8 */
#else
    const float qmax = bits == 8 ? 127.0f : 7.0f;
#endif
#if ORACLE_MUTANT == 15
    const int64_t width = per_row ? N : 64; /* groups of 64 columns */
#else
    const int64_t width = per_row ? N : ORACLE_GROUP;
#endif
    const int64_t groups = N == 0 ? 0 : (per_row ? 1 : n_groups(N));
    double err = 0.0;
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t g = 0; g < groups; ++g) {
            const int64_t j0 = g * width;
            const int64_t j1 = j0 + width < N ? j0 + width : N;
            float a = 0.0f;
            for (int64_t j = j0; j < j1; ++j) {
                const float m = fabsf(w_in(w_kind, W, i * N + j));
                if (m > a) a = m;
            }
            const float s = a / qmax;
            uint16_t s16 = oracle_enc16(s);
            if (s16 == 0x7C00u) s16 = 0x7BFFu;
            scales[i * groups + g] = s16;
            const float sf = (float)oracle_dec16(s16);
            for (int64_t j = j0; j < j1; ++j) {
                const float w = w_in(w_kind, W, i * N + j);
                float q = 0.0f;
                if (sf != 0.0f && w == w) {
#if ORACLE_MUTANT == 14
                    q = truncf(w / sf); /* truncation instead of rounding */
#else
                    q = rintf(w / sf);
#endif
                    q = q > qmax ? qmax : (q < -qmax ? -qmax : q);
                }
                const int code = (int)q;
                if (bits == 8) {
                    ((int8_t *)A)[i * N + j] = (int8_t)code;
                } else {
                    uint8_t *b = (uint8_t *)A + i * (N / 2) + j / 2;
                    const uint8_t nib = (uint8_t)(code & 0xF);
                    *b = (j % 2) ? (uint8_t)((*b & 0x0F) | (nib << 4)) : (uint8_t)((*b & 0xF0) | nib);
                }
                const double d = (double)w - (double)sf * (double)code;
                err += d * d;
            }
        }
    }
    if (sq_err) *sq_err = err;
    return 0;
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }
