/*
 * CPU oracle for the batch-invariant exact GEMM — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct definitions of what the CUDA path computes.
 * Only the tests, the smoke check and the bench's CPU-baseline leg may load this
 * library; the product path never does. It shares no code, header or table with
 * the CUDA library: it is written from the definitions on the source pages.
 *
 * Build flags: -O2 -ffp-contract=off -fno-fast-math (no FMA contraction, IEEE
 * semantics, subnormals kept). OpenMP over output rows only.
 *
 * Sources (page title, section):
 *  [P4] "Deterministic LLM Inference Across GPU Kernels: Power-of-Two INT8
 *       Quantization Scales and the Limits of Tolerance-Based Conformance",
 *       §II "Pipeline and alibi" (Y = (A W^T) * s_a s_w, int32 accumulation,
 *       one rounding to bf16; pow2 commutation), §II.E "Measurement design"
 *       (int64 reference accumulator), §V / §V.C (nearest and ceiling pow2 arms,
 *       weights requantized under the pow2 scale).
 *  [P3] "GPU Mechanism", §3 "Method", Interventions (a) ExactGEMM (frexp-scaled
 *       7-bit integer slices, exact integer slice products, fixed-order fp64
 *       recombination, one rounding); §2 "Exact GEMM by error-free
 *       transformation" (Ozaki scheme).
 *  [P1] "Taming Bitwise Behavior in GPU Kernels with Tensor Core", §3.2.2
 *       (split-K cuts the contracted axis into contiguous parts).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - bf16 rounding is IEEE round-to-nearest-even with subnormals and overflow
 *    to infinity; acc = 0 gives +0; a negative value that underflows gives -0.
 *  - "nearest" power of two is nearest in the log domain; "ceiling" never
 *    shrinks the scale. Quantized values are round-half-even, clamped to +-127.
 *  - slice digits are truncated toward zero, 7 bits each, signed, with the
 *    exponent e of the row/column max from frexp (max|x| < 2^e).
 *  - the slice pairs kept are s + t <= max_diag with slices numbered from 1;
 *    diagonals are combined from the smallest weight (g = max_diag) up to g = 2.
 *
 * Status codes: 0 ok, 3 precondition (|acc| >= 2^31), 8 non-finite input.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_PRECONDITION 3
#define ORACLE_ERR_NONFINITE 8

/* ------------------------------------------------------------------------------------ */
/* Round a double to the nearest bfloat16, ties to even (IEEE 754 RNE).                  */
/* bf16: 8 significant bits, exponent range of fp32, subnormal spacing 2^-133.           */
/* ------------------------------------------------------------------------------------ */
uint16_t oracle_rne_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isinf(a)) return sign | 0x7F80;
    if (a == 0.0) return sign;
    int k;
    frexp(a, &k);                        /* a in [2^(k-1), 2^k) */
    int p = k - 1;                       /* a in [2^p, 2^(p+1)) */
    int q = (p < -126) ? -133 : p - 7;   /* log2 of the bf16 spacing at a */
    double n = ldexp(a, -q);             /* exact: power-of-two scaling */
    double fl = floor(n);
    double fr = n - fl;                  /* exact */
    if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    double r = ldexp(fl, q);             /* exact: fl <= 256 */
    if (r >= 0x1p128) return sign | 0x7F80;
    float f = (float)r;                  /* exact: r is on the bf16 grid */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return sign | (uint16_t)((bits >> 16) & 0x7FFF);
}

static int clamp_exp(int64_t e) {
    /* beyond +-1200 every |acc| * 2^e is 0 or inf in bf16/fp32 after the fp64 step */
    if (e > 1200) return 1200;
    if (e < -1200) return -1200;
    return (int)e;
}

/* ------------------------------------------------------------------------------------ */
/* W8A8 [P4 §II]: acc_ij = sum_k A_ik * W_jk (int64, must fit int32),                    */
/*                C_ij   = rne_bf16(acc_ij * 2^(ea_i + ew_j)).                           */
/* A [M x K] row-major (lda), W [N x K] row-major (ldw) = B^T, C [rows x N] (ldc).        */
/* rows == NULL: all M rows; else output row r is A-row rows[r].                         */
/* ------------------------------------------------------------------------------------ */
int oracle_w8a8(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw, const int32_t* ea,
                const int32_t* ew, uint16_t* C, int64_t ldc, int M, int N, int K,
                const int32_t* rows, int nrows) {
    int n_out = rows ? nrows : M;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int r = 0; r < n_out; ++r) {
        int i = rows ? rows[r] : r;
        for (int j = 0; j < N; ++j) {
            int64_t acc = 0;
            for (int k = 0; k < K; ++k) acc += (int64_t)A[(int64_t)i * lda + k] * (int64_t)W[(int64_t)j * ldw + k];
            if (acc >= 2147483648LL || acc < -2147483648LL) bad = 1;
            double v = ldexp((double)acc, clamp_exp((int64_t)ea[i] + (int64_t)ew[j]));
            C[(int64_t)r * ldc + j] = oracle_rne_bf16(v);
        }
    }
    return bad ? ORACLE_ERR_PRECONDITION : ORACLE_OK;
}

/* ------------------------------------------------------------------------------------ */
/* W8A8 with a bias: the epilogue's one rounding [P4 §II] taken of the exact sum          */
/*   C_ij = rne_bf16(acc_ij * 2^(ea_i + ew_j) + b_j),   b_j a bfloat16 value.             */
/* Readings: b = +-0 leaves the W8A8 result unchanged (x + 0 = x, including the sign of   */
/* an underflowing x); a non-finite b is returned unchanged; an exact zero sum gives +0.  */
/* Route: x = acc * 2^E and b are exact doubles; the double sum s and its error t (the    */
/* classical two-sum, exact without overflow) give the exact sum s + t. Rounding s to     */
/* bf16 is right unless s lies exactly halfway between two bf16 numbers while t != 0:    */
/* every bf16 halfway point is a double, so s and the exact sum are on the same side of   */
/* every other one; in that case the sign of t picks the neighbour.                      */
/* ------------------------------------------------------------------------------------ */
static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

uint16_t oracle_bias_round(int64_t acc, int64_t E, uint16_t b) {
    if ((b & 0x7F80) == 0x7F80) return b;                    /* +-inf, NaN */
    double x = ldexp((double)acc, clamp_exp(E));
    if ((b & 0x7FFF) == 0) return oracle_rne_bf16(x);        /* x + (+-0) = x */
    double bv = bf16_to_double(b);
    if (acc == 0) return oracle_rne_bf16(bv);                /* = b */
    double s = x + bv;
    double z = s - x;
    double t = (x - (s - z)) + (bv - z);                     /* s + t = x + bv exactly */
    if (s == 0.0) return 0;                                  /* exact zero sum: +0 */
    if (isinf(s) || t == 0.0) return oracle_rne_bf16(s);
    double a = fabs(s);
    int k;
    frexp(a, &k);
    int p = k - 1;
    int q = (p < -126) ? -133 : p - 7;                       /* log2 of the bf16 spacing at a */
    double n = ldexp(a, -q);
    double fl = floor(n);
    if (n - fl != 0.5) return oracle_rne_bf16(s);            /* not a halfway point */
    int up = (t > 0.0) == (s > 0.0);                         /* exact |sum| above a? */
    double r = ldexp(up ? fl + 1.0 : fl, q);                 /* on the bf16 grid (or 2^128) */
    return oracle_rne_bf16(s > 0.0 ? r : -r);
}

int oracle_w8a8_bias(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw, const int32_t* ea,
                     const int32_t* ew, const uint16_t* bias, uint16_t* C, int64_t ldc, int M, int N,
                     int K, const int32_t* rows, int nrows) {
    int n_out = rows ? nrows : M;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int r = 0; r < n_out; ++r) {
        int i = rows ? rows[r] : r;
        for (int j = 0; j < N; ++j) {
            int64_t acc = 0;
            for (int k = 0; k < K; ++k) acc += (int64_t)A[(int64_t)i * lda + k] * (int64_t)W[(int64_t)j * ldw + k];
            if (acc >= 2147483648LL || acc < -2147483648LL) bad = 1;
            C[(int64_t)r * ldc + j] = oracle_bias_round(acc, (int64_t)ea[i] + (int64_t)ew[j], bias[j]);
        }
    }
    return bad ? ORACLE_ERR_PRECONDITION : ORACLE_OK;
}

/* The exact int32 accumulator alone: C_ij = sum_k A_ik * W_jk. */
int oracle_gemm_s8_i32(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw, int32_t* C,
                       int64_t ldc, int M, int N, int K, const int32_t* rows, int nrows) {
    int n_out = rows ? nrows : M;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int r = 0; r < n_out; ++r) {
        int i = rows ? rows[r] : r;
        for (int j = 0; j < N; ++j) {
            int64_t acc = 0;
            for (int k = 0; k < K; ++k) acc += (int64_t)A[(int64_t)i * lda + k] * (int64_t)W[(int64_t)j * ldw + k];
            if (acc >= 2147483648LL || acc < -2147483648LL) bad = 1;
            C[(int64_t)r * ldc + j] = (int32_t)acc;
        }
    }
    return bad ? ORACLE_ERR_PRECONDITION : ORACLE_OK;
}

/* ------------------------------------------------------------------------------------ */
/* Pow2 quantization [P4 §V, §V.C]: per row a = max|x|; s = a / 127;                     */
/*   ceiling arm: e = smallest integer with 2^e >= s   (never shrinks the scale)         */
/*   nearest arm: e = the integer nearest to log2(s)   (may clip the row's outliers)     */
/*   q = clamp(rne(x / 2^e), -127, 127).   a == 0: e = 0, q = 0.                          */
/* x_dtype 0 = bf16 bits, 1 = fp32. mode 0 = nearest, 1 = ceiling.                       */
/* ------------------------------------------------------------------------------------ */
static double load_x(const void* X, int x_dtype, int64_t idx) {
    if (x_dtype == 0) {
        uint32_t bits = (uint32_t)((const uint16_t*)X)[idx] << 16;
        float f;
        memcpy(&f, &bits, 4);
        return (double)f;
    }
    return (double)((const float*)X)[idx];
}

int oracle_quantize_pow2(const void* X, int x_dtype, int64_t ldx, int rows, int cols, int mode,
                         int8_t* Q, int64_t ldq, int32_t* e_out) {
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
    for (int i = 0; i < rows; ++i) {
        double a = 0.0;
        for (int j = 0; j < cols; ++j) {
            double x = load_x(X, x_dtype, (int64_t)i * ldx + j);
            if (!isfinite(x)) bad = 1;
            if (fabs(x) > a) a = fabs(x);
        }
        if (!isfinite(a)) { e_out[i] = 0; continue; }
        int e = 0;
        if (a > 0.0) {
            /* smallest e with 127 * 2^e >= a, found by exact comparisons */
            e = ilogb(a) - 7;
            while (ldexp(127.0, e) < a) ++e;
            while (ldexp(127.0, e - 1) >= a) --e;
            if (mode == 0) {
                /* log2(s) >= e - 1/2  <=>  s^2 >= 2^(2e-1)  <=>  a^2 >= 127^2 * 2^(2e-1)
                 * (a has <= 24 significant bits, so a*a is exact in fp64; no tie exists) */
                if (!(a * a >= ldexp(16129.0, 2 * e - 1))) e -= 1;
            }
        }
        e_out[i] = e;
        for (int j = 0; j < cols; ++j) {
            double x = load_x(X, x_dtype, (int64_t)i * ldx + j);
            double q = nearbyint(ldexp(x, -e)); /* default rounding mode: ties to even */
            if (q > 127.0) q = 127.0;
            if (q < -127.0) q = -127.0;
            Q[(int64_t)i * ldq + j] = (int8_t)q;
        }
    }
    return bad ? ORACLE_ERR_NONFINITE : ORACLE_OK;
}

/* ------------------------------------------------------------------------------------ */
/* Ozaki slicing [P3 §3 (a)]: one shared exponent per row (axis 0) or column (axis 1):   */
/*   e = frexp exponent of the max |x|   (max|x| < 2^e; e = 0 for an all-zero line)      */
/*   r = x * 2^-e  in (-1, 1)                                                            */
/*   for t = 1..nslices:  d_t = trunc(r * 2^7);  r = r * 2^7 - d_t                       */
/* All steps are exact in fp64. Output planes S[t-1]:                                    */
/*   axis 0: [rows x cols] row-major;  axis 1: [cols x rows] (each column contiguous).   */
/* ------------------------------------------------------------------------------------ */
static double load_line(const void* X, int f64, int64_t idx) {
    return f64 ? ((const double*)X)[idx] : (double)((const float*)X)[idx];
}

static void slice_line(const void* X, int f64, int64_t stride, int len, int nslices, int8_t* S,
                       int64_t plane, int64_t sstride, int32_t* e_out, int* bad) {
    double a = 0.0;
    for (int k = 0; k < len; ++k) {
        double x = load_line(X, f64, (int64_t)k * stride);
        if (!isfinite(x)) *bad = 1;
        if (fabs(x) > a) a = fabs(x);
    }
    int e = 0;
    if (a > 0.0 && isfinite(a)) frexp(a, &e);
    *e_out = e;
    for (int k = 0; k < len; ++k) {
        double r = ldexp(load_line(X, f64, (int64_t)k * stride), -e);
        if (!isfinite(r)) r = 0.0;
        for (int t = 0; t < nslices; ++t) {
            double v = r * 128.0;
            double d = trunc(v);
            r = v - d;
            S[(int64_t)t * plane + (int64_t)k * sstride] = (int8_t)d;
        }
    }
}

static int slice_any(const void* X, int f64, int64_t ldx, int rows, int cols, int axis, int nslices,
                     int8_t* S, int32_t* e_out) {
    int bad = 0;
    int64_t plane = (int64_t)rows * cols;
    const size_t es = f64 ? sizeof(double) : sizeof(float);
    if (axis == 0) {
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
        for (int i = 0; i < rows; ++i) {
            int b = 0;
            slice_line((const char*)X + (size_t)i * (size_t)ldx * es, f64, 1, cols, nslices,
                       S + (int64_t)i * cols, plane, 1, e_out + i, &b);
            bad |= b;
        }
    } else {
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
        for (int j = 0; j < cols; ++j) {
            int b = 0;
            slice_line((const char*)X + (size_t)j * es, f64, ldx, rows, nslices, S + (int64_t)j * rows,
                       plane, 1, e_out + j, &b);
            bad |= b;
        }
    }
    return bad ? ORACLE_ERR_NONFINITE : ORACLE_OK;
}

int oracle_slice_f32(const float* X, int64_t ldx, int rows, int cols, int axis, int nslices,
                     int8_t* S, int32_t* e_out) {
    return slice_any(X, 0, ldx, rows, cols, axis, nslices, S, e_out);
}

/* The same slicing of an fp64 matrix (every step is still exact in fp64). */
int oracle_slice_f64(const double* X, int64_t ldx, int rows, int cols, int axis, int nslices,
                     int8_t* S, int32_t* e_out) {
    return slice_any(X, 1, ldx, rows, cols, axis, nslices, S, e_out);
}

/* ------------------------------------------------------------------------------------ */
/* Ozaki recombination of one element [P3 §3 (a): fixed-order fp64 recombination, one   */
/* rounding]. T[g] (g = 2..max_diag) are the exact diagonal sums of weight 2^(-7g):       */
/*   acc = 0.0;  for g = max_diag down to 2:  acc = acc + T_g * 2^(-7g)   (fp64)         */
/*   C = (float) (acc * 2^(e + f))                 (one rounding to fp32, RNE)           */
/* ------------------------------------------------------------------------------------ */
static float combine_one(const int64_t* T, int max_diag, int32_t e, int32_t f) {
    double acc = 0.0;
    for (int g = max_diag; g >= 2; --g) acc = acc + ldexp((double)T[g], -7 * g);
    return (float)ldexp(acc, clamp_exp((int64_t)e + (int64_t)f));
}

/* The fp64-target form: the same loop, then C = acc * 2^(e + f) rounded to fp64 (exact   */
/* unless the result is subnormal or overflows). |acc| lies in [2^-126, 2^144), so        */
/* exponents beyond +-2200 give 0 or inf either way.                                      */
static double combine_one_f64(const int64_t* T, int max_diag, int32_t e, int32_t f) {
    double acc = 0.0;
    for (int g = max_diag; g >= 2; --g) acc = acc + ldexp((double)T[g], -7 * g);
    int64_t k = (int64_t)e + (int64_t)f;
    if (k > 2200) k = 2200;
    if (k < -2200) k = -2200;
    return ldexp(acc, (int)k);
}

/* The recombination step alone: T int32 [max_diag - 1][M][ldT], plane p holding the     */
/* diagonal g = max_diag - p; e [M], f [N]; C fp32 [M x N] (row stride ldc).              */
int oracle_ozaki_combine(const int32_t* T, int64_t ldT, int max_diag, const int32_t* e,
                         const int32_t* f, float* C, int64_t ldc, int M, int N) {
    int64_t plane = (int64_t)M * ldT;
#pragma omp parallel for schedule(static)
    for (int i = 0; i < M; ++i) {
        int64_t Tg[19];
        for (int j = 0; j < N; ++j) {
            for (int g = 0; g <= max_diag; ++g) Tg[g] = 0;
            for (int g = 2; g <= max_diag; ++g)
                Tg[g] = T[(int64_t)(max_diag - g) * plane + (int64_t)i * ldT + j];
            C[(int64_t)i * ldc + j] = combine_one(Tg, max_diag, e[i], f[j]);
        }
    }
    return ORACLE_OK;
}

int oracle_ozaki_combine_f64(const int32_t* T, int64_t ldT, int max_diag, const int32_t* e,
                             const int32_t* f, double* C, int64_t ldc, int M, int N) {
    int64_t plane = (int64_t)M * ldT;
#pragma omp parallel for schedule(static)
    for (int i = 0; i < M; ++i) {
        int64_t Tg[19];
        for (int j = 0; j < N; ++j) {
            for (int g = 0; g <= max_diag; ++g) Tg[g] = 0;
            for (int g = 2; g <= max_diag; ++g)
                Tg[g] = T[(int64_t)(max_diag - g) * plane + (int64_t)i * ldT + j];
            C[(int64_t)i * ldc + j] = combine_one_f64(Tg, max_diag, e[i], f[j]);
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------ */
/* Ozaki fp32 GEMM [P3 §3 (a)]: C = A B with A [M x K], B [K x N] fp32 row-major.         */
/*   slice A per row (e_i, DA_s) and B per column (f_j, DB_t);                           */
/*   T_g = sum_{s+t=g, 1<=s,t<=nslices} sum_k DA_s[i,k] * DB_t[k,j]   (exact, int64)     */
/*   acc = 0.0;  for g = max_diag down to 2:  acc = acc + T_g * 2^(-7g)   (fp64)         */
/*   C_ij = (float) (acc * 2^(e_i + f_j))          (one rounding to fp32, RNE)           */
/* rows == NULL: all rows; else output row r is A-row rows[r].                           */
/* ------------------------------------------------------------------------------------ */
static int ozaki_any(const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                     int f64, int M, int N, int K, int nslices, int max_diag, const int32_t* rows,
                     int nrows) {
    int n_out = rows ? nrows : M;
    const size_t es = f64 ? sizeof(double) : sizeof(float);
    int8_t* DB = (int8_t*)malloc((size_t)nslices * N * K);
    int32_t* f = (int32_t*)malloc(sizeof(int32_t) * N);
    int8_t* DA = (int8_t*)malloc((size_t)nslices * n_out * K);
    int32_t* e = (int32_t*)malloc(sizeof(int32_t) * n_out);
    if (!DB || !f || !DA || !e) { free(DB); free(f); free(DA); free(e); return 1; }
    int bad = slice_any(B, f64, ldb, K, N, 1, nslices, DB, f) != 0;
    /* slice the requested rows of A */
    int bad_rows = 0;
    for (int r = 0; r < n_out; ++r) {
        int i = rows ? rows[r] : r;
        int b = 0;
        slice_line((const char*)A + (size_t)i * (size_t)lda * es, f64, 1, K, nslices, DA + (int64_t)r * K,
                   (int64_t)n_out * K, 1, e + r, &b);
        bad_rows |= b;
    }
    int64_t planeA = (int64_t)n_out * K, planeB = (int64_t)N * K;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n_out; ++r) {
        int64_t* T = (int64_t*)malloc(sizeof(int64_t) * (size_t)(max_diag + 1));
        for (int j = 0; j < N; ++j) {
            for (int g = 0; g <= max_diag; ++g) T[g] = 0;
            for (int g = 2; g <= max_diag; ++g) {
                for (int s = 1; s <= nslices; ++s) {
                    int t = g - s;
                    if (t < 1 || t > nslices) continue;
                    const int8_t* da = DA + (int64_t)(s - 1) * planeA + (int64_t)r * K;
                    const int8_t* db = DB + (int64_t)(t - 1) * planeB + (int64_t)j * K;
                    int64_t acc = 0;
                    for (int k = 0; k < K; ++k) acc += (int64_t)da[k] * (int64_t)db[k];
                    T[g] += acc;
                }
            }
            if (f64)
                ((double*)C)[(int64_t)r * ldc + j] = combine_one_f64(T, max_diag, e[r], f[j]);
            else
                ((float*)C)[(int64_t)r * ldc + j] = combine_one(T, max_diag, e[r], f[j]);
        }
        free(T);
    }
    free(DB); free(f); free(DA); free(e);
    return (bad || bad_rows) ? ORACLE_ERR_NONFINITE : ORACLE_OK;
}

int oracle_ozaki_f32(const float* A, int64_t lda, const float* B, int64_t ldb, float* C,
                     int64_t ldc, int M, int N, int K, int nslices, int max_diag,
                     const int32_t* rows, int nrows) {
    return ozaki_any(A, lda, B, ldb, C, ldc, 0, M, N, K, nslices, max_diag, rows, nrows);
}

/* fp64-target Ozaki GEMM: the same slicing of fp64 operands (nslices digits of 7 bits),  */
/* the same exact diagonal sums and fixed-order fp64 combine, and the result              */
/* C_ij = acc * 2^(e_i + f_j) rounded to fp64.                                            */
int oracle_ozaki_f64(const double* A, int64_t lda, const double* B, int64_t ldb, double* C,
                     int64_t ldc, int M, int N, int K, int nslices, int max_diag,
                     const int32_t* rows, int nrows) {
    return ozaki_any(A, lda, B, ldb, C, ldc, 1, M, N, K, nslices, max_diag, rows, nrows);
}

/* Per-diagonal exact sums T_g (int64) for one output element set, for tests of the     */
/* slice GEMMs: T[(r * N + j) * (max_diag + 1) + g].                                     */
int oracle_ozaki_diagonals(const int8_t* DA, const int8_t* DB, int M, int N, int K, int nslices,
                           int max_diag, int64_t* T) {
    int64_t planeA = (int64_t)M * K, planeB = (int64_t)N * K;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < M; ++i) {
        for (int j = 0; j < N; ++j) {
            int64_t* Tij = T + ((int64_t)i * N + j) * (max_diag + 1);
            for (int g = 0; g <= max_diag; ++g) Tij[g] = 0;
            for (int g = 2; g <= max_diag; ++g)
                for (int s = 1; s <= nslices; ++s) {
                    int t = g - s;
                    if (t < 1 || t > nslices) continue;
                    for (int k = 0; k < K; ++k)
                        Tij[g] += (int64_t)DA[(int64_t)(s - 1) * planeA + (int64_t)i * K + k] *
                                  (int64_t)DB[(int64_t)(t - 1) * planeB + (int64_t)j * K + k];
                }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------
 * Fixed-order fp16 / bf16 GEMM under the tensor-core block-FMA model ("GPU Arithmetic
 * Emulator" README, section "Tensor Core Matmul"): the accumulator walks K in blocks of
 * nfma products, from +0, and each block is one block FMA:
 *   1. each product of two significands is formed exactly as an integer, its exponent the
 *      sum of the two exponents (not renormalised);
 *   2. e_max = the largest exponent among the block's nonzero products and the fp32
 *      accumulator (when nonzero);
 *   3. every term is aligned to e_max in a fixed-point window whose lowest bit weighs
 *      2^(e_max - 23 - neab) (23 fraction bits of fp32 plus neab extra bits); bits below
 *      the window are dropped (truncation toward zero of each term's magnitude);
 *   4. the window's integer sum is converted to fp32 by truncation toward zero.
 * The page gives nfma = 16 and neab = 2 for one K = 16 step on H100; the same parameters
 * reproduce GB300's tensor cores (tcgen05.mma kind::f16 and mma.sync) bit for bit.
 * Inputs are bit patterns: dtype 0 = bf16, 3 = fp16 (finite values). Output: fp32 bits.
 * Readings where the page is silent: a zero sum gives +0; a sum at or beyond 2^128 gives
 * the largest finite fp32 of its sign (truncation toward zero); a sum below 2^-126 keeps
 * the fp32 subnormal grid (multiples of 2^-149, truncated).
 * ------------------------------------------------------------------------------------ */
static void decode_half(uint16_t bits, int dtype, int* neg, int64_t* m, int* e) {
    int ebits = dtype == 0 ? 8 : 5, fbits = dtype == 0 ? 7 : 10, bias = dtype == 0 ? 127 : 15;
    int be = (bits >> fbits) & ((1 << ebits) - 1);
    int64_t f = bits & ((1 << fbits) - 1);
    *neg = (bits >> 15) & 1;
    *m = be ? (f | ((int64_t)1 << fbits)) : f; /* value = m * 2^(e - fbits) */
    *e = be ? be - bias : 1 - bias;
}

/* fp32 bits of S * 2^u rounded toward zero */
static uint32_t rz_f32_bits(int64_t S, int u) {
    if (S == 0) return 0;
    uint32_t sign = S < 0 ? 0x80000000u : 0u;
    uint64_t a = S < 0 ? (uint64_t)(-S) : (uint64_t)S;
    int b = 63;
    while (!((a >> b) & 1)) --b;
    int E = b + u;
    if (E > 127) return sign | 0x7F7FFFFFu;
    if (E >= -126) {
        uint64_t top = b >= 23 ? a >> (b - 23) : a << (23 - b);
        return sign | ((uint32_t)(E + 127) << 23) | (uint32_t)(top & 0x7FFFFF);
    }
    int s = -(u + 149); /* units of 2^-149 */
    uint64_t q = s >= 64 ? 0 : (s >= 0 ? a >> s : a << (-s));
    return sign | (uint32_t)q;
}

int oracle_gemm_blockfma(const uint16_t* A, int64_t lda, const uint16_t* W, int64_t ldw, int dtype, int nfma,
                         int neab, uint32_t* C, int64_t ldc, int M, int N, int K) {
    if (nfma < 1 || nfma > 64 || neab < 0 || neab > 8 || (dtype != 0 && dtype != 3)) return 3;
    const int p = dtype == 0 ? 7 : 10;
#pragma omp parallel for schedule(dynamic)
    for (int i = 0; i < M; ++i) {
        for (int j = 0; j < N; ++j) {
            uint32_t acc = 0; /* fp32 bits */
            for (int k0 = 0; k0 < K; k0 += nfma) {
                int64_t pm[64];
                int pe[64], cnt = 0;
                int emax = INT32_MIN;
                for (int k = k0; k < k0 + nfma && k < K; ++k) {
                    int na, nb, xa, xb;
                    int64_t ma, mb;
                    decode_half(A[(int64_t)i * lda + k], dtype, &na, &ma, &xa);
                    decode_half(W[(int64_t)j * ldw + k], dtype, &nb, &mb, &xb);
                    if (ma == 0 || mb == 0) continue;
                    pm[cnt] = (na ^ nb) ? -(ma * mb) : ma * mb; /* value pm * 2^(pe - 2p) */
                    pe[cnt] = xa + xb;
                    if (pe[cnt] > emax) emax = pe[cnt];
                    ++cnt;
                }
                const int acc_nz = (acc & 0x7FFFFFFFu) != 0;
                int aexp = 0;
                int64_t aman = 0;
                if (acc_nz) {
                    int be = (acc >> 23) & 0xFF;
                    aman = (acc & 0x7FFFFF) | (be ? 0x800000 : 0); /* value aman * 2^(aexp - 23) */
                    aexp = be ? be - 127 : -126;
                    if (acc >> 31) aman = -aman;
                    if (aexp > emax) emax = aexp;
                }
                if (cnt == 0 && !acc_nz) continue;
                const int u = emax - 23 - neab; /* weight of the window's lowest bit */
                int64_t S = 0;
                for (int t = 0; t < cnt; ++t) {
                    int sh = pe[t] - 2 * p - u; /* aligned magnitude |pm| * 2^sh, truncated */
                    int64_t mag = pm[t] < 0 ? -pm[t] : pm[t];
                    int64_t al = sh >= 0 ? mag << sh : (-sh >= 63 ? 0 : mag >> (-sh));
                    S += pm[t] < 0 ? -al : al;
                }
                if (acc_nz) {
                    int sh = aexp - 23 - u;
                    int64_t mag = aman < 0 ? -aman : aman;
                    int64_t al = sh >= 0 ? mag << sh : (-sh >= 63 ? 0 : mag >> (-sh));
                    S += aman < 0 ? -al : al;
                }
                acc = rz_f32_bits(S, u);
            }
            C[(int64_t)i * ldc + j] = acc;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------------------
 * Gated linear unit epilogue (SiLU(gate) * up), rounded once to bf16. The gate and up GEMMs
 * of a W8A8 FFN give exact int32 accumulators; with power-of-two scales the exact values are
 * g = gacc * 2^Eg and u = uacc * 2^Eu ("Deterministic LLM Inference ...", §II "Pipeline and
 * alibi": the epilogue rounds once). The output is the one round-to-nearest-even of the real
 * number y = SiLU(g) * u = g * u / (1 + e^-g) to bf16 (subnormals kept, overflow to inf).
 * y is evaluated in 113-bit floating point (IEEE binary128: __float128 with libquadmath on
 * x86-64, long double on AArch64), whose relative error here is below 2^-100; a y within
 * that bound of a rounding boundary is decided by the rule below or reported (status 9).
 *  - gacc == 0 or uacc == 0: y = 0 exactly, result +0.
 *  - y rounds to zero magnitude only when |y| < 2^-134: the sign is that of g * u.
 *  - the only y the 113-bit value cannot place is P * sigma(g) for large g > 0 with the exact
 *    dyadic P = g * u on a rounding boundary (a midpoint); then y is strictly smaller in
 *    magnitude than P (0 < sigma(g) < 1), so it rounds toward zero from P.
 * ------------------------------------------------------------------------------------ */
#if defined(__aarch64__)
typedef long double qreal;
#define QEXP expl
#define QLDEXP ldexpl
#define QFREXP frexpl
#define QFLOOR floorl
#else
#include <quadmath.h>
typedef __float128 qreal;
#define QEXP expq
#define QLDEXP ldexpq
#define QFREXP frexpq
#define QFLOOR floorq
#endif

/* bf16 rounding of a positive quad y known to relative error releps: 0 ok, 1 undecidable
 * (with *at_mid = 1 when the value sits within the bound of a midpoint) */
static int bf16_round_quad(qreal y, qreal releps, uint16_t* mag, int* at_mid) {
    *at_mid = 0;
    int e;
    QFREXP(y, &e); /* y = f * 2^e, f in [0.5, 1): leading bit 2^(e-1) */
    int lead = e - 1;
    qreal m;    /* y in units of the bf16 spacing at y */
    int base;   /* bit pattern of the bf16 value m = 0 (units of the spacing) in this binade */
    if (lead >= -126) {
        if (lead > 127) {
            *mag = 0x7F80;
            return 0;
        }
        m = QLDEXP(y, 7 - lead); /* in [128, 256) */
        base = ((lead + 127) << 7) - 128;
    } else {
        m = QLDEXP(y, 133); /* units of 2^-133, in [0, 128) */
        base = 0;
    }
    qreal fl = QFLOOR(m);
    qreal fr = m - fl;
    qreal tol = releps * m;
    qreal d = fr - (qreal)0.5;
    if (d < 0) d = -d;
    if (d <= tol) {
        *at_mid = 1;
        *mag = (uint16_t)(base + (int)fl); /* the value below the midpoint */
        return 1;
    }
    int q = (int)fl + (fr > (qreal)0.5 ? 1 : 0);
    int bits = base + q; /* a carry into the next binade or to inf works by itself */
    if (bits > 0x7F80) bits = 0x7F80;
    *mag = (uint16_t)bits;
    return 0;
}

int oracle_silu_mul_bf16(int32_t gacc, int32_t uacc, int32_t Eg, int32_t Eu, uint16_t* out) {
    if (gacc == 0 || uacc == 0) {
        *out = 0x0000;
        return 0;
    }
    if (Eg < -16000 || Eg > 16000 || Eu < -16000 || Eu > 16000) return 3;
    const qreal g = QLDEXP((qreal)gacc, Eg);
    const qreal u = QLDEXP((qreal)uacc, Eu);
    const int neg = (gacc < 0) != (uacc < 0);
    const qreal P = g * u; /* exact: two 31-bit significands */
    const qreal y = P / (1 + QEXP(-g));
    const qreal ay = y < 0 ? -y : y;
    if (ay == 0 || ay < QLDEXP((qreal)1, -134)) {
        *out = neg ? 0x8000 : 0x0000;
        return 0;
    }
    uint16_t mag;
    int at_mid;
    if (bf16_round_quad(ay, QLDEXP((qreal)1, -100), &mag, &at_mid) == 0) {
        *out = (uint16_t)(mag | (neg ? 0x8000 : 0));
        return 0;
    }
    /* within 2^-100 of a midpoint: only P on a midpoint with e^-g below the precision (g > 0
     * large) can land here; y is just below |P|, which rounds toward zero */
    uint16_t pmag;
    int pmid;
    const qreal aP = P < 0 ? -P : P;
    if (g > 0 && bf16_round_quad(aP, 0, &pmag, &pmid) == 1 && pmid && ay <= aP) {
        *out = (uint16_t)(pmag | (neg ? 0x8000 : 0));
        return 0;
    }
    return 9;
}

/* C = rne_bf16(SiLU(g) * u) for the gate GEMM A Wg^T and the up GEMM A Wu^T (int64 sums,
 * exponents ea_i + ewg_j and ea_i + ewu_j); rows: optional subset of output rows */
int oracle_w8a8_swiglu(const int8_t* A, int64_t lda, const int8_t* Wg, const int8_t* Wu, int64_t ldw,
                       const int32_t* ea, const int32_t* ewg, const int32_t* ewu, uint16_t* C, int64_t ldc, int M,
                       int N, int K, const int32_t* rows, int nrows) {
    const int R = rows ? nrows : M;
    int status = 0;
#pragma omp parallel for schedule(dynamic)
    for (int r = 0; r < R; ++r) {
        const int i = rows ? rows[r] : r;
        for (int j = 0; j < N; ++j) {
            int64_t g = 0, u = 0;
            for (int k = 0; k < K; ++k) {
                g += (int64_t)A[(int64_t)i * lda + k] * Wg[(int64_t)j * ldw + k];
                u += (int64_t)A[(int64_t)i * lda + k] * Wu[(int64_t)j * ldw + k];
            }
            int st = 3;
            if (g > INT32_MIN && g <= INT32_MAX && u > INT32_MIN && u <= INT32_MAX)
                st = oracle_silu_mul_bf16((int32_t)g, (int32_t)u, ea[i] + ewg[j], ea[i] + ewu[j],
                                          &C[(int64_t)r * ldc + j]);
            if (st) {
#pragma omp atomic write
                status = st;
            }
        }
    }
    return status;
}
