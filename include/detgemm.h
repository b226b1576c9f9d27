/*
 * detgemm — batch-invariant exact GEMM for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libdetgemm.so. Every output bit is a function of the operands alone:
 * it does not depend on the tile shape, the split-K count, the number of rows M
 * or the launch configuration, because every reduction is an exact integer sum
 * and every result is rounded exactly once.
 *
 * Sources (page title, section):
 *  [P4] "Deterministic LLM Inference Across GPU Kernels: Power-of-Two INT8
 *       Quantization Scales and the Limits of Tolerance-Based Conformance",
 *       §II "Pipeline and alibi"; §V and §V.C (power-of-two requantization).
 *  [P3] "GPU Mechanism", §3 "Method", Interventions (a) ExactGEMM; §2 "Exact GEMM
 *       by error-free transformation" (Ozaki scheme).
 *  [P1] "Taming Bitwise Behavior in GPU Kernels with Tensor Core", §3.2.2
 *       (split-K: contiguous parts of the contracted axis, summed afterwards).
 *
 * Conventions for every call:
 *  - All array pointers are DEVICE pointers owned by the caller. The library
 *    allocates no device memory on any call; scratch space is the caller's
 *    `ws` buffer of at least the size the matching *_workspace_size() returns.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *  - Argument, alignment and precondition errors are detected on the host before
 *    anything is launched; the call then returns the error and has no effect.
 *  - Conditions only the device can see (a non-finite input to the quantizer or
 *    the slicer; a bounded wait that expired) set a per-device status word that
 *    detgemm_get_device_status() reads and clears.
 *  - Matrices are row-major with a leading dimension in ELEMENTS. Operands of the
 *    integer GEMMs are K-major: A is [M x K] (lda >= K), W = B^T is [N x K]
 *    (ldw >= K), as an nn.Linear weight is stored.
 *  - Base pointers must be 16-byte aligned and every leading dimension times the
 *    element size a multiple of 16 bytes (DETGEMM_ERR_ALIGNMENT otherwise).
 *  - The library is thread-safe; it keeps only a mutex-guarded per-device cache
 *    of device properties. It never falls back to a CPU path.
 */
#ifndef DETGEMM_H
#define DETGEMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DETGEMM_API __attribute__((visibility("default")))
#else
#define DETGEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* detgemm_stream_t; /* identical to cudaStream_t */

typedef enum detgemm_status {
    DETGEMM_OK = 0,
    DETGEMM_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad enum value */
    DETGEMM_ERR_ALIGNMENT = 2,          /* pointer or leading dimension not 16-byte aligned */
    DETGEMM_ERR_PRECONDITION = 3,       /* the int32 accumulator could overflow (K too large) */
    DETGEMM_ERR_WORKSPACE = 4,          /* ws missing or smaller than *_workspace_size() */
    DETGEMM_ERR_UNSUPPORTED_DEVICE = 5, /* current device is not compute capability 10.3 */
    DETGEMM_ERR_CUDA = 6,               /* a CUDA runtime call or launch failed */
    DETGEMM_ERR_TIMEOUT = 7,            /* a bounded device-side wait expired */
    DETGEMM_ERR_NONFINITE = 8,          /* inf or NaN in a floating-point input */
    DETGEMM_ERR_RANGE = 9               /* a scale exponent outside an epilogue's range */
} detgemm_status;

enum { DETGEMM_DTYPE_BF16 = 0, DETGEMM_DTYPE_F32 = 1, DETGEMM_DTYPE_F64 = 2, DETGEMM_DTYPE_F16 = 3 };
enum { DETGEMM_POW2_NEAREST = 0, DETGEMM_POW2_CEIL = 1 };
enum { DETGEMM_AXIS_ROWS = 0, DETGEMM_AXIS_COLS = 1 };

/* Largest K for which K * 128^2 < 2^31: below it, int8 operands of any value
 * accumulate exactly in int32, which is the bound under which [P4] §II argues that
 * every tiling and split of K produces the same accumulator. */
#define DETGEMM_MAX_K 131071

/* Human-readable name of a status code (static string, never NULL). */
DETGEMM_API const char* detgemm_status_string(detgemm_status status);

/* Library version as 10000*major + 100*minor + patch. */
DETGEMM_API int detgemm_version(void);

/*
 * W8A8 linear layer [P4 §II "Pipeline and alibi"]:
 *     acc_ij = sum_k A_ik * W_jk                      (exact, int32)
 *     C_ij   = rne_bf16(acc_ij * 2^(ea_i + ew_j))     (one rounding, IEEE RNE,
 *                                                      subnormals kept, overflow -> inf)
 * The activation and weight scales are the powers of two s_a = 2^ea, s_w = 2^ew,
 * so the scale is applied exactly and the only rounding is the final one.
 *
 *   A   int8  [M x K], row stride lda          ea  int32 [M]  activation exponents
 *   W   int8  [N x K], row stride ldw (= B^T)  ew  int32 [N]  weight exponents
 *   C   bf16 bit patterns (uint16) [M x N], row stride ldc
 *   split_k  number of contiguous K parts computed by separate CTAs and summed
 *            exactly ([P1] §3.2.2); 1 <= split_k <= ceil(K / 64). The output bits do
 *            not depend on it. Decode-shaped problems (M <= 64, bound by reading W)
 *            choose their own cut: K <= 4096 gives each CTA whole rows of W over all of
 *            K, longer K is divided among all SMs so that every SM streams the same
 *            number of bytes; split_k is then accepted but does not change the cut.
 *            Elsewhere split_k is an upper bound: the tensor-core engine lowers it until
 *            every K part of every output tile runs in one round of its CTA pairs and each
 *            part keeps at least 256 K (more parts would only add rounds).
 *   ws       scratch of ws_bytes >= detgemm_w8a8_workspace_size(M, N, K, split_k)
 *            (nonzero for decode-shaped problems at any split_k, and for split_k > 1).
 * Empty problems (M == 0 or N == 0) return DETGEMM_OK and launch nothing.
 * Errors: INVALID_ARG (K < 1, M or N < 0, split_k out of range, null pointer),
 *         PRECONDITION (K > DETGEMM_MAX_K), ALIGNMENT, WORKSPACE, UNSUPPORTED_DEVICE, CUDA.
 */
DETGEMM_API detgemm_status detgemm_w8a8(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw,
                            const int32_t* ea, const int32_t* ew, uint16_t* C, int64_t ldc,
                            int M, int N, int K, int split_k, void* ws, size_t ws_bytes,
                            detgemm_stream_t stream);

/* Bytes of scratch detgemm_w8a8 needs for this problem (0 is a valid answer). */
DETGEMM_API size_t detgemm_w8a8_workspace_size(int M, int N, int K, int split_k);

/*
 * detgemm_w8a8 with the K cut made exactly as asked, for verifying batch invariance
 * [P4 §II "Pipeline and alibi": the int32 accumulator, hence every output bit, is the
 * same for every tiling and split of K; P1 §3.2.2: split-K as contiguous parts of K whose
 * partial sums are added afterwards]. detgemm_w8a8 treats split_k as a bound and may run
 * fewer parts, or (decode-shaped problems) its own cut; this call runs the requested cut,
 * whatever it costs, so that tests can compare results across cuts that really differ.
 *  - M > 64 (tensor-core engine): every 256-row output tile's 64-wide K blocks are cut
 *    into exactly split_k contiguous parts (part z: blocks [z*B/split_k, (z+1)*B/split_k)
 *    of B), whose exact int32 partials are added in the split workspace.
 *  - M <= 64 (decode kernels): every 128-row block of W has its 128-wide K blocks cut
 *    into exactly min(split_k, ceil(K / 128)) contiguous parts, one CTA each, whose
 *    partials meet through int32 atomics; this holds at split_k == 1 too (one CTA per row
 *    block over all of K), where detgemm_w8a8 would use its whole-K kernel for K <= 4096.
 *   parts_run  if not NULL, receives the number of K parts actually run (0 on error).
 * Arguments, layout, result bits, workspace (detgemm_w8a8_workspace_size with the same
 * split_k) and errors are those of detgemm_w8a8. Slower than detgemm_w8a8 at most cuts.
 */
DETGEMM_API detgemm_status detgemm_w8a8_split_exact(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw,
                                                    const int32_t* ea, const int32_t* ew, uint16_t* C, int64_t ldc,
                                                    int M, int N, int K, int split_k, void* ws, size_t ws_bytes,
                                                    int* parts_run, detgemm_stream_t stream);

/*
 * W8A8 linear layer with a bias, still rounded once [P4 §II "Pipeline and alibi": the
 * epilogue is the single rounding of the exactly scaled int32 accumulator; the bias is
 * added to that exact value before the rounding, not to the rounded output]:
 *     C_ij = rne_bf16(acc_ij * 2^(ea_i + ew_j) + b_j)
 * The sum is exact (both terms are dyadic), so the bits depend on the operands alone,
 * as for detgemm_w8a8. An exact zero sum gives +0; b_j = +-0 gives detgemm_w8a8's bits; a
 * non-finite b_j (+-inf, NaN) is returned unchanged in column j.
 *   bias  bf16 bit patterns [N], device memory, 2-byte aligned, not NULL
 * Everything else (operands, split_k, scratch: detgemm_w8a8_workspace_size, errors) as
 * detgemm_w8a8; a NULL bias is INVALID_ARG, an odd address ALIGNMENT.
 */
DETGEMM_API detgemm_status detgemm_w8a8_bias(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw,
                                             const int32_t* ea, const int32_t* ew, const uint16_t* bias,
                                             uint16_t* C, int64_t ldc, int M, int N, int K, int split_k,
                                             void* ws, size_t ws_bytes, detgemm_stream_t stream);

/*
 * The exact integer accumulator alone [P4 §II: the int32 accumulator is the same for
 * every tiling, split of K and summation order]:  C_ij = sum_k A_ik * W_jk (int32).
 * Same operands, layout, split_k and errors as detgemm_w8a8; C is int32 [M x N].
 * Scratch: detgemm_w8a8_workspace_size(M, N, K, split_k).
 */
DETGEMM_API detgemm_status detgemm_gemm_s8_i32(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw,
                                   int32_t* C, int64_t ldc, int M, int N, int K, int split_k,
                                   void* ws, size_t ws_bytes, detgemm_stream_t stream);

/*
 * Power-of-two quantization of each row [P4 §V, §V.C: scales requantized to a power
 * of two, and the int8 values requantized under that scale]:
 *     a_i = max_j |X_ij|;   s_i = a_i / 127
 *     mode NEAREST: e_i = the integer nearest to log2(s_i)   (may clip outliers)
 *     mode CEIL:    e_i = the smallest integer with 2^e_i >= s_i   (never clips)
 *     Q_ij = clamp(rne(X_ij / 2^e_i), -127, 127);   a_i == 0 gives e_i = 0, Q = 0.
 *   X  [rows x cols], bf16 bit patterns (x_dtype BF16) or fp32 (x_dtype F32), stride ldx
 *   Q  int8 [rows x cols], stride ldq;   e  int32 [rows]
 * Used for activations (rows = tokens) and for weights (rows = output channels of W).
 * A non-finite input sets DETGEMM_ERR_NONFINITE in the device status word; the
 * affected row then gets e = 0 and Q = 0.
 */
DETGEMM_API detgemm_status detgemm_quantize_pow2(const void* X, int x_dtype, int64_t ldx, int rows, int cols,
                                     int mode, int8_t* Q, int64_t ldq, int32_t* e,
                                     detgemm_stream_t stream);

/*
 * W8A8 linear layer on floating-point activations [P4 §II "Pipeline and alibi" with
 * the activation side quantized under a power-of-two scale as in §V]: the two calls
 * detgemm_quantize_pow2 + detgemm_w8a8 in one, with the same result bits:
 *     (Q, ea) = quantize_pow2(X, mode)                   (per row, as detgemm_quantize_pow2)
 *     C_ij    = rne_bf16((sum_k Q_ik W_jk) * 2^(ea_i + ew_j))
 * Outside the decode-shaped problems (M <= 64) the quantizer writes the activation
 * operand directly in the tensor cores' exact fp16 carrier form, so no int8 copy of it is
 * written or widened.
 *   X      [M x K] bf16 bit patterns (x_dtype BF16) or fp32 (x_dtype F32), stride ldx
 *   mode   DETGEMM_POW2_NEAREST or DETGEMM_POW2_CEIL
 *   W      int8 [N x K] (ldw), ew int32 [N]
 *   W16    optional (may be NULL): the same weight widened once by detgemm_widen_i8_f16
 *          (fp16 [N x ldw16], ldw16 a multiple of 8); when given, the tensor-core path
 *          reads it instead of widening W on every call (a static weight widened at
 *          load time); the decode-shaped path reads the int8 W
 *   C      bf16 bit patterns [M x N] (ldc)
 *   ea_out optional (may be NULL): int32 [M] receives the activation exponents
 *   split_k, errors: as detgemm_w8a8; a non-finite row of X raises
 *          DETGEMM_ERR_NONFINITE in the device status word (that row is quantized to 0)
 *   ws     scratch of at least detgemm_linear_w8a8_workspace_size(M, N, K, split_k,
 *          W16 != NULL) bytes, 256-byte aligned
 */
DETGEMM_API detgemm_status detgemm_linear_w8a8(const void* X, int x_dtype, int64_t ldx, int mode, const int8_t* W,
                                               int64_t ldw, const uint16_t* W16, int64_t ldw16, const int32_t* ew,
                                               uint16_t* C, int64_t ldc, int32_t* ea_out, int M, int N, int K,
                                               int split_k, void* ws, size_t ws_bytes, detgemm_stream_t stream);

DETGEMM_API size_t detgemm_linear_w8a8_workspace_size(int M, int N, int K, int split_k, int have_w16);

/*
 * detgemm_linear_w8a8 with a bias per output column, added before the one rounding as in
 * detgemm_w8a8_bias:  C_ij = rne_bf16((sum_k Q_ik W_jk) * 2^(ea_i + ew_j) + b_j).
 *   bias  bf16 bit patterns [N], device memory, 2-byte aligned, not NULL
 * Scratch: detgemm_linear_w8a8_workspace_size; other arguments and errors as
 * detgemm_linear_w8a8.
 */
DETGEMM_API detgemm_status detgemm_linear_w8a8_bias(const void* X, int x_dtype, int64_t ldx, int mode,
                                                    const int8_t* W, int64_t ldw, const uint16_t* W16,
                                                    int64_t ldw16, const int32_t* ew, const uint16_t* bias,
                                                    uint16_t* C, int64_t ldc, int32_t* ea_out, int M, int N,
                                                    int K, int split_k, void* ws, size_t ws_bytes,
                                                    detgemm_stream_t stream);

/*
 * Ozaki slicing of an fp32 matrix [P3 §3 (a): each operand becomes 7-bit integer
 * slices under a power-of-two scale taken from frexp]. One shared exponent per row
 * (axis ROWS) or per column (axis COLS):
 *     e = the frexp exponent of the line's max |x|  (max|x| < 2^e; 0 for a zero line)
 *     r = x * 2^-e in (-1, 1);  for t = 1..nslices: d_t = trunc(128 r), r = 128 r - d_t
 * so that x = 2^e * sum_t d_t 2^(-7t) + (a remainder below 2^(e - 7 nslices)).
 *   X  fp32 [rows x cols], stride ldx
 *   S  int8 digit planes, packed: axis ROWS -> [nslices][rows][cols];
 *      axis COLS -> [nslices][cols][rows] (each column contiguous, i.e. K-major for B)
 *   e  int32 [rows] (ROWS) or [cols] (COLS);   1 <= nslices <= 9
 * A non-finite input sets DETGEMM_ERR_NONFINITE in the device status word.
 */
DETGEMM_API detgemm_status detgemm_slice_f32(const float* X, int64_t ldx, int rows, int cols, int axis,
                                 int nslices, int8_t* S, int32_t* e, detgemm_stream_t stream);

/*
 * Ozaki-scheme fp32 GEMM C = A B [P3 §3 (a) ExactGEMM]:
 *   slice A per row (e_i, DA_s) and B per column (f_j, DB_t), s, t = 1..nslices;
 *   T_g = sum_{s+t=g} DA_s DB_t^T                     (exact int32, g = 2..max_diag)
 *   acc = 0.0;  for g = max_diag down to 2: acc = acc + T_g * 2^(-7g)      (fp64)
 *   C_ij = (float)(acc * 2^(e_i + f_j))                (the one rounding, IEEE RNE)
 *   A fp32 [M x K] (lda), B fp32 [K x N] row-major (ldb), C fp32 [M x N] (ldc)
 *   nslices in [1, 9], max_diag in [2, 2 * nslices]; split_k >= 1 (bits independent).
 * Precondition: every T_g stays in int32: (max_diag - 1) * K * 127^2 < 2^31.
 * Errors as detgemm_w8a8; non-finite inputs set DETGEMM_ERR_NONFINITE on the device.
 */
DETGEMM_API detgemm_status detgemm_ozaki_f32(const float* A, int64_t lda, const float* B, int64_t ldb,
                                 float* C, int64_t ldc, int M, int N, int K, int nslices,
                                 int max_diag, int split_k, void* ws, size_t ws_bytes,
                                 detgemm_stream_t stream);

/* Bytes of scratch detgemm_ozaki_f32 needs for this problem. */
DETGEMM_API size_t detgemm_ozaki_workspace_size(int M, int N, int K, int nslices, int max_diag, int split_k);

/*
 * detgemm_ozaki_f32 with every diagonal's slice-product sum cut into exactly split_k
 * contiguous K parts, for verifying that the result does not depend on the cut [P3 §3 (a):
 * each T_g is an exact integer; P1 §3.2.2: split-K as contiguous parts of K]. For each
 * 256 x 256 output tile of diagonal g, the flattened range of its (g - 1 slice pairs) x
 * (64-wide K blocks) is cut into split_k parts whose exact int32 partials are added in
 * the split workspace. detgemm_ozaki_f32 may run fewer parts than split_k.
 *   parts_run  if not NULL, receives the number of parts run (0 on error).
 * Arguments, result bits, workspace (detgemm_ozaki_workspace_size with the same split_k)
 * and errors are those of detgemm_ozaki_f32.
 */
DETGEMM_API detgemm_status detgemm_ozaki_f32_split_exact(const float* A, int64_t lda, const float* B,
                                                         int64_t ldb, float* C, int64_t ldc, int M, int N, int K,
                                                         int nslices, int max_diag, int split_k, void* ws,
                                                         size_t ws_bytes, int* parts_run,
                                                         detgemm_stream_t stream);

/*
 * The recombination step of the Ozaki GEMMs alone [P3 §3 (a): the exact slice products
 * are recombined in a fixed order in fp64 and rounded once]:
 *   acc = 0.0;  for g = max_diag down to 2: acc = acc + T_g * 2^(-7g)      (fp64, RNE)
 *   C_ij = acc * 2^(e_i + f_j) rounded once to the output type           (IEEE RNE,
 *          c_dtype DETGEMM_DTYPE_F32 as detgemm_ozaki_f32,                 subnormals kept,
 *          or DETGEMM_DTYPE_F64 as detgemm_ozaki_f64)                      overflow -> inf)
 *   T  int32 [max_diag - 1][M][ldT]: plane p holds the diagonal sum T_g with
 *      g = max_diag - p (largest g first, the order of the loop); ldT >= N
 *   e  int32 [M] row exponents, f int32 [N] column exponents (any values)
 *   C  fp32 or fp64 [M x N], row stride ldc;   2 <= max_diag <= 18
 * The result bits are those of the fp64 loop as written, whichever way the library
 * evaluates it. Errors: INVALID_ARG, ALIGNMENT (T and C 16-byte aligned, ldT a multiple
 * of 4, ldc times the element size a multiple of 16; e and f 4-byte aligned),
 * UNSUPPORTED_DEVICE, CUDA.
 */
DETGEMM_API detgemm_status detgemm_ozaki_combine(const int32_t* T, int64_t ldT, int max_diag, const int32_t* e,
                                                 const int32_t* f, void* C, int c_dtype, int64_t ldc, int M, int N,
                                                 detgemm_stream_t stream);

/*
 * Ozaki slicing of an fp64 matrix: detgemm_slice_f32's definition applied to fp64
 * values (every step is exact), 1 <= nslices <= 12 (84 bits; 8 cover fp64's 53-bit
 * significand with 3 bits of headroom below the line's largest element).
 */
DETGEMM_API detgemm_status detgemm_slice_f64(const double* X, int64_t ldx, int rows, int cols, int axis,
                                             int nslices, int8_t* S, int32_t* e, detgemm_stream_t stream);

/*
 * Ozaki-scheme fp64 GEMM C = A B (DGEMM emulation on exact integer slice products) —
 * [P3 §3 (a)] applied to fp64 operands:
 *   slice A per row (e_i, DA_s) and B per column (f_j, DB_t), s, t = 1..nslices;
 *   T_g = sum_{s+t=g} DA_s DB_t^T                     (exact int32, g = 2..max_diag)
 *   acc = 0.0;  for g = max_diag down to 2: acc = acc + T_g * 2^(-7g)      (fp64)
 *   C_ij = acc * 2^(e_i + f_j) rounded to fp64        (exact unless subnormal / overflow)
 *   A fp64 [M x K] (lda), B fp64 [K x N] row-major (ldb), C fp64 [M x N] (ldc)
 *   1 <= nslices <= 12, 2 <= max_diag <= min(2 nslices, 18); the usual choice is
 *   nslices = 8, max_diag = 9 (36 slice pairs). Accuracy is relative to the lines'
 *   largest elements: |C - AB|_ij <= 2^-53 |C_ij| + 10 K 2^(e_i + f_j - 53) for
 *   nslices = 8, max_diag = 9 (more slices for operands that span many binades).
 * Precondition: min(max_diag - 1, nslices) * K * 127^2 < 2^31 (K <= 16644 for 8 slices).
 * Errors as detgemm_ozaki_f32; non-finite inputs set DETGEMM_ERR_NONFINITE on the device.
 */
DETGEMM_API detgemm_status detgemm_ozaki_f64(const double* A, int64_t lda, const double* B, int64_t ldb,
                                             double* C, int64_t ldc, int M, int N, int K, int nslices,
                                             int max_diag, int split_k, void* ws, size_t ws_bytes,
                                             detgemm_stream_t stream);

/* Bytes of scratch detgemm_ozaki_f64 needs for this problem. */
DETGEMM_API size_t detgemm_ozaki_f64_workspace_size(int M, int N, int K, int nslices, int max_diag, int split_k);

/*
 * Exact int8 -> fp16 copy (every int8 value is an fp16 value): Y[r][k] = X[r][k] for
 * k < cols and Y[r][k] = 0 for cols <= k < ldy, i.e. the whole row stride of Y is written.
 * The tensor-core W8A8 path consumes operands in this form; widening a static weight
 * once (at load time) and calling detgemm_w8a8_f16ops skips that step per call.
 *   X int8 [rows x cols] (ldx, multiple of 16); Y fp16 bit patterns [rows x ldy]
 *   (ldy >= cols, multiple of 8). Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED_DEVICE, CUDA.
 */
DETGEMM_API detgemm_status detgemm_widen_i8_f16(const int8_t* X, int64_t ldx, int rows, int cols, uint16_t* Y,
                                                int64_t ldy, detgemm_stream_t stream);

/*
 * Gated-linear-unit epilogue on exact accumulators [P4 §II "Pipeline and alibi": the epilogue
 * is one rounding of the exactly scaled int32 accumulator; an FFN's gate SiLU(g) = g / (1 + e^-g)
 * and the product with the up projection join before that rounding]:
 *     g = G_ij 2^(ea_i + ewg_j),  u = U_ij 2^(ea_i + ewu_j)          (exact)
 *     C_ij = rne_bf16(SiLU(g) * u)            (one rounding of the real value; +0 when g or u is 0)
 * The value is transcendental; it is evaluated in fp32, float-float, fp64 and double-double
 * arithmetic in turn, each with a proven error bound, until no bf16 rounding boundary lies
 * within the bound (a gate g >= 64 is decided exactly from g * u), so the result is the
 * correctly rounded one and depends on the operands alone.
 *   G, U  int32 [M x N] (e.g. from detgemm_gemm_s8_i32 on the gate and up weights), row
 *         strides ldg, ldu;   ea int32 [M], ewg, ewu int32 [N];   C bf16 bits [M x N] (ldc)
 * The exponent sums ea_i + ewg_j and ea_i + ewu_j must lie in [-60, 40]; otherwise that
 * output is a NaN and DETGEMM_ERR_RANGE is set in the device status word (also raised, at a
 * rate far below one in 2^60 outputs, by a value within 2^-90 of a rounding boundary).
 * All pointers device memory, 4-byte aligned (C 2-byte). Errors: INVALID_ARG, ALIGNMENT,
 * UNSUPPORTED_DEVICE, CUDA.
 */
DETGEMM_API detgemm_status detgemm_swiglu_bf16(const int32_t* G, int64_t ldg, const int32_t* U, int64_t ldu,
                                               const int32_t* ea, const int32_t* ewg, const int32_t* ewu,
                                               uint16_t* C, int64_t ldc, int M, int N, detgemm_stream_t stream);

/*
 * Gated-linear-unit W8A8 layer, fused: the gate and up GEMMs on the same activations and the
 * epilogue above, in one tensor-core pass [P4 §II "Pipeline and alibi"]:
 *     C_ij = rne_bf16(SiLU(sum_k A_ik Wg_jk * 2^(ea_i + ewg_j)) * sum_k A_ik Wu_jk * 2^(ea_i + ewu_j))
 * Exact int32 accumulation as in detgemm_w8a8, one rounding per output, bits identical to
 * detgemm_gemm_s8_i32 on Wg and Wu followed by detgemm_swiglu_bf16. Every M runs on the
 * tensor-core engine (rows of the gate and up weights interleaved in its B operand tile).
 *   A  int8 [M x K] (lda);  Wg, Wu int8 [N x K] with the same row stride ldw;
 *   ea int32 [M], ewg, ewu int32 [N];  C bf16 bits [M x N] (ldc)
 *   ws scratch of ws_bytes >= detgemm_w8a8_swiglu_workspace_size(M, N, K), 256-byte aligned
 * Exponent sums outside [-60, 40] give NaN and DETGEMM_ERR_RANGE on the device.
 * Errors: INVALID_ARG, PRECONDITION (K > DETGEMM_MAX_K), ALIGNMENT, WORKSPACE,
 * UNSUPPORTED_DEVICE, CUDA.
 */
DETGEMM_API detgemm_status detgemm_w8a8_swiglu(const int8_t* A, int64_t lda, const int8_t* Wg, const int8_t* Wu,
                                               int64_t ldw, const int32_t* ea, const int32_t* ewg,
                                               const int32_t* ewu, uint16_t* C, int64_t ldc, int M, int N, int K,
                                               void* ws, size_t ws_bytes, detgemm_stream_t stream);

DETGEMM_API size_t detgemm_w8a8_swiglu_workspace_size(int M, int N, int K);

/*
 * Fixed-order (batch-invariant) fp16 / bf16 GEMM. A floating-point GEMM's bits are fixed by
 * its reduction order, which can be written down as a descriptor [P1 §3.2.1-§3.2.2]; here the
 * order is the tensor core's own, one block FMA per 16 products ["GPU Arithmetic Emulator"
 * README, "Tensor Core Matmul": the block's exact products and the fp32 accumulator are
 * aligned to their largest exponent, 23 + 2 fraction bits kept by truncation toward zero, and
 * the sum truncated to fp32]:
 *     acc = +0;  for k0 = 0, 16, 32, ... < K:  acc = block_fma(acc, A_i[k0 .. k0+15], W_j[k0 .. k0+15])
 *     C_ij = acc   (fp32; a tail block is padded with zeros)
 * Descriptor: K walked in increasing 16-wide blocks from a +0 accumulator, never split. Each
 * output depends only on its row of A and its row of W: the bits do not depend on M, N, the
 * tiling or the launch. Products of the tensor core, measured on GB300, follow this model
 * bit for bit with the parameters above (16 products per block, 2 extra window bits).
 *   A  [M x K] fp16 or bf16 bit patterns, row stride lda (a multiple of 8)
 *   W  [N x K] (= B^T) of the same type, row stride ldw (a multiple of 8)
 *   C  fp32 [M x N], row stride ldc (a multiple of 4);   dtype DETGEMM_DTYPE_F16 or _BF16
 * Inputs must be finite; outputs whose partial sums overflow fp32 or fall below its normal
 * range are outside the model this library is checked against. No workspace.
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED_DEVICE, CUDA.
 */
DETGEMM_API detgemm_status detgemm_gemm_fixed_f16(const uint16_t* A, int64_t lda, const uint16_t* W, int64_t ldw,
                                                  float* C, int64_t ldc, int M, int N, int K, int dtype,
                                                  detgemm_stream_t stream);

/*
 * detgemm_w8a8 on operands already widened to fp16 by detgemm_widen_i8_f16: the same
 * definition ([P4] §II), the same result bits. A16 [M x K] (lda) and W16 [N x K] (ldw)
 * must hold integers in [-128, 127] — exactness rests on it; other values give
 * unspecified results (never a fault). lda, ldw and ldc are multiples of 8 elements.
 * Scratch: detgemm_w8a8_f16ops_workspace_size (only split-K needs any; 256-byte aligned).
 * Errors as detgemm_w8a8.
 */
DETGEMM_API detgemm_status detgemm_w8a8_f16ops(const uint16_t* A16, int64_t lda, const uint16_t* W16, int64_t ldw,
                                               const int32_t* ea, const int32_t* ew, uint16_t* C, int64_t ldc,
                                               int M, int N, int K, int split_k, void* ws, size_t ws_bytes,
                                               detgemm_stream_t stream);

DETGEMM_API size_t detgemm_w8a8_f16ops_workspace_size(int M, int N, int K, int split_k);

/*
 * detgemm_w8a8 on operands in HOST memory [P4 §II: a row's int32 accumulator, and so
 * its bf16 result, does not depend on which rows are computed with it]: the rows of A
 * are cut into chunks, and each chunk's host-to-device copy, its computation (the same
 * exact path as detgemm_w8a8) and the copy of its result back to host memory overlap
 * with those of its neighbours. The result bits are those of detgemm_w8a8.
 *   A int8 [M x K] (lda), W int8 [N x K] (ldw), ea int32 [M], ew int32 [N],
 *   C bf16 bit patterns [M x N] (ldc): all HOST pointers, no alignment rule; page-locked
 *   (pinned) memory lets the copies run asynchronously and overlap (pageable memory
 *   works, without the overlap).
 *   buf  DEVICE scratch of buf_bytes >= detgemm_w8a8_host_buffer_size(M, N, K),
 *        256-byte aligned; it holds the weight, its fp16 copy and two chunks.
 * Asynchronous on `stream`: C is complete when the stream has been synchronized. The
 * library creates two copy streams and a few events once per device (no device memory).
 * Errors: INVALID_ARG, PRECONDITION (K > DETGEMM_MAX_K), WORKSPACE, ALIGNMENT (buf),
 *         UNSUPPORTED_DEVICE, CUDA.
 */
DETGEMM_API detgemm_status detgemm_w8a8_host(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw,
                                             const int32_t* ea, const int32_t* ew, uint16_t* C, int64_t ldc,
                                             int M, int N, int K, void* buf, size_t buf_bytes,
                                             detgemm_stream_t stream);

DETGEMM_API size_t detgemm_w8a8_host_buffer_size(int M, int N, int K);

/*
 * Self-check of the failure detection: launches a one-thread kernel whose bounded wait
 * on a barrier that nothing ever arrives on expires after limit_ms (1 .. 2000). After it,
 * detgemm_get_device_status returns DETGEMM_ERR_TIMEOUT and the CUDA context stays usable.
 * Every wait of the GEMM engine uses the same bounded mechanism (limit 4 s).
 */
DETGEMM_API detgemm_status detgemm_selftest_timeout(int limit_ms, detgemm_stream_t stream);

/*
 * Synchronizes `stream`, then returns and clears the current device's status word:
 * DETGEMM_OK, DETGEMM_ERR_NONFINITE, DETGEMM_ERR_TIMEOUT or DETGEMM_ERR_RANGE (the first one raised
 * since the last read), or DETGEMM_ERR_CUDA if the synchronization itself failed.
 */
DETGEMM_API detgemm_status detgemm_get_device_status(detgemm_stream_t stream);

/*
 * detgemm_w8a8 without a caller-supplied workspace. The source pages have no
 * counterpart to this call; it exists for callers that cannot allocate device memory
 * when they run the GEMM — for example a plugin inside an inference server that is
 * handed only its input and output tensors, or a latency-critical serving loop that
 * bans cudaMalloc because an allocation can synchronize the device.
 *
 * Same operands, layout and result bits as detgemm_w8a8. The split-K scratch lives in a
 * fixed device array of DETGEMM_NOALLOC_SCRATCH_BYTES inside the library, which every GPU
 * that loads the library keeps until the process exits. The call is refused with
 * DETGEMM_ERR_WORKSPACE, before anything is launched, when the scratch it really uses,
 * detgemm_w8a8_noalloc_scratch_size(M, N, K, split_k), exceeds that size:
 *  - M <= 64: the decode kernels' accumulator and fp16 copy of A, M * N * 4 + M * K * 2
 *    bytes (rounded up), at any split_k, as detgemm_w8a8 needs them;
 *  - M > 64: M * N * 4 bytes plus a counter per tile when split_k > 1, else nothing.
 * Problems of more than 64 rows run here on the int8 warp-MMA tile kernel (mma.sync
 * m16n8k32, exact int32 accumulation, about 147 TOPS on GB300), not on the tcgen05 engine
 * of detgemm_w8a8, whose fp16 operand copies would need tens of MB of scratch: the bits
 * are the same, the throughput at large M is an order of magnitude lower.
 * Errors are those of detgemm_w8a8, checked in the same order, except that the scratch
 * size is checked last (after the device check) instead of detgemm_w8a8's workspace check.
 *  - The first call on each device looks up the array's device address (set-up done
 *    once per device, with that device current); make that first call before any
 *    stream capture begins.
 *  - All calls share the one array and each clears the part it uses: calls that may
 *    overlap on the GPU (different streams, or different host threads) race and must
 *    be serialized by the caller.
 *  - The call allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
#define DETGEMM_NOALLOC_SCRATCH_BYTES (8u << 20)

/* Bytes of the fixed scratch array detgemm_w8a8_noalloc uses for this problem (0 for
 * M > 64 at split_k == 1; 0 for empty or invalid sizes). */
DETGEMM_API size_t detgemm_w8a8_noalloc_scratch_size(int M, int N, int K, int split_k);

DETGEMM_API detgemm_status detgemm_w8a8_noalloc(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw,
                                                const int32_t* ea, const int32_t* ew, uint16_t* C,
                                                int64_t ldc, int M, int N, int K, int split_k,
                                                detgemm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DETGEMM_H */
