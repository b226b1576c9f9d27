/*
 * detgemm conformance instrument: epilogue fault injection. A debug entry point for
 * measuring what a conformance check can see; no product call reaches it.
 *
 * Source: "Deterministic LLM Inference Across GPU Kernels: Power-of-Two INT8 Quantization
 * Scales and the Limits of Tolerance-Based Conformance", §III "Nine Faults" (injected fault
 * families, three severities, checkpoint-native or power-of-two scales) and §IV "How much can
 * a tolerance see?" (epilogue faults move an output by at most one bfloat16 spacing; under
 * power-of-two scales the precision and order faults change nothing and only an equality
 * check sees a wrong rounding mode). The pages name the faults without defining them; the
 * readings implemented here are:
 *   F1 scale precision       s = fp32(s_a * s_w); out = rne_bf16(fp32(fp32(acc) * s))
 *   F2 double rounding       out = rne_bf16(rne_fp32(acc * s_a * s_w))
 *   F3 multiplication order  out = rne_bf16(fp32(fp32(fp32(acc) * s_a) * s_w))
 *   F4 output truncation     out = the exact acc * s_a * s_w rounded toward zero
 *   none (the null fault F8) out = the exact acc * s_a * s_w rounded once, nearest-even
 * fp32(.) is one IEEE rounding to nearest-even; F2 scales its fp32 rounding by 2^X, so it
 * equals one rounding to fp32 wherever that result is a normal fp32 number.
 */
#ifndef DETGEMM_CONFORMANCE_H
#define DETGEMM_CONFORMANCE_H

#include "detgemm.h"

#ifdef __cplusplus
extern "C" {
#endif

enum {
    DETGEMM_FAULT_NONE = 0,
    DETGEMM_FAULT_F1_SCALE_PRECISION = 1,
    DETGEMM_FAULT_F2_DOUBLE_ROUNDING = 2,
    DETGEMM_FAULT_F3_ORDER = 3,
    DETGEMM_FAULT_F4_TRUNCATION = 4
};
/* which outputs carry the fault: one element (picked from seed), about one percent (a hash of
 * the element index and seed below 1/100), or every element; the others get the correct one */
enum { DETGEMM_SEVERITY_ONE = 0, DETGEMM_SEVERITY_ONE_PERCENT = 1, DETGEMM_SEVERITY_ALL = 2 };
/* the scales: per-row and per-column powers of two given by int32 exponents (the library's
 * W8A8 scales), or arbitrary finite fp32 values (a checkpoint's own scales) */
enum { DETGEMM_SCALES_POW2 = 0, DETGEMM_SCALES_F32 = 1 };

/*
 * The W8A8 epilogue, or one injected fault, applied to exact int32 accumulators:
 *   acc  int32 [M x N], row stride ldacc (e.g. from detgemm_gemm_s8_i32), device memory
 *   sa   [M] and sw [N]: int32 exponents (DETGEMM_SCALES_POW2) or fp32 scales (_F32), device
 *   C    bf16 bit patterns [M x N], row stride ldc, device memory
 * With DETGEMM_FAULT_NONE and power-of-two scales the output is bit-identical to detgemm_w8a8
 * on the same operands. An exact zero gives +0. Asynchronous on stream.
 * Errors: INVALID_ARG (enums, sizes, null pointers, ld < N), ALIGNMENT (4-byte acc, sa, sw;
 * 2-byte C), UNSUPPORTED_DEVICE, CUDA.
 */
DETGEMM_API detgemm_status detgemm_epilogue_inject(const int32_t* acc, int64_t ldacc, int scales, const void* sa,
                                                   const void* sw, int fault, int severity, uint32_t seed,
                                                   uint16_t* C, int64_t ldc, int M, int N, detgemm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DETGEMM_CONFORMANCE_H */
