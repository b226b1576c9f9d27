// Epilogue fault injection for the conformance instrument ("Deterministic LLM Inference
// Across GPU Kernels: Power-of-Two INT8 Quantization Scales ...", §III "Nine Faults" and §IV
// "How much can a tolerance see?"). The pages inject faults into the epilogue of a W8A8
// kernel (the step that applies s_a s_w to the exact int32 accumulator and rounds to
// bfloat16) and ask which conformance checks see them. They name the faults but print no
// definition; this file implements written readings of four of them, applied on the GPU to
// exact accumulators produced by the library's own GEMM (detgemm_gemm_s8_i32):
//   F1 scale precision      s = fp32(s_a * s_w), then fp32(fp32(acc) * s), then bf16 RNE
//   F2 double rounding      the exact value rounded to fp32, then to bf16 (RNE both times)
//   F3 multiplication order fp32(fp32(fp32(acc) * s_a) * s_w), then bf16 RNE
//   F4 output truncation    the exact value rounded toward zero instead of to nearest even
// and the correct epilogue (the null fault F8): the exact value acc * s_a * s_w rounded once
// to bfloat16, nearest-even. Scales are either powers of two (int32 exponents, the product's
// E1, bit-identical to detgemm_w8a8) or arbitrary finite fp32 values (a checkpoint's own
// scales; the exact product acc * s_a * s_w of up to 79 bits is formed in 128-bit integer
// arithmetic and rounded once). No product call reaches this code.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/detgemm.h"
#include "../../include/detgemm_conformance.h"
#include "common.cuh"
#include "internal.h"

namespace detgemm {
namespace {

struct InjArgs {
    const int32_t* acc;
    int64_t ldacc;
    int scales;  // DETGEMM_SCALES_POW2 or DETGEMM_SCALES_F32
    const void* sa;
    const void* sw;
    int fault, severity;
    uint32_t seed;
    uint16_t* C;
    int64_t ldc;
    int M, N;
};

// 32-bit integer mixer (xorshift-multiply rounds) used to pick the faulted outputs
__device__ __forceinline__ uint32_t mix32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

// an fp32 value as sign, integer significand and exponent: |x| = m * 2^e
__device__ __forceinline__ void split_f32(float x, uint32_t& neg, uint64_t& m, int& e) {
    const uint32_t b = __float_as_uint(x);
    neg = b >> 31;
    const uint32_t be = (b >> 23) & 0xFFu;
    m = (b & 0x7FFFFFu) | (be ? 0x800000u : 0u);
    e = (be ? (int)be : 1) - 150;
}

// The exact value acc * s_a * s_w as S * 2^X with a signed int64 S of at most 62 significant
// bits: the product of the significands (up to 79 bits) is shifted right as far as needed
// and any dropped bit is kept as a set last bit (rounding to odd at >= 62 bits, which a later
// rounding to 8 or 24 bits cannot tell from the exact value). zero: the value is 0.
__device__ __forceinline__ void exact_value(int32_t acc, float sa, float sw, long long& S, int& X, bool& zero) {
    uint32_t na, nw;
    uint64_t ma, mw;
    int xa, xw;
    split_f32(sa, na, ma, xa);
    split_f32(sw, nw, mw, xw);
    const uint64_t u = acc < 0 ? (uint64_t)(-(int64_t)acc) : (uint64_t)acc;
    zero = u == 0 || ma == 0 || mw == 0;
    if (zero) {
        S = 0;
        X = 0;
        return;
    }
    const uint64_t t = u * ma;  // < 2^55
    const uint64_t lo = t * mw, hi = __umul64hi(t, mw);
    int sh = 0;
    uint64_t q = lo;
    if (hi != 0 || (lo >> 62) != 0) {
        const int msb = hi != 0 ? 127 - __clzll((long long)hi) : 63 - __clzll((long long)lo);
        sh = msb - 61;  // keep bits [sh, msb]: 62 bits
        q = sh >= 64 ? (hi >> (sh - 64)) : ((lo >> sh) | (hi << (64 - sh)));
        const bool dropped = sh >= 64 ? (lo != 0 || (hi & ((1ull << (sh - 64)) - 1)) != 0)
                                      : (lo & ((1ull << sh) - 1)) != 0;
        q |= dropped ? 1ull : 0ull;
    }
    const bool neg = ((acc < 0) ? 1u : 0u) ^ na ^ nw;
    S = neg ? -(long long)q : (long long)q;
    X = xa + xw + sh;
}

// bf16 bits of S * 2^X rounded toward zero (S != 0)
__device__ __forceinline__ uint16_t rz_bf16(long long S, int X) {
    const uint16_t sign = S < 0 ? 0x8000 : 0;
    const uint64_t a = S < 0 ? (uint64_t)(-S) : (uint64_t)S;
    const int b = 63 - __clzll((long long)a);  // a in [2^b, 2^(b+1))
    const int E = b + X;                       // value in [2^E, 2^(E+1))
    if (E > 127) return sign | 0x7F7F;         // beyond the largest finite: toward zero
    if (E >= -126) {
        const uint64_t top = b >= 7 ? a >> (b - 7) : a << (7 - b);  // 8 significant bits
        return sign | (uint16_t)(((uint32_t)(E + 127) << 7) | (uint32_t)(top & 0x7F));
    }
    // subnormal: units of 2^-133
    const int s = -(X + 133);
    const uint64_t q = s >= 64 ? 0 : (s >= 0 ? a >> s : a << (-s));
    return sign | (uint16_t)q;
}

__device__ __forceinline__ uint16_t bf16_rn_f32(float y) { return __bfloat16_as_ushort(__float2bfloat16_rn(y)); }

__global__ void epilogue_inject_kernel(const InjArgs p) {
    const int64_t total = (int64_t)p.M * p.N;
    const uint32_t pick_i = mix32(p.seed) % (uint32_t)p.M;
    const uint32_t pick_j = mix32(p.seed ^ 0x9E3779B9u) % (uint32_t)p.N;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(idx / p.N), j = (int)(idx - (int64_t)i * p.N);
        const int32_t acc = p.acc[(int64_t)i * p.ldacc + j];
        float sa, sw;
        int32_t ea = 0, ew = 0;
        if (p.scales == DETGEMM_SCALES_POW2) {
            ea = static_cast<const int32_t*>(p.sa)[i];
            ew = static_cast<const int32_t*>(p.sw)[j];
            sa = ldexpf(1.0f, ea);
            sw = ldexpf(1.0f, ew);
        } else {
            sa = static_cast<const float*>(p.sa)[i];
            sw = static_cast<const float*>(p.sw)[j];
        }
        bool sel;
        if (p.severity == DETGEMM_SEVERITY_ALL) sel = true;
        else if (p.severity == DETGEMM_SEVERITY_ONE_PERCENT) sel = mix32((uint32_t)idx ^ p.seed) % 100u == 0u;
        else sel = (uint32_t)i == pick_i && (uint32_t)j == pick_j;
        const int f = sel ? p.fault : DETGEMM_FAULT_NONE;
        uint16_t out;
        if (f == DETGEMM_FAULT_F1_SCALE_PRECISION) {
            out = bf16_rn_f32(__fmul_rn(__int2float_rn(acc), __fmul_rn(sa, sw)));
        } else if (f == DETGEMM_FAULT_F3_ORDER) {
            out = bf16_rn_f32(__fmul_rn(__fmul_rn(__int2float_rn(acc), sa), sw));
        } else if (p.scales == DETGEMM_SCALES_POW2 && f == DETGEMM_FAULT_NONE) {
            out = bf16_from_acc_pow2(acc, ea, ew);  // the product's E1, any exponents
        } else {
            long long S;
            int X;
            bool zero;
            if (p.scales == DETGEMM_SCALES_POW2) {
                // beyond +-2000 the value is 0 or infinite in bf16 either way
                const long long e = (long long)ea + ew;
                S = acc;
                X = (int)(e < -2000 ? -2000 : (e > 2000 ? 2000 : e));
                zero = acc == 0;
            } else {
                exact_value(acc, sa, sw, S, X, zero);
            }
            if (zero) {
                out = 0x0000;
            } else if (f == DETGEMM_FAULT_F2_DOUBLE_ROUNDING) {
                out = bf16_rn_f32(ldexpf(__ll2float_rn(S), X));
            } else if (f == DETGEMM_FAULT_F4_TRUNCATION) {
                out = rz_bf16(S, X);
            } else {
                out = bf16_from_i64_pow2(S, X);  // the correct one rounding
            }
        }
        p.C[(int64_t)i * p.ldc + j] = out;
    }
}

}  // namespace
}  // namespace detgemm

using namespace detgemm;

extern "C" DETGEMM_API detgemm_status detgemm_epilogue_inject(const int32_t* acc, int64_t ldacc, int scales,
                                                              const void* sa, const void* sw, int fault,
                                                              int severity, uint32_t seed, uint16_t* C,
                                                              int64_t ldc, int M, int N, detgemm_stream_t stream) {
    if (M < 0 || N < 0) return DETGEMM_ERR_INVALID_ARG;
    if (scales != DETGEMM_SCALES_POW2 && scales != DETGEMM_SCALES_F32) return DETGEMM_ERR_INVALID_ARG;
    if (fault < DETGEMM_FAULT_NONE || fault > DETGEMM_FAULT_F4_TRUNCATION) return DETGEMM_ERR_INVALID_ARG;
    if (severity < DETGEMM_SEVERITY_ONE || severity > DETGEMM_SEVERITY_ALL) return DETGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DETGEMM_OK;
    if (!acc || !sa || !sw || !C || ldacc < N || ldc < N) return DETGEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(acc) & 3u) || (reinterpret_cast<uintptr_t>(sa) & 3u) ||
        (reinterpret_cast<uintptr_t>(sw) & 3u) || (reinterpret_cast<uintptr_t>(C) & 1u))
        return DETGEMM_ERR_ALIGNMENT;
    if (!device_is_supported()) return DETGEMM_ERR_UNSUPPORTED_DEVICE;
    InjArgs a;
    a.acc = acc;
    a.ldacc = ldacc;
    a.scales = scales;
    a.sa = sa;
    a.sw = sw;
    a.fault = fault;
    a.severity = severity;
    a.seed = seed;
    a.C = C;
    a.ldc = ldc;
    a.M = M;
    a.N = N;
    const int64_t total = (int64_t)M * N;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    epilogue_inject_kernel<<<(unsigned)blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
    return cudaGetLastError() == cudaSuccess ? DETGEMM_OK : DETGEMM_ERR_CUDA;
}
