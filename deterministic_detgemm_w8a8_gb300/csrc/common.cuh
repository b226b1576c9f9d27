// Shared device helpers of libdetgemm: status word, exact epilogues, bit utilities.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/detgemm.h"

namespace detgemm {

// Device status bits (first error wins in the host-visible translation).
enum : uint32_t { DEV_NONFINITE = 1u, DEV_TIMEOUT = 2u, DEV_RANGE = 4u };

// Device status word. Every translation unit that raises a device-side condition owns
// one (internal linkage, so no relocatable device code is needed) and exports a host
// accessor built with DETGEMM_STATUS_ACCESSOR; the C ABI ORs them together.
static __device__ uint32_t g_device_status = 0;

__device__ __forceinline__ void raise_status(uint32_t bit) { atomicOr(&g_device_status, bit); }

// Defines `cudaError_t fn(uint32_t* bits)`: reads and clears this unit's status word on
// the current device (synchronous; the caller has synchronized the stream).
#define DETGEMM_STATUS_ACCESSOR(fn)                                                      \
    cudaError_t fn(uint32_t* bits) {                                                     \
        uint32_t zero = 0;                                                               \
        cudaError_t e = cudaMemcpyFromSymbol(bits, g_device_status, sizeof(uint32_t));   \
        if (e == cudaSuccess && *bits != 0)                                              \
            e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(uint32_t));            \
        return e;                                                                        \
    }

// ------------------------------------------------------------------------------------
// Epilogue E1 — "Deterministic LLM Inference Across GPU Kernels: Power-of-Two INT8
// Quantization Scales ...", §II "Pipeline and alibi": the int32 accumulator is scaled
// by the power of two 2^(ea + ew) and rounded once to bfloat16.
//
// Integer-only construction of rne_bf16(acc * 2^E): no floating-point operation takes
// part, so no intermediate rounding can occur. bf16 keeps 8 significant bits; normal
// numbers carry the biased exponent eb = msb + E + 127, subnormals count units of
// 2^-133. In both cases the result is base + q, where q is |acc| shifted right by sh
// and rounded half-to-even; a carry out of q moves into the exponent field on its own,
// and anything at or above 0x7F80 is infinity.
// ------------------------------------------------------------------------------------
// General case (any exponent): subnormal results and overflow handled explicitly.
static __device__ __noinline__ uint16_t bf16_from_acc_pow2_general(int32_t acc, int E) {
    uint32_t sign = acc < 0 ? 0x8000u : 0u;
    uint32_t m = acc < 0 ? (uint32_t)(-(long long)acc) : (uint32_t)acc;
    int p = 31 - __clz(m);      // m in [2^p, 2^(p+1))
    int eb = p + E + 127;       // biased exponent of a normal result
    int sh;
    uint32_t base;
    if (eb >= 1) {
        sh = p - 7;
        base = (uint32_t)(eb - 1) << 7;
    } else {
        sh = -(E + 133);
        base = 0;
    }
    uint32_t q;
    if (sh <= 0) {
        q = m << (-sh);  // exact (at most 8 significant bits result)
    } else if (sh > 40) {
        q = 0;           // |value| < 2^-31 units: rounds to zero
    } else {
        unsigned long long mm = m;
        unsigned long long qq = mm >> sh;
        unsigned long long rem = mm - (qq << sh);
        unsigned long long half = 1ull << (sh - 1);
        if (rem > half || (rem == half && (qq & 1ull))) qq += 1;
        q = (uint32_t)qq;
    }
    uint32_t bits = base + q;
    if (bits >= 0x7F80u) bits = 0x7F80u;
    return (uint16_t)(sign | bits);
}

// Fast path for results in the normal bf16 range: normalise |acc| so its leading one
// sits at bit 31, keep the top 8 bits and round half-to-even on the 24 dropped bits;
// the carry of a round-up moves into the exponent field by itself.
__device__ __forceinline__ uint16_t bf16_from_acc_pow2(int32_t acc, int32_t ea, int32_t ew) {
    if (acc == 0) return 0;
    long long El = (long long)ea + (long long)ew;
    int E = (int)(El > 300 ? 300 : (El < -300 ? -300 : El));
    const uint32_t sign = (uint32_t)acc >> 31 << 15;
    const uint32_t m = acc < 0 ? 0u - (uint32_t)acc : (uint32_t)acc;  // |INT_MIN| = 2^31 fits
    const int lz = __clz(m);
    const int eb = 31 - lz + E + 127;
    if (eb < 1 || eb > 254) return bf16_from_acc_pow2_general(acc, E);
    const uint32_t n = m << lz;
    uint32_t q = n >> 24;  // 1.xxxxxxx
    const uint32_t rem = n & 0xFFFFFFu;
    q += (rem > 0x800000u) | ((rem == 0x800000u) & q);
    uint32_t bits = ((uint32_t)(eb - 1) << 7) + q;
    bits = bits >= 0x7F80u ? 0x7F80u : bits;
    return (uint16_t)(sign | bits);
}

// ------------------------------------------------------------------------------------
// Epilogue E1 with a bias: rne_bf16(acc * 2^E + b), b a bfloat16 per output column,
// rounded once. The pages define the epilogue as the one rounding of the exactly scaled
// int32 accumulator ("Deterministic LLM Inference Across GPU Kernels ...", §II "Pipeline
// and alibi"); the bias joins the exact value before that rounding, so the result is
// still a function of the operands alone.
//
// Both terms are integers times powers of two: x = acc * 2^E and b = mb * 2^eb (mb < 2^8).
// They are aligned on the smaller exponent in an int64 and the sum is rounded once. When
// one term lies entirely below 2^-9 of the other's last unit, only its sign can matter (it
// decides a tie or a value sitting on the bf16 grid, nothing else), so it is replaced by
// one signed unit below that last unit, which keeps the int64 in range.
// ------------------------------------------------------------------------------------
// rne_bf16(S * 2^X) for an int64 S != 0 (|S| <= 2^63).
static __device__ __noinline__ uint16_t bf16_from_i64_pow2(long long S, int X) {
    const uint32_t sign = S < 0 ? 0x8000u : 0u;
    const unsigned long long m = S < 0 ? 0ull - (unsigned long long)S : (unsigned long long)S;
    const int p = 63 - __clzll(m);  // m in [2^p, 2^(p+1))
    const int eb = p + X + 127;
    int sh;
    uint32_t base;
    if (eb >= 1) {
        sh = p - 7;
        base = (uint32_t)(eb - 1) << 7;
    } else {
        sh = -(X + 133);
        base = 0;
    }
    unsigned long long q;
    if (sh <= 0) {
        q = m << (-sh);  // at most 8 significant bits
    } else if (sh > 63) {
        q = 0;           // below half of the smallest subnormal (or exactly half: even)
    } else {
        q = m >> sh;
        const unsigned long long rem = m - (q << sh);
        const unsigned long long half = 1ull << (sh - 1);
        if (rem > half || (rem == half && (q & 1ull))) q += 1;
    }
    unsigned long long bits = base + q;
    if (bits >= 0x7F80ull) bits = 0x7F80ull;
    return (uint16_t)(sign | (uint32_t)bits);
}

// General case: any accumulator, any exponents, any bias (a non-finite bias passes
// through; an exact zero sum gives +0).
static __device__ __noinline__ uint16_t bf16_from_acc_pow2_bias_general(int32_t acc, int32_t ea, int32_t ew,
                                                                        uint16_t b) {
    if ((b & 0x7FFFu) == 0) return bf16_from_acc_pow2(acc, ea, ew);  // x + (+-0) = x
    if ((b & 0x7F80u) == 0x7F80u) return b;                           // +-inf, NaN
    if (acc == 0) return b;                                           // b is on the grid
    long long El = (long long)ea + (long long)ew;
    const int E = (int)(El > 300 ? 300 : (El < -300 ? -300 : El));
    const int field = (b >> 7) & 0xFF;
    const int mbu = field == 0 ? (b & 0x7F) : ((b & 0x7F) | 0x80);
    const int eb = field == 0 ? -133 : field - 134;
    const long long mb = (b & 0x8000u) ? -(long long)mbu : (long long)mbu;
    long long S;
    int X;
    if (E >= eb) {
        if (E - eb > 31) {  // |b| < 2^(E - 23): a signed unit at 2^(E - 31)
            S = ((long long)acc << 31) + (mb > 0 ? 1 : -1);
            X = E - 31;
        } else {
            S = ((long long)acc << (E - eb)) + mb;
            X = eb;
        }
    } else {
        if (eb - E > 40) {  // |x| < 2^(eb - 9): a signed unit at 2^(eb - 40)
            S = (mb << 40) + (acc > 0 ? 1 : -1);
            X = eb - 40;
        } else {
            S = (mb << (eb - E)) + (long long)acc;
            X = E;
        }
    }
    if (S == 0) return 0;
    return bf16_from_i64_pow2(S, X);
}

// Fast form: sc = 2^(ea + ew) as an fp32 number with ea + ew in [-120, 80], |acc| < 2^24
// and |b| < 2^64. Then x = acc * sc is an exact fp32 number and the sum x + b is rounded
// both down and up: equal results mean the sum is exact (an exact zero comes out as +0 from
// the upward rounding); otherwise the one toward zero with its last bit set is the sum
// rounded to odd at 24 bits. Rounding to odd at 24 >= 8 + 2 bits and then to nearest-even at
// 8 bits equals one rounding to nearest, so the result is that of the general form. (A sum
// in the fp32 subnormal range is a multiple of 2^-133, hence exact.)
__device__ __forceinline__ uint16_t bf16_from_scaled_bias_ro(int32_t acc, float sc, uint32_t b) {
    const float x = __fmul_rn(__int2float_rn(acc), sc);
    const float bv = __uint_as_float(b << 16);
    const float lo = __fadd_rd(x, bv);
    const float hi = __fadd_ru(x, bv);
    const uint32_t r = lo == hi ? __float_as_uint(hi) : (__float_as_uint(lo >= 0.0f ? lo : hi) | 1u);
    const __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(r));
    return *reinterpret_cast<const uint16_t*>(&h);
}

// The fast form's scale for one output: 2^(ea + ew) when ea and ew lie in [-60, 40] and the
// bias is below 2^64 in magnitude, else 0 (the general form).
__device__ __forceinline__ float bias_fast_scale(int32_t ea, int32_t ew, uint32_t b) {
    const bool ok = ea >= -60 && ea <= 40 && ew >= -60 && ew <= 40 && ((b >> 7) & 0xFFu) < 191u;
    return ok ? __uint_as_float((uint32_t)(ea + ew + 127) << 23) : 0.0f;
}

// rne_bf16(acc * 2^(ea + ew) + b): the fast form where it applies, else the general one.
__device__ __forceinline__ uint16_t bf16_from_acc_pow2_bias(int32_t acc, int32_t ea, int32_t ew, uint32_t b) {
    const float sc = bias_fast_scale(ea, ew, b);
    const uint32_t ua = acc < 0 ? 0u - (uint32_t)acc : (uint32_t)acc;
    if (sc != 0.0f && ua < (1u << 24)) return bf16_from_scaled_bias_ro(acc, sc, b);
    return bf16_from_acc_pow2_bias_general(acc, ea, ew, (uint16_t)b);
}

// Exact power of two as a double for |k| <= 1022.
__device__ __forceinline__ double pow2_f64(int k) {
    return __longlong_as_double((long long)(k + 1023) << 52);
}

// |x| of an fp32 bit pattern normalised to x = M * 2^(p - 23), M in [2^23, 2^24).
// Returns false for zero. Subnormals are normalised.
__device__ __forceinline__ bool f32_normalise(uint32_t absbits, uint32_t& M, int& p) {
    uint32_t ef = absbits >> 23;
    uint32_t fr = absbits & 0x7FFFFFu;
    if (ef == 0) {
        if (fr == 0) return false;
        int b = 31 - __clz(fr);          // msb of the subnormal fraction
        M = fr << (23 - b);
        p = b - 149;
        return true;
    }
    M = fr | 0x800000u;
    p = (int)ef - 127;
    return true;
}

// Eight consecutive small integers (int8 range), packed for one store: as int8 (8 bytes)
// or as exact fp16 values (16 bytes; d + 1152 is placed under the fp16 exponent of 1024
// and 1152 is subtracted, both exact).
template <typename T>
struct Pack8;
template <>
struct Pack8<int8_t> {
    typedef uint2 type;
    static __device__ __forceinline__ int8_t one(int8_t d) { return d; }
    static __device__ __forceinline__ uint2 make(const int8_t (&d)[8]) {
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo |= (uint32_t)(uint8_t)d[i] << (8 * i);
            hi |= (uint32_t)(uint8_t)d[i + 4] << (8 * i);
        }
        return make_uint2(lo, hi);
    }
};
template <>
struct Pack8<__half> {
    typedef uint4 type;
    static __device__ __forceinline__ __half one(int8_t d) { return __short_as_half((short)(two(d, 0) & 0xFFFFu)); }
    static __device__ __forceinline__ uint32_t two(int8_t a, int8_t b) {
        const uint32_t w = (0x6400u | (uint32_t)(a + 128)) | ((0x6400u | (uint32_t)(b + 128)) << 16);
        const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
        const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&w), bias);
        return *reinterpret_cast<const uint32_t*>(&r);
    }
    static __device__ __forceinline__ uint4 make(const int8_t (&d)[8]) {
        return make_uint4(two(d[0], d[1]), two(d[2], d[3]), two(d[4], d[5]), two(d[6], d[7]));
    }
};

}  // namespace detgemm
