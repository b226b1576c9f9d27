// Gated-linear-unit epilogue: rne_bf16(SiLU(g) * u) of exact scaled accumulators, rounded
// once. The W8A8 epilogue rounds the exactly scaled int32 accumulator once ("Deterministic
// LLM Inference Across GPU Kernels ...", §II "Pipeline and alibi"); an FFN applies the gate
// SiLU(g) = g / (1 + e^-g) to the gate GEMM's output and multiplies by the up GEMM's before
// that rounding. With g = gacc * 2^Eg and u = uacc * 2^Eu exact, y = g * u / (1 + e^-g) is a
// real number (transcendental unless 0), and its one correct rounding to bf16 is found by
// evaluations of increasing precision, each with a proven bound on its relative error; an
// evaluation decides when no bf16 rounding boundary (a midpoint between neighbours) lies
// within its bound of the computed value:
//   exact zero   gacc == 0 or uacc == 0: +0;
//   g >= 64      e^-g < 2^-92 while the exact dyadic P = g * u (62 significant bits) is either
//                on a midpoint or at least 2^-62 |P| from every one: y = P sigma(g) rounds as
//                P does, except that a P on a midpoint rounds toward zero (|y| < |P|);
//   g <= -700    |y| < 2^-800: a zero with the sign of g * u;
//   fp32         g > -80: expf (at most 2 ulp) on fp32 g and u; relative error below
//                (12 + |g|) 2^-24, i.e. (12 + |g|) units of the last place of the fp32 result,
//                which decides unless its low 16 bits are that close to 0x8000 (the midpoint);
//   fp64         exp (at most 2 ulp) on the exact g and u: relative error below 2^-49;
//   double-double e^-g by range reduction with a double-double ln 2 and a Taylor series, and
//                y = P / (1 + e^-g), in double-double arithmetic (the error-free sums and
//                products of Dekker and Knuth): relative error below 2^-90.
// What even the last evaluation cannot decide (an output within 2^-90 of a midpoint, far
// rarer than one in 2^60 outputs) raises DEV_RANGE and returns its nearest-even rounding.
// The exponents must lie in [-60, 40] (g and u within 2^71; outputs of a scaled int8 layer
// sit far inside): otherwise DEV_RANGE is raised and the output is a NaN.
#pragma once

#include "common.cuh"

namespace detgemm {

// rne_bf16 (or, with ties_toward_zero, the rounding that resolves a tie toward zero) of the
// exact value S * 2^X, S != 0 an int64 (|S| < 2^63)
__device__ __forceinline__ uint16_t bf16_round_i64(long long S, int X, bool ties_toward_zero) {
    const uint16_t sign = S < 0 ? 0x8000 : 0;
    const unsigned long long a = S < 0 ? (unsigned long long)(-S) : (unsigned long long)S;
    const int b = 63 - __clzll((long long)a);
    int E = b + X;
    int sh;  // bits dropped
    int base;
    if (E >= -126) {
        sh = b - 7;
        base = (E + 127) << 7;
    } else {
        sh = -(X + 133);  // units of 2^-133
        base = 0;
    }
    unsigned long long q;
    bool up = false;
    if (sh <= 0) {
        q = sh <= -64 ? 0 : a << (-sh);
    } else if (sh >= 64) {
        q = 0;  // |value| < 2^-134 or so: rounds to zero
    } else {
        q = a >> sh;
        const unsigned long long rem = a & ((1ull << sh) - 1), half = 1ull << (sh - 1);
        up = rem > half || (rem == half && !ties_toward_zero && (q & 1));
    }
    q += up ? 1 : 0;
    int bits;
    if (E >= -126) {
        // q in [128, 256]; 256 carries into the next binade
        bits = base + (int)(q - 128);
        if (q == 256) bits = ((E + 1 + 127) << 7);
        if (bits >= 0x7F80) bits = 0x7F80;
    } else {
        bits = (int)q;  // 128 is the smallest normal, 0x0080
    }
    return sign | (uint16_t)bits;
}

// ---------------------------------------------------------------- double-double arithmetic
struct Dd {
    double hi, lo;
};
__device__ __forceinline__ Dd dd_two_sum(double a, double b) {
    const double s = __dadd_rn(a, b);
    const double bb = __dsub_rn(s, a);
    const double e = __dadd_rn(__dsub_rn(a, __dsub_rn(s, bb)), __dsub_rn(b, bb));
    return {s, e};
}
__device__ __forceinline__ Dd dd_fast_two_sum(double a, double b) {  // |a| >= |b| or a == 0
    const double s = __dadd_rn(a, b);
    return {s, __dsub_rn(b, __dsub_rn(s, a))};
}
__device__ __forceinline__ Dd dd_two_prod(double a, double b) {
    const double p = __dmul_rn(a, b);
    return {p, __fma_rn(a, b, -p)};
}
__device__ __forceinline__ Dd dd_add(Dd a, Dd b) {
    Dd s = dd_two_sum(a.hi, b.hi);
    const Dd t = dd_two_sum(a.lo, b.lo);
    s.lo = __dadd_rn(s.lo, t.hi);
    s = dd_fast_two_sum(s.hi, s.lo);
    s.lo = __dadd_rn(s.lo, t.lo);
    return dd_fast_two_sum(s.hi, s.lo);
}
__device__ __forceinline__ Dd dd_neg(Dd a) { return {-a.hi, -a.lo}; }
__device__ __forceinline__ Dd dd_mul(Dd a, Dd b) {
    Dd p = dd_two_prod(a.hi, b.hi);
    p.lo = __dadd_rn(p.lo, __dadd_rn(__dmul_rn(a.hi, b.lo), __dmul_rn(a.lo, b.hi)));
    return dd_fast_two_sum(p.hi, p.lo);
}
__device__ __forceinline__ Dd dd_mul_d(Dd a, double b) {
    Dd p = dd_two_prod(a.hi, b);
    p.lo = __fma_rn(a.lo, b, p.lo);
    return dd_fast_two_sum(p.hi, p.lo);
}
// a / b by long division: three quotient digits, each remainder formed exactly enough
__device__ __forceinline__ Dd dd_div(Dd a, Dd b) {
    const double q1 = __ddiv_rn(a.hi, b.hi);
    Dd r = dd_add(a, dd_neg(dd_mul_d(b, q1)));
    const double q2 = __ddiv_rn(r.hi, b.hi);
    r = dd_add(r, dd_neg(dd_mul_d(b, q2)));
    const double q3 = __ddiv_rn(r.hi, b.hi);
    return dd_add(dd_fast_two_sum(q1, q2), Dd{q3, 0.0});
}
__device__ __forceinline__ Dd dd_div_d(Dd a, double b) { return dd_div(a, Dd{b, 0.0}); }

// e^x for |x| < 709 in double-double: x = k ln 2 + r with |r| <= ln(2) / 2 + tiny (ln 2 as a
// double-double, error below 2^-106, so r is off by at most ~2^-96 for |k| <= 1024), then the
// Taylor series of e^r to degree 24 (remainder below 2^-110 for |r| < 0.35) by Horner's rule,
// then the exact scaling by 2^k
__device__ __forceinline__ Dd dd_exp(double x) {
    const double LN2_HI = 6.93147180559945286227e-01;  // ln 2 rounded to double
    const double LN2_LO = 2.31904681384629955842e-17;  // ln 2 - LN2_HI rounded to double
    const double k = rint(x * 1.44269504088896338700e+00);
    Dd r = dd_add(Dd{x, 0.0}, dd_neg(dd_two_prod(k, LN2_HI)));
    r = dd_add(r, dd_neg(dd_two_prod(k, LN2_LO)));
    Dd p = {1.0, 0.0};
    for (int n = 24; n >= 1; --n) p = dd_add(Dd{1.0, 0.0}, dd_mul(dd_div_d(r, (double)n), p));
    const int ki = (int)k;
    return {scalbn(p.hi, ki), scalbn(p.lo, ki)};
}

// The bf16 rounding of a nonzero double-double value v = hi + lo known to relative error
// eps: returns true with the bits when no midpoint lies within eps |v| of v.
__device__ __forceinline__ bool bf16_decide(double hi, double lo, double eps, uint16_t& out) {
    const uint16_t sign = hi < 0 ? 0x8000 : 0;
    if (hi < 0) {
        hi = -hi;
        lo = -lo;
    }
    int lead = ilogb(hi);
    if (hi == scalbn(1.0, lead) && lo < 0) --lead;  // the value lies just below a power of two
    if (lead > 127) {
        out = sign | 0x7F80;
        return true;
    }
    const int sc = lead >= -126 ? 7 - lead : 133;
    const int base = lead >= -126 ? ((lead + 127) << 7) - 128 : 0;
    const double mh = scalbn(hi, sc), ml = scalbn(lo, sc);  // the value in units of the spacing
    double fl = floor(mh);
    if (fl == mh && ml < 0) fl -= 1.0;
    const double d = __dadd_rn(__dsub_rn(__dsub_rn(mh, fl), 0.5), ml);  // fraction - 1/2
    if (fabs(d) <= eps * mh) return false;
    int bits = base + (int)fl + (d > 0 ? 1 : 0);
    if (bits > 0x7F80) bits = 0x7F80;
    out = sign | (uint16_t)bits;
    return true;
}

// rne_bf16(SiLU(gacc 2^Eg) * uacc 2^Eu); `bad` is set on an exponent outside [-60, 40] or
// an output no evaluation could decide
static __device__ __noinline__ uint16_t bf16_silu_mul(int32_t gacc, int32_t uacc, long long Eg, long long Eu, bool& bad) {
    if (gacc == 0 || uacc == 0) return 0x0000;
    if (Eg < -60 || Eg > 40 || Eu < -60 || Eu > 40) {
        bad = true;
        return 0x7FC0;
    }
    const double g = scalbn((double)gacc, (int)Eg), u = scalbn((double)uacc, (int)Eu);  // exact
    const bool neg = (gacc < 0) != (uacc < 0);
    if (g >= 64.0) return bf16_round_i64((long long)gacc * (long long)uacc, (int)(Eg + Eu), true);
    if (g <= -700.0) return neg ? 0x8000 : 0x0000;
    if (g > -80.0) {
        const float g32 = __fmul_rn(__int2float_rn(gacc), scalbnf(1.0f, (int)Eg));
        const float u32 = __fmul_rn(__int2float_rn(uacc), scalbnf(1.0f, (int)Eu));
        const float y = __fdiv_rn(__fmul_rn(g32, u32), __fadd_rn(1.0f, expf(-g32)));
        const float ay = fabsf(y);
        if (ay >= 0x1p-125f && ay < 0x1p127f) {
            const int low = (int)(__float_as_uint(y) & 0xFFFFu);
            const int tol = 14 + (int)fabsf(g32);
            if (abs(low - 0x8000) > tol) return __bfloat16_as_ushort(__float2bfloat16_rn(y));
        }
    }
    uint16_t out;
    {
        const double y = __ddiv_rn(__dmul_rn(g, u), __dadd_rn(1.0, exp(-g)));
        if (y != 0.0 && bf16_decide(y, 0.0, 0x1p-49, out)) return out;
    }
    const Dd P = dd_two_prod(g, u);  // exact
    const Dd y = dd_div(P, dd_add(Dd{1.0, 0.0}, dd_exp(-g)));
    if (bf16_decide(y.hi, y.lo, 0x1p-90, out)) return out;
    bad = true;
    return __bfloat16_as_ushort(__float2bfloat16_rn((float)y.hi));
}

}  // namespace detgemm
