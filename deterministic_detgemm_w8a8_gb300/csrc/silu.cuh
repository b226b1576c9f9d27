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
//   fp32         -87 < g < 64 (by the fp32 value g32, within 2^-24 of g): one fp32
//                evaluation with relative error below 13 * 2^-24, i.e. 13 units of the last
//                place of the fp32 result (bf16_silu_mul_fast), which decides unless its low
//                16 bits are within 16 of 0x8000 (the midpoint) -- about one output in two
//                thousand, so that the slower evaluations below stay rare;
//   g >= 64      e^-g < 2^-92 while the exact dyadic P = g * u (62 significant bits) is either
//                on a midpoint or at least 2^-62 |P| from every one: y = P sigma(g) rounds as
//                P does, except that a P on a midpoint rounds toward zero (|y| < |P|);
//   g <= -700    |y| < 2^-800: a zero with the sign of g * u;
//   float-float  -80 < g < 64, |y| in [2^-100, 2^127): the same formula in fp32
//                float-float arithmetic (error-free sums and products), e^-g by range
//                reduction and a Taylor series: relative error below 2^-40;
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

// ---------------------------------------------------------------- float-float arithmetic
// The same error-free transformations in fp32 (a value is hi + lo, about 48 significant bits).
struct Ff {
    float hi, lo;
};
__device__ __forceinline__ Ff ff_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ Ff ff_fast_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ Ff ff_add(Ff a, Ff b) {
    Ff s = ff_two_sum(a.hi, b.hi);
    const Ff t = ff_two_sum(a.lo, b.lo);
    s.lo = __fadd_rn(s.lo, t.hi);
    s = ff_fast_two_sum(s.hi, s.lo);
    s.lo = __fadd_rn(s.lo, t.lo);
    return ff_fast_two_sum(s.hi, s.lo);
}
__device__ __forceinline__ Ff ff_mul(Ff a, Ff b) {
    const float p = __fmul_rn(a.hi, b.hi);
    float e = __fmaf_rn(a.hi, b.hi, -p);
    e = __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, e));
    return ff_fast_two_sum(p, e);
}
__device__ __forceinline__ Ff ff_div(Ff a, Ff b) {
    const float q1 = __fdiv_rn(a.hi, b.hi);
    const Ff r = ff_add(a, ff_mul(b, Ff{-q1, 0.0f}));
    const float q2 = __fdiv_rn(r.hi, b.hi);
    const Ff r2 = ff_add(r, ff_mul(b, Ff{-q2, 0.0f}));
    const float q3 = __fdiv_rn(r2.hi, b.hi);
    return ff_add(ff_fast_two_sum(q1, q2), Ff{q3, 0.0f});
}

// e^x for x = xh + xl, |x| < 81, in float-float: x = k ln 2 + r with ln 2 in three floats (the
// first with 16 significant bits, so that k * LN2_A is exact for |k| < 128), the Taylor series
// of e^r to degree 12 (remainder below 2^-50 for |r| < 0.35) by Horner's rule with the
// coefficients 1 / n as float-float values, then the exact scaling by 2^k. Relative error
// below 2^-42 (a dozen float-float operations of about 2^-46 each, the reduction's ~2^-44).
__device__ __forceinline__ Ff ff_exp(float xh, float xl) {
    const float LN2_A = 0x1.62e4p-1f;     // ln 2 to 16 bits (45426 / 2^16)
    const float LN2_B = 0x1.7f7d1cp-20f;  // ln 2 - LN2_A rounded to fp32
    const float LN2_C = 0x1.ef357ap-45f;  // ln 2 - LN2_A - LN2_B rounded to fp32 (sum off by < 2^-69)
    const float k = rintf(xh * 1.44269504f);
    Ff r = ff_two_sum(__fsub_rn(xh, k * LN2_A), xl);  // k * LN2_A exact; xh - k LN2_A exact (Sterbenz)
    const float kb = __fmul_rn(k, LN2_B);
    r = ff_add(r, Ff{-kb, -__fmaf_rn(k, LN2_B, -kb)});
    r = ff_add(r, Ff{-__fmul_rn(k, LN2_C), 0.0f});
    // 1 / n as float-float values (the fp32 rounding and the rounded remainder)
    const float inv_hi[12] = {0x1p+0f, 0x1p-1f, 0x1.555556p-2f, 0x1p-2f, 0x1.99999ap-3f, 0x1.555556p-3f,
                              0x1.24924ap-3f, 0x1p-3f, 0x1.c71c72p-4f, 0x1.99999ap-4f, 0x1.745d18p-4f,
                              0x1.555556p-4f};
    const float inv_lo[12] = {0.0f, 0.0f, -0x1.555556p-27f, 0.0f, -0x1.99999ap-29f, -0x1.555556p-28f,
                              -0x1.b6db6ep-28f, 0.0f, -0x1.c71c72p-31f, -0x1.99999ap-30f, -0x1.745d18p-29f,
                              -0x1.555556p-29f};
    Ff p = {1.0f, 0.0f};
#pragma unroll
    for (int n = 12; n >= 1; --n) p = ff_add(Ff{1.0f, 0.0f}, ff_mul(ff_mul(r, Ff{inv_hi[n - 1], inv_lo[n - 1]}), p));
    const float s = scalbnf(1.0f, (int)k);
    return {__fmul_rn(p.hi, s), __fmul_rn(p.lo, s)};
}

// The bf16 rounding of the float-float value hi + lo (|value| in [2^-100, 2^127)) known to
// relative error eps: true with the bits when no midpoint lies within eps of it.
__device__ __forceinline__ bool bf16_decide_ff(float hi, float lo, float eps, uint16_t& out) {
    const uint16_t sign = hi < 0 ? 0x8000 : 0;
    if (hi < 0) {
        hi = -hi;
        lo = -lo;
    }
    int lead = ilogbf(hi);
    if (hi == scalbnf(1.0f, lead) && lo < 0) --lead;
    if (lead < -100 || lead > 126) return false;
    const int sc = lead >= -126 ? 7 - lead : 133;
    const int base = ((lead + 127) << 7) - 128;
    const float mh = scalbnf(hi, sc), ml = scalbnf(lo, sc);  // in units of the bf16 spacing
    float fl = floorf(mh);
    if (fl == mh && ml < 0) fl -= 1.0f;
    const float d = __fadd_rn(__fsub_rn(__fsub_rn(mh, fl), 0.5f), ml);
    if (fabsf(d) <= eps * mh) return false;
    int bits = base + (int)fl + (d > 0 ? 1 : 0);
    if (bits > 0x7F80) bits = 0x7F80;
    out = sign | (uint16_t)bits;
    return true;
}

// x = hi + lo exactly with hi = fp32(x) (nearest-even) and lo the remainder (|lo| <= 64), by
// fp32 additions alone (no conversion instruction): x = xh 2^16 + xl with xh = x >> 16 and xl
// the low 16 bits, each exact in fp32 through the 2^23 bias; hi = fma(xh, 2^16, xl) rounds the
// exact sum once, and since |xh 2^16| >= xl whenever xh != 0, the remainder of that sum is
// exact by the fast two-sum.
__device__ __forceinline__ void split_i32(int32_t x, float& hi, float& lo) {
    const float xh = __fsub_rn(__int_as_float(0x4B400000 + (x >> 16)), 12582912.0f);       // 1.5 * 2^23 + xh
    const float xl = __fsub_rn(__int_as_float(0x4B000000 | (x & 0xFFFF)), 8388608.0f);     // 2^23 + xl
    hi = __fmaf_rn(xh, 65536.0f, xl);
    lo = __fsub_rn(xl, __fmaf_rn(-xh, 65536.0f, hi));
}

// The exact operands split for fp32 arithmetic: g = g32 + gl and u = u32 + ul exactly (the
// accumulators split by split_i32, both parts scaled exactly by the powers of two; no fp64 and
// no 64-bit conversion, which GB300 runs at a small fraction of its fp32 rate), and g u = ph +
// pl + corr (ph + pl = g32 u32 exactly, corr the cross terms rounded once). Eg, Eu in [-60, 40].
struct SiluParts {
    float g32, gl, u32, ul, ph, pl, corr;
};
__device__ __forceinline__ SiluParts silu_parts(int32_t gacc, int32_t uacc, int Eg, int Eu) {
    SiluParts s;
    const float sg = __uint_as_float((uint32_t)(Eg + 127) << 23), su = __uint_as_float((uint32_t)(Eu + 127) << 23);
    float gh, glo, uh, ulo;
    split_i32(gacc, gh, glo);
    split_i32(uacc, uh, ulo);
    s.g32 = __fmul_rn(gh, sg);
    s.gl = __fmul_rn(glo, sg);
    s.u32 = __fmul_rn(uh, su);
    s.ul = __fmul_rn(ulo, su);
    s.ph = __fmul_rn(s.g32, s.u32);
    s.pl = __fmaf_rn(s.g32, s.u32, -s.ph);
    s.corr = __fmaf_rn(s.g32, s.ul, __fmaf_rn(s.gl, s.u32, __fmul_rn(s.gl, s.ul)));
    return s;
}

// An fp32 estimate of y for -80 < g32 < 64 (relative error below 11 * 2^-24: expf 4, the fma
// 1, 1 + t 1, the sum 1, __fdividef 4), which places y for the float-float evaluation.
__device__ __forceinline__ float silu_mul_f32(const SiluParts& s) {
    const float t0 = expf(-s.g32);
    const float t = __fmaf_rn(-s.gl, t0, t0);
    const float q = __fadd_rn(s.ph, __fadd_rn(s.pl, s.corr));
    return __fdividef(q, __fadd_rn(1.0f, t));
}

// SiLU(gacc 2^Eg) * uacc 2^Eu by one fp32 evaluation, for exponents already known to lie in
// [-60, 40], given as the fp32 powers of two sg = 2^Eg and su = 2^Eu (exact): returns y with
// `zero` (g u = 0 exactly when an accumulator is 0: otherwise |g u| >= 2^-120) and `ok` (y is
// decided: its nearest-even bf16 rounding is the correct one), for -87 < g32 < 64, where
//   g32 = fp32(g) and gl = g - g32 exactly (split_i32 and the exact power-of-two scaling),
//   e^-g = expf(-g32) (at most 2 ulp) times (1 - gl), to first order (gl^2 < 2^-34),
//   g u as fp32(g32 u32) with u32 = fp32(u),
//   y = __fdividef(g u, 1 + e^-g) (at most 2 ulp; 1 + e^-g lies in [1, e^87] within 2^126);
// in units of 2^-24 relative: g u 3, e^-g 5 (expf 4, the fma 1), 1 + e^-g 6, the quotient 4:
// 13, so that the fp32 result decides unless its low 16 bits lie within 13 (+3 spare) of
// 0x8000, the midpoint, or |y| < 2^-100 (|y| < 2^77 here); what is neither zero nor decided
// goes to bf16_silu_mul_careful. No function call is reachable from here, so a caller holding
// many live registers keeps them in registers.
__device__ __forceinline__ float silu_mul_f32_scaled(int32_t gacc, int32_t uacc, float sg, float su, bool& zero,
                                                     bool& ok) {
    // straight-line code (the decision is a predicate, not a branch), so that the evaluations
    // of neighbouring outputs interleave
    float gh, glo;
    split_i32(gacc, gh, glo);
    const float g32 = __fmul_rn(gh, sg);
    const float q = __fmul_rn(g32, __fmul_rn(__int2float_rn(uacc), su));
    const float t0 = expf(-g32);
    const float t = __fmaf_rn(-__fmul_rn(glo, sg), t0, t0);
    const float y = __fdividef(q, __fadd_rn(1.0f, t));
    const uint32_t b = __float_as_uint(y);
    zero = q == 0.0f;
    ok = (g32 > -87.0f) & (g32 < 64.0f) & ((b & 0x7FFFFFFFu) >= 0x0D800000u) & ((b & 0xFFFFu) - (0x8000u - 16u) > 32u);
    return y;
}

// the same with int exponents: the rounded bits, or `undecided` (and 0)
__device__ __forceinline__ uint16_t bf16_silu_mul_fast(int32_t gacc, int32_t uacc, int Eg, int Eu, bool& undecided) {
    bool zero, ok;
    const float y = silu_mul_f32_scaled(gacc, uacc, __uint_as_float((uint32_t)(Eg + 127) << 23),
                                        __uint_as_float((uint32_t)(Eu + 127) << 23), zero, ok);
    undecided = !(zero | ok);
    return zero ? (uint16_t)0 : __bfloat16_as_ushort(__float2bfloat16_rn(y));
}

// The evaluations for what bf16_silu_mul_fast leaves undecided (about one output in two
// thousand; GB300 runs fp64 arithmetic at a small fraction of its fp32 rate, so the common
// path stays free of it): g >= 64 by the exact product, g <= -700 as a signed zero, then
// float-float (|y| in [2^-100, 2^127) and -80 < g32 < 64), fp64 and double-double.
// Exponents in [-60, 40], gacc and uacc nonzero. Returns the bits, with bit 16 set when even
// the last evaluation could not decide (DEV_RANGE).
static __device__ __noinline__ uint32_t bf16_silu_mul_careful(int32_t gacc, int32_t uacc, int Eg, int Eu) {
    uint16_t out;
    const SiluParts s = silu_parts(gacc, uacc, Eg, Eu);
    if (s.g32 >= 64.0f) return bf16_round_i64((long long)gacc * (long long)uacc, Eg + Eu, true);
    if (s.g32 <= -700.0f) return ((gacc ^ uacc) < 0) ? 0x8000 : 0x0000;
    if (s.g32 > -80.0f) {
        const float ay = fabsf(silu_mul_f32(s));
        if (ay >= 0x1p-100f && ay < 0x1p127f) {
            // relative error below 2^-40: e^-g 2^-42, g u to 2^-46, the sum and the quotient
            // about 2^-45 each (measured below 2^-46 over millions of random inputs)
            const Ff gu = ff_add(Ff{s.ph, s.pl}, Ff{s.corr, 0.0f});
            const Ff yy = ff_div(gu, ff_add(Ff{1.0f, 0.0f}, ff_exp(-s.g32, -s.gl)));
            if (bf16_decide_ff(yy.hi, yy.lo, 0x1p-40f, out)) return out;
        }
    }
    const double g = scalbn((double)gacc, Eg), u = scalbn((double)uacc, Eu);  // exact
    {
        const double y = __ddiv_rn(__dmul_rn(g, u), __dadd_rn(1.0, exp(-g)));
        if (y != 0.0 && bf16_decide(y, 0.0, 0x1p-49, out)) return out;
    }
    const Dd P = dd_two_prod(g, u);  // exact
    const Dd y = dd_div(P, dd_add(Dd{1.0, 0.0}, dd_exp(-g)));
    if (bf16_decide(y.hi, y.lo, 0x1p-90, out)) return out;
    return 0x10000u | __bfloat16_as_ushort(__float2bfloat16_rn((float)y.hi));
}

// rne_bf16(SiLU(gacc 2^Eg) * uacc 2^Eu) for any exponents; `bad` is set on an exponent outside
// [-60, 40] or an output no evaluation could decide.
__device__ __forceinline__ uint16_t bf16_silu_mul(int32_t gacc, int32_t uacc, long long Eg, long long Eu, bool& bad) {
    if (gacc == 0 || uacc == 0) return 0x0000;
    if (Eg < -60 || Eg > 40 || Eu < -60 || Eu > 40) {
        bad = true;
        return 0x7FC0;
    }
    bool undecided = false;
    const uint16_t v = bf16_silu_mul_fast(gacc, uacc, (int)Eg, (int)Eu, undecided);
    if (!undecided) return v;
    const uint32_t r = bf16_silu_mul_careful(gacc, uacc, (int)Eg, (int)Eu);
    bad |= (r >> 16) != 0;
    return (uint16_t)r;
}

// bf16_silu_mul out of line, with `bad` as bit 16 of the result
static __device__ __noinline__ uint32_t bf16_silu_mul_any(int32_t gacc, int32_t uacc, long long Eg, long long Eu) {
    bool bad = false;
    const uint16_t v = bf16_silu_mul(gacc, uacc, Eg, Eu, bad);
    return v | (bad ? 0x10000u : 0u);
}

}  // namespace detgemm
