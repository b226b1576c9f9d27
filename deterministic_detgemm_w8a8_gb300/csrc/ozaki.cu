// Ozaki recombination — "GPU Mechanism", §3 "Method", Interventions (a) ExactGEMM:
// the exact diagonal sums are recombined in a fixed order in fp64 and rounded once.
//
//   acc = 0.0;  for g = D .. 2:  acc = acc + T_g * 2^(-7g);      (D = max_diag; fp64, RNE)
//   C_ij = fp32_rne(acc * 2^(e_i + f_j)).
//
// T is [D - 1][M][ldT] int32, plane d holding the diagonal g = D - d.
//
// GB300 issues fp64 arithmetic at a small fraction of its integer rate (the direct fp64
// form of this loop made the kernel bound by its ~23 fp64 operations per element, not by
// memory), so for D <= 13 the same roundings are reproduced with integer arithmetic:
// every value the fp64 loop produces is an integer multiple of 2^(-7D), so at the scale
// 2^(7D) the loop is
//     Z = 0;  for g = D .. 2:  Z = rne53(Z + T_g * 2^(7 (D - g)))
// where rne53 rounds an integer to 53 significant bits, half to even — exactly what one
// fp64 addition of two exact operands does (no intermediate can be subnormal: a nonzero
// |value| is at least 2^(-7D) >= 2^-91, and at most 2^108 < 2^127 fits a signed 128-bit
// integer for D <= 13). The first four sums are below 2^53 and need no rounding. The
// result Z * 2^(e_i + f_j - 7D) is then rounded once to fp32 (subnormals kept, overflow
// to infinity), as the fp64 product and the fp32 conversion do: the product is exact in
// fp64 because it stays inside fp64's normal range. For D > 13 the loop runs in fp64.
//
// Traffic per element: 4 (D - 1) B read + 4 B written; each thread takes four
// consecutive columns (16-byte loads and stores).
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace detgemm {

namespace {

typedef unsigned __int128 u128;
typedef __int128 i128;

__device__ __forceinline__ int bitlen128(u128 m) {
    const uint64_t hi = (uint64_t)(m >> 64), lo = (uint64_t)m;
    return hi ? 128 - __clzll((long long)hi) : 64 - __clzll((long long)lo);
}

// x (|x| < 2^127) rounded to 53 significant bits, ties to even, returned as q * 2^sh
// with q an int64. Works on the two's complement words directly: the shift is a floor,
// rem = x - q 2^sh is in [0, 2^sh), and rounding up on rem > half (or on a tie with q
// odd) is round-half-even for either sign. The bit length of |x| is taken from x ^ sign
// (= -x - 1 for x < 0), which differs from |x| only when |x| is a power of two, which
// needs no rounding either way. Here |x| < 2^109, so 1 <= sh <= 56.
__device__ __forceinline__ long long rne53(i128 x, int& sh_out) {
    const uint64_t lo = (uint64_t)x;
    const int64_t hi = (int64_t)(x >> 64);
    const int64_t sm = hi >> 63;
    const uint64_t yhi = (uint64_t)(hi ^ sm), ylo = lo ^ (uint64_t)sm;
    const int nb = yhi ? 128 - __clzll((long long)yhi) : 64 - __clzll((long long)ylo);
    if (nb <= 53) {  // |x| <= 2^53: exact, and it fits the low word
        sh_out = 0;
        return (long long)lo;
    }
    const int sh = nb - 53;
    long long q = (long long)((lo >> sh) | ((uint64_t)hi << (64 - sh)));
    const uint64_t rem = lo & ((1ull << sh) - 1ull);
    const uint64_t half = 1ull << (sh - 1);
    q += (long long)((rem > half) | ((rem == half) & ((uint64_t)q & 1ull)));
    sh_out = sh;
    return q;
}

// X (|X| < 2^63) rounded to 53 significant bits, ties to even, as q * 2^s (|q| <= 2^53):
// the same rounding as rne53 for a value that fits a 64-bit word, on its magnitude
__device__ __forceinline__ long long rne53_i64(long long X, int& s) {
    const uint64_t a = X < 0 ? 0ull - (uint64_t)X : (uint64_t)X;
    const int nb = 64 - __clzll((long long)a);
    if (nb <= 53) {
        s = 0;
        return X;
    }
    s = nb - 53;
    uint64_t qq = a >> s;
    const uint64_t rem = a & ((1ull << s) - 1ull);
    const uint64_t half = 1ull << (s - 1);
    qq += (uint64_t)((rem > half) | ((rem == half) & (qq & 1ull)));
    return X < 0 ? -(long long)qq : (long long)qq;
}

// q * 2^sh as a 128-bit integer (0 <= sh <= 63)
__device__ __forceinline__ i128 widen_shifted(long long q, int sh) {
    const uint64_t lo = (uint64_t)q << sh;
    const int64_t hi = sh ? (q >> (64 - sh)) : (q >> 63);
    return (i128)(((u128)(uint64_t)hi << 64) | (u128)lo);
}

// fp32 round-to-nearest-even of Z * 2^s (Z an integer, |Z| < 2^127), subnormals kept,
// overflow to infinity; +0 for Z == 0
__device__ __noinline__ float f32_from_i128_pow2(i128 Z, int s) {
    if (Z == 0) return 0.0f;
    const uint32_t sign = Z < 0 ? 0x80000000u : 0u;
    const u128 m = Z < 0 ? (u128)0 - (u128)Z : (u128)Z;
    const int nb = bitlen128(m);
    const int E = nb - 1 + s;  // exponent of the leading bit
    if (E > 127) return __uint_as_float(sign | 0x7F800000u);
    int sh;
    uint32_t base;
    if (E >= -126) {
        sh = nb - 24;
        base = (uint32_t)(E + 126) << 23;  // (biased exponent - 1): q carries the leading one
    } else {
        sh = -149 - s;                      // subnormal: units of 2^-149
        base = 0u;
    }
    uint32_t q;
    if (sh <= 0) {
        q = (uint32_t)m << (-sh);  // m < 2^24 here
    } else if (sh > nb) {
        q = 0u;  // below half a unit
    } else {
        const u128 qq = m >> sh;
        const u128 rem = m - (qq << sh);
        const u128 half = (u128)1 << (sh - 1);
        q = (uint32_t)qq + (uint32_t)((rem > half) | ((rem == half) & ((uint32_t)qq & 1u)));
    }
    uint32_t bits = base + q;
    if (bits >= 0x7F800000u) bits = 0x7F800000u;
    return __uint_as_float(sign | bits);
}

// fp32 round-to-nearest-even of q * 2^t. When the result is a normal number the
// hardware conversion rounds q to 24 bits (exactly the same rounding, as scaling by a
// power of two commutes with rounding there) and t is added to the exponent field;
// subnormal and overflowing results take the integer construction.
__device__ __forceinline__ float f32_from_q(long long q, int t) {
    if (q == 0) return 0.0f;
    const uint64_t a = q < 0 ? 0ull - (uint64_t)q : (uint64_t)q;
    const int E = 63 - __clzll((long long)a) + t;  // exponent of the leading bit
    if (E >= -126 && E <= 126) {                   // stays normal after a round-up
        const float f = __ll2float_rn(q);
        return __uint_as_float(__float_as_uint(f) + ((uint32_t)t << 23));
    }
    return f32_from_i128_pow2((i128)q, t);
}

// fp64 round-to-nearest-even of q * 2^t (|q| <= 2^53): exact for normal results (q has at
// most 53 significant bits), rounded at 2^-1074 for subnormal ones, infinity on overflow
__device__ __forceinline__ double f64_from_q(long long q, int t) {
    if (q == 0) return 0.0;
    const uint64_t sign = q < 0 ? 0x8000000000000000ull : 0ull;
    const uint64_t a = q < 0 ? 0ull - (uint64_t)q : (uint64_t)q;
    const int nb = 64 - __clzll((long long)a);
    const int E = nb - 1 + t;
    if (E > 1023) return __longlong_as_double((long long)(sign | 0x7FF0000000000000ull));
    uint64_t bits;
    if (E >= -1022) {
        const uint64_t m = nb <= 53 ? a << (53 - nb) : a >> (nb - 53);  // a = 2^53 drops a zero
        bits = ((uint64_t)(E + 1023) << 52) | (m & 0x000FFFFFFFFFFFFFull);
    } else {
        const int up = t + 1074;  // value in units of 2^-1074 is a * 2^up
        if (up >= 0) {
            bits = a << up;  // < 2^52: exact
        } else {
            const int sh = -up;
            if (sh > nb) {
                bits = 0;  // below half a unit
            } else {
                const uint64_t qq = sh >= 64 ? 0ull : a >> sh;
                const uint64_t rem = a - (sh >= 64 ? 0ull : qq << sh);
                const uint64_t half = 1ull << (sh - 1);
                bits = qq + (uint64_t)((rem > half) | ((rem == half) & (qq & 1ull)));
            }
        }
    }
    return __longlong_as_double((long long)(sign | bits));
}

template <typename OutT>
struct Out;
template <>
struct Out<float> {
    static constexpr int KMAX = 300;  // |acc| in [2^-91, 2^109): beyond, 0 or inf either way
    static __device__ __forceinline__ float from_q(long long q, int t) { return f32_from_q(q, t); }
};
template <>
struct Out<double> {
    static constexpr int KMAX = 2200;
    static __device__ __forceinline__ double from_q(long long q, int t) { return f64_from_q(q, t); }
};

// the fixed-order combine of one element; t[d] = T_(D - d)
template <int D, typename OutT>
__device__ __forceinline__ OutT combine_int(const int32_t (&t)[D - 1], int32_t ei, int32_t fj) {
    long long q = 0;
    constexpr int EXACT = D - 1 < 4 ? D - 1 : 4;
#pragma unroll
    for (int d = 0; d < EXACT; ++d) q += (long long)t[d] * (1ll << (7 * d));  // |q| < 2^53: no rounding
    int sh = 0;
    // Each rounding step forms Z * 2^sh + T * 2^(7d) and rounds it to 53 bits. While the sum,
    // taken in units of 2^sh, fits a 64-bit word (|q| <= 2^53 and |T| 2^(7d - sh) < 2^62),
    // it is formed and rounded in int64 — the same value and the same rounding; otherwise in
    // 128 bits from there on.
    bool fast = true;
#pragma unroll
    for (int d = EXACT; d < D - 1; ++d) {
        if (fast) {
            const int k = 7 * d - sh;
            const uint32_t at = t[d] < 0 ? 0u - (uint32_t)t[d] : (uint32_t)t[d];
            if (k >= 0 && 32 - __clz(at) + k <= 62) {
                int s2;
                q = rne53_i64(q + (long long)t[d] * (1ll << k), s2);
                sh += s2;
                continue;
            }
            fast = false;
        }
        q = rne53(widen_shifted(q, sh) + (i128)((u128)(i128)t[d] << (7 * d)), sh);
    }
    long long k = (long long)ei + (long long)fj;
    k = k > Out<OutT>::KMAX ? Out<OutT>::KMAX : (k < -Out<OutT>::KMAX ? -Out<OutT>::KMAX : k);
    return Out<OutT>::from_q(q, sh + (int)k - 7 * D);
}

template <int D, typename OutT>
__global__ void __launch_bounds__(256) ozaki_combine_int_kernel(const int32_t* __restrict__ T, int64_t ldT,
                                                                const int32_t* __restrict__ e,
                                                                const int32_t* __restrict__ f, OutT* __restrict__ C,
                                                                int64_t ldc, int M, int N) {
    const int j0 = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    const int i = blockIdx.y;
    if (j0 >= N || i >= M) return;
    const int64_t plane = (int64_t)M * ldT;
    const int64_t idx = (int64_t)i * ldT + j0;
    const int32_t ei = __ldg(e + i);
    OutT* c = C + (int64_t)i * ldc + j0;
    if (j0 + 4 <= N) {
        int4 v[D - 1];
#pragma unroll
        for (int d = 0; d < D - 1; ++d) v[d] = __ldcs(reinterpret_cast<const int4*>(T + d * plane + idx));
        const int4 fv = __ldg(reinterpret_cast<const int4*>(f + j0));
        OutT out[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            int32_t t[D - 1];
#pragma unroll
            for (int d = 0; d < D - 1; ++d) t[d] = q == 0 ? v[d].x : q == 1 ? v[d].y : q == 2 ? v[d].z : v[d].w;
            const int32_t fj = q == 0 ? fv.x : q == 1 ? fv.y : q == 2 ? fv.z : fv.w;
            out[q] = combine_int<D, OutT>(t, ei, fj);
        }
        if (sizeof(OutT) == 4) {
            __stcs(reinterpret_cast<float4*>(c), *reinterpret_cast<const float4*>(out));
        } else {
            __stcs(reinterpret_cast<double2*>(c), *reinterpret_cast<const double2*>(out));
            __stcs(reinterpret_cast<double2*>(c) + 1, *(reinterpret_cast<const double2*>(out) + 1));
        }
    } else {
        for (int q = 0; j0 + q < N; ++q) {
            int32_t t[D - 1];
#pragma unroll
            for (int d = 0; d < D - 1; ++d) t[d] = T[d * plane + idx + q];
            c[q] = combine_int<D, OutT>(t, ei, f[j0 + q]);
        }
    }
}

// any D (up to 18): the loop in fp64 as written; for fp64 output the final scaling is one
// exact multiply that keeps acc normal and one that rounds (|acc| in [2^-126, 2^144))
__device__ __forceinline__ float scale_out(double acc, long long k, float*) {
    k = k > 300 ? 300 : (k < -300 ? -300 : k);
    return __double2float_rn(__dmul_rn(acc, pow2_f64((int)k)));
}
__device__ __forceinline__ double scale_out(double acc, long long k, double*) {
    k = k > 2200 ? 2200 : (k < -2200 ? -2200 : k);
    const long long k1 = k > 800 ? 800 : (k < -800 ? -800 : k);
    long long k2 = k - k1;
    k2 = k2 > 1000 ? 1000 : (k2 < -1000 ? -1000 : k2);  // beyond: 0 or inf either way
    return __dmul_rn(__dmul_rn(acc, pow2_f64((int)k1)), pow2_f64((int)k2));
}

template <typename OutT>
__global__ void ozaki_combine_f64_kernel(const int32_t* __restrict__ T, int64_t ldT, int max_diag,
                                         const int32_t* __restrict__ e, const int32_t* __restrict__ f,
                                         OutT* __restrict__ C, int64_t ldc, int M, int N) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    const int i = blockIdx.y;
    if (j >= N) return;
    const int64_t plane = (int64_t)M * ldT;
    const int64_t idx = (int64_t)i * ldT + j;
    double acc = 0.0;
    for (int g = max_diag; g >= 2; --g)
        acc = __dadd_rn(acc, __dmul_rn((double)__ldg(T + (int64_t)(max_diag - g) * plane + idx), pow2_f64(-7 * g)));
    C[(int64_t)i * ldc + j] = scale_out(acc, (long long)e[i] + (long long)f[j], (OutT*)nullptr);
}

template <int D, typename OutT>
cudaError_t launch_int(const int32_t* T, int64_t ldT, const int32_t* e, const int32_t* f, OutT* C, int64_t ldc,
                       int M, int N, cudaStream_t s) {
    dim3 grid((unsigned)(((N + 3) / 4 + 255) / 256), (unsigned)M);
    ozaki_combine_int_kernel<D, OutT><<<grid, 256, 0, s>>>(T, ldT, e, f, C, ldc, M, N);
    return cudaGetLastError();
}

template <typename OutT>
cudaError_t combine_launch(const int32_t* T, int64_t ldT, int max_diag, const int32_t* e, const int32_t* f, OutT* C,
                           int64_t ldc, int M, int N, cudaStream_t s) {
    if (M == 0 || N == 0) return cudaSuccess;
    // the integer kernels use 16-byte loads of T and f and 16-byte stores of C
    const bool vec = (ldT % 4) == 0 && ((ldc * (int64_t)sizeof(OutT)) % 16) == 0 &&
                     (reinterpret_cast<uintptr_t>(T) & 15u) == 0 && (reinterpret_cast<uintptr_t>(f) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(C) & 15u) == 0;
    if (vec) {
        switch (max_diag) {
            case 2: return launch_int<2>(T, ldT, e, f, C, ldc, M, N, s);
            case 3: return launch_int<3>(T, ldT, e, f, C, ldc, M, N, s);
            case 4: return launch_int<4>(T, ldT, e, f, C, ldc, M, N, s);
            case 5: return launch_int<5>(T, ldT, e, f, C, ldc, M, N, s);
            case 6: return launch_int<6>(T, ldT, e, f, C, ldc, M, N, s);
            case 7: return launch_int<7>(T, ldT, e, f, C, ldc, M, N, s);
            case 8: return launch_int<8>(T, ldT, e, f, C, ldc, M, N, s);
            case 9: return launch_int<9>(T, ldT, e, f, C, ldc, M, N, s);
            case 10: return launch_int<10>(T, ldT, e, f, C, ldc, M, N, s);
            case 11: return launch_int<11>(T, ldT, e, f, C, ldc, M, N, s);
            case 12: return launch_int<12>(T, ldT, e, f, C, ldc, M, N, s);
            case 13: return launch_int<13>(T, ldT, e, f, C, ldc, M, N, s);
            default: break;
        }
    }
    dim3 grid((N + 255) / 256, M);
    ozaki_combine_f64_kernel<OutT><<<grid, 256, 0, s>>>(T, ldT, max_diag, e, f, C, ldc, M, N);
    return cudaGetLastError();
}

}  // namespace

cudaError_t ozaki_combine_launch(const int32_t* T, int64_t ldT, int max_diag, const int32_t* e, const int32_t* f,
                                 float* C, int64_t ldc, int M, int N, cudaStream_t s) {
    return combine_launch<float>(T, ldT, max_diag, e, f, C, ldc, M, N, s);
}

cudaError_t ozaki_combine_f64out_launch(const int32_t* T, int64_t ldT, int max_diag, const int32_t* e,
                                        const int32_t* f, double* C, int64_t ldc, int M, int N, cudaStream_t s) {
    return combine_launch<double>(T, ldT, max_diag, e, f, C, ldc, M, N, s);
}

}  // namespace detgemm
