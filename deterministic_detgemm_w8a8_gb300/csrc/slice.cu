// Ozaki slicing — "GPU Mechanism", §3 "Method", Interventions (a) ExactGEMM: each
// operand is cut into 7-bit integer slices scaled by powers of two from frexp.
//
// One exponent per line (row of A, column of B): e = frexp exponent of the line's max
// |x|, so max|x| < 2^e. A value's digits are the signed base-128 digits of
//     R = trunc(|x| * 2^(7 n - e))            (n = nslices)
// most significant first; this equals the iteration d_t = trunc(128 r),
// r <- 128 r - d_t on r = x 2^-e, because truncation toward zero is sign-symmetric.
// With |x| = M 2^(p - mb) (M the significand with its leading one, mb its fraction bits),
// digit t (t = 0 first) is floor(M 2^(p - mb - e + 7 (t + 1))) mod 128, taken with one
// shift of M, so the digits are exact for fp32 and fp64 inputs and any n.
//
// The line exponent is the frexp exponent of the line's largest |x| (taken as a maximum
// of bit patterns), carried as an int with sentinels for zero and for inf/NaN; across
// row chunks of a column these exponents combine with atomicMax (frexp's exponent is
// monotone in |x|). Rows: one CTA per row, two passes (exponent, then digits), eight columns
// per thread. Columns: a kernel reduces the column exponents with atomicMax, then a 64 x 64
// tiled transpose writes every digit plane K-major ([t][col][row]), then a small kernel
// turns the sentinels into exponents (0) and flags non-finite columns.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace detgemm {

namespace {

constexpr int SROW_THREADS = 256;
constexpr int KEY_NONFINITE = INT_MAX;
constexpr int KEY_ZERO = (int)0x80808080u;  // below every exponent; a byte-wise memset value

template <typename X>
struct FP;
template <>
struct FP<float> {
    typedef uint32_t Bits;
    static constexpr int MB = 23, BIAS = 127;
    static constexpr uint32_t ABS = 0x7FFFFFFFu, EXP_ALL = 0xFFu;
};
template <>
struct FP<double> {
    typedef uint64_t Bits;
    static constexpr int MB = 52, BIAS = 1023;
    static constexpr uint64_t ABS = 0x7FFFFFFFFFFFFFFFull, EXP_ALL = 0x7FFull;
};

template <typename X>
__device__ __forceinline__ typename FP<X>::Bits bits_of(X x);
template <>
__device__ __forceinline__ uint32_t bits_of<float>(float x) {
    return __float_as_uint(x);
}
template <>
__device__ __forceinline__ uint64_t bits_of<double>(double x) {
    return (uint64_t)__double_as_longlong(x);
}

// |x| = M 2^(p - MB) with M holding the leading one at bit MB; false for zero
template <typename X>
__device__ __forceinline__ bool normalise(typename FP<X>::Bits b, uint64_t& M, int& p) {
    typedef FP<X> F;
    const uint64_t a = (uint64_t)(b & F::ABS);
    const int ef = (int)(a >> F::MB);
    const uint64_t fr = a & ((1ull << F::MB) - 1ull);
    if (ef == 0) {
        if (fr == 0) return false;
        const int msb = 63 - __clzll((long long)fr);
        M = fr << (F::MB - msb);
        p = msb + 1 - F::BIAS - F::MB;
        return true;
    }
    M = fr | (1ull << F::MB);
    p = ef - F::BIAS;
    return true;
}

// frexp exponent of x (|x| < 2^e <= 2 |x|), or a sentinel for zero / inf / NaN
template <typename X>
__device__ __forceinline__ int exp_key(typename FP<X>::Bits b) {
    typedef FP<X> F;
    if (((b & F::ABS) >> F::MB) == F::EXP_ALL) return KEY_NONFINITE;
    uint64_t M;
    int p;
    if (!normalise<X>(b, M, p)) return KEY_ZERO;
    return p + 1;
}

// x (bits b) prepared for digit extraction under the line exponent e. Up to 9 slices the
// whole digit string R = trunc(|x| 2^(7 n - e)) < 2^63 is formed once and digit t is one
// shift of it; beyond, digit t is taken from the significand with its own shift. Either way
// nothing is indexed by t, so everything stays in registers.
struct Digits {
    uint64_t M;  // R (n <= 9) or the significand (n > 9)
    int base;    // p - mb - e (n > 9)
    bool neg, nz;
};

template <typename X>
__device__ __forceinline__ Digits prep_digits(typename FP<X>::Bits b, int e, int n) {
    Digits g;
    int p = 0;
    g.M = 0;
    g.nz = normalise<X>(b, g.M, p);
    g.neg = (b >> (8 * sizeof(b) - 1)) != 0;
    g.base = p - FP<X>::MB - e;
    if (n <= 9) {
        const int sh = g.base + 7 * n;  // R = M 2^sh
        g.M = !g.nz ? 0ull : sh >= 0 ? g.M << sh : (-sh >= 64 ? 0ull : g.M >> (-sh));
    }
    return g;
}

__device__ __forceinline__ int8_t digit_at(const Digits& g, int t, int n) {
    uint32_t v;
    if (n <= 9) {
        v = (uint32_t)(g.M >> (7 * (n - 1 - t))) & 127u;
    } else {
        const int sh = g.base + 7 * (t + 1);
        if (!g.nz || sh >= 7) v = 0u;
        else if (sh >= 0) v = (uint32_t)(g.M << sh) & 127u;
        else v = (-sh >= 64) ? 0u : (uint32_t)(g.M >> (-sh)) & 127u;
    }
    return (int8_t)(g.neg ? -(int)v : (int)v);
}

// digit planes are stored as int8 (the public slicer) or as exact fp16 values (the
// operand planes of the tensor-core engine)
template <typename T>
__device__ __forceinline__ T digit_out(int8_t d) {
    return Pack8<T>::one(d);
}

__device__ __forceinline__ int max_key_block(int key, int* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = key;
    __syncthreads();
    key = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) key = max(key, red[w]);
    return key;
}

// eight consecutive elements' bits (zero beyond cols), 16-byte loads when aligned
template <typename X>
__device__ __forceinline__ void load8(const X* x, int j0, int cols, bool vec, typename FP<X>::Bits (&v)[8]) {
    typedef typename FP<X>::Bits B;
    constexpr int PER = (int)(16 / sizeof(X));  // elements per 16-byte load
    if (vec && j0 + 8 <= cols) {
        const uint4* q = reinterpret_cast<const uint4*>(x + j0);
#pragma unroll
        for (int i = 0; i < 8 / PER; ++i) {
            const uint4 a = __ldg(q + i);
            const B* w = reinterpret_cast<const B*>(&a);
#pragma unroll
            for (int k = 0; k < PER; ++k) v[i * PER + k] = w[k];
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = j0 + i < cols ? bits_of<X>(x[j0 + i]) : (B)0;
    }
}

// One CTA per row, eight columns per thread: pass 1 reduces the row's exponent, pass 2
// re-reads the row (cache resident) and writes each plane's eight digits with one store
// (when the plane's row stride allows it).
template <typename X, typename T>
__global__ void __launch_bounds__(SROW_THREADS) slice_rows_kernel(const X* __restrict__ Xm, int64_t ldx, int rows,
                                                                  int cols, int nslices, T* __restrict__ S,
                                                                  int64_t lds, int32_t* __restrict__ e_out) {
    typedef typename FP<X>::Bits B;
    __shared__ int red[SROW_THREADS / 32];
    const int64_t row = blockIdx.x;
    const X* x = Xm + row * ldx;
    const bool vec_in = ((ldx * (int64_t)sizeof(X)) % 16) == 0 && (reinterpret_cast<uintptr_t>(Xm) & 15u) == 0;
    // max |x| as bits (for non-negative floating-point values the bit order is the value
    // order, and inf/NaN bits lie above every finite value), then its exponent once
    B amax = 0;
    for (int j0 = threadIdx.x * 8; j0 < cols; j0 += SROW_THREADS * 8) {
        B v[8];
        load8<X>(x, j0, cols, vec_in, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = max(amax, (B)(v[i] & FP<X>::ABS));
    }
    int key = max_key_block(exp_key<X>(amax), red);
    const bool bad = key == KEY_NONFINITE;  // inf or NaN in the row: digits written as zero
    const bool zero = key == KEY_ZERO;
    const int e = (bad || zero) ? 0 : key;
    if (threadIdx.x == 0) {
        if (bad) raise_status(DEV_NONFINITE);
        e_out[row] = e;
    }
    const int64_t plane = (int64_t)rows * lds;
    T* srow = S + row * lds;
    const bool vec_out = (lds % 8) == 0 && (reinterpret_cast<uintptr_t>(S) & 15u) == 0;
    for (int j0 = threadIdx.x * 8; j0 < lds; j0 += SROW_THREADS * 8) {
        B v[8];
        load8<X>(x, j0, cols, vec_in, v);  // zero beyond cols: the padding up to lds gets zero digits
        Digits g[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) g[i] = prep_digits<X>((bad || zero) ? (B)0 : v[i], e, nslices);
        for (int t = 0; t < nslices; ++t) {
            int8_t dt[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) dt[i] = digit_at(g[i], t, nslices);
            T* dst = srow + t * plane + j0;
            if (vec_out) {
                *reinterpret_cast<typename Pack8<T>::type*>(dst) = Pack8<T>::make(dt);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (j0 + i < lds) dst[i] = digit_out<T>(dt[i]);
            }
        }
    }
}

// column exponents: block (32 columns) x (8 row lanes), one chunk of rows per blockIdx.y;
// keys[c] starts at KEY_ZERO (byte-wise memset) and takes the atomic max
constexpr int CM_ROWS = 256;

template <typename X>
__global__ void col_key_kernel(const X* __restrict__ Xm, int64_t ldx, int rows, int cols, int* __restrict__ keys) {
    __shared__ int red[8][32];
    const int j = blockIdx.x * 32 + threadIdx.x;
    const int r0 = blockIdx.y * CM_ROWS;
    const int r1 = min(rows, r0 + CM_ROWS);
    typename FP<X>::Bits amax = 0;
    if (j < cols)
        for (int r = r0 + threadIdx.y; r < r1; r += 8) amax = max(amax, bits_of<X>(Xm[(int64_t)r * ldx + j]) & FP<X>::ABS);
    int m = exp_key<X>(amax);
    red[threadIdx.y][threadIdx.x] = m;
    __syncthreads();
    if (threadIdx.y == 0 && j < cols) {
#pragma unroll
        for (int y = 1; y < 8; ++y) m = max(m, red[y][threadIdx.x]);
        if (m != KEY_ZERO) atomicMax(keys + j, m);
    }
}

// 64 x 64 tile of X (rows r0.., columns c0..), 256 threads: each thread loads four
// columns of four consecutive rows, its digits go to a shared tile [t][col][row] (four rows
// per 32-bit store), then each plane is
// written K-major, S[t][col][row], eight rows per store (each column's 64 rows are 128
// contiguous bytes of fp16).
constexpr int SC_TILE = 64;
constexpr int SC_PITCH = SC_TILE + 4;  // bytes per (t, col) line of the shared tile

template <typename X, typename T>
__global__ void __launch_bounds__(256) slice_cols_kernel(const X* __restrict__ Xm, int64_t ldx, int rows, int cols,
                                                         int nslices, const int32_t* __restrict__ keys,
                                                         T* __restrict__ S, int64_t lds) {
    typedef typename FP<X>::Bits B;
    constexpr int PER = (int)(16 / sizeof(X));
    extern __shared__ __align__(16) int8_t tile[];  // [nslices][SC_TILE][SC_PITCH]
    const int r0 = blockIdx.y * SC_TILE, c0 = blockIdx.x * SC_TILE;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 column quads x 16 row lanes
    const bool vec_in = ((ldx * (int64_t)sizeof(X)) % 16) == 0 && (reinterpret_cast<uintptr_t>(Xm) & 15u) == 0;
    const int cq = c0 + 4 * tx;
    int ecol[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) ecol[q] = cq + q < cols ? keys[cq + q] : KEY_ZERO;
    // rows 4 ty .. 4 ty + 3 of columns cq .. cq + 3: all four rows are loaded first, then each
    // (plane, column) gets its four row digits in one 32-bit shared-memory store
    B v[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + 4 * ty + i;
#pragma unroll
        for (int q = 0; q < 4; ++q) v[i][q] = 0;
        if (r < rows) {
            const X* xr = Xm + (int64_t)r * ldx;
            if (vec_in && cq + 4 <= cols) {
                const uint4* qp = reinterpret_cast<const uint4*>(xr + cq);
#pragma unroll
                for (int h = 0; h < 4 / PER; ++h) {
                    const uint4 a = __ldg(qp + h);
                    const B* w = reinterpret_cast<const B*>(&a);
#pragma unroll
                    for (int k = 0; k < PER; ++k) v[i][h * PER + k] = w[k];
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) v[i][q] = cq + q < cols ? bits_of<X>(xr[cq + q]) : (B)0;
            }
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        // a column marked non-finite or all-zero (or outside the matrix) gets zero digits
        const bool live = ecol[q] != KEY_NONFINITE && ecol[q] != KEY_ZERO;
        Digits g[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) g[i] = prep_digits<X>(live ? v[i][q] : (B)0, live ? ecol[q] : 0, nslices);
        for (int t = 0; t < nslices; ++t) {
            uint32_t w = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) w |= (uint32_t)(uint8_t)digit_at(g[i], t, nslices) << (8 * i);
            *reinterpret_cast<uint32_t*>(&tile[(t * SC_TILE + 4 * tx + q) * SC_PITCH + 4 * ty]) = w;
        }
    }
    __syncthreads();
    const int64_t plane = (int64_t)cols * lds;
    const bool vec_out = (lds % 8) == 0 && (reinterpret_cast<uintptr_t>(S) & 15u) == 0;
    const int chunks = nslices * SC_TILE * (SC_TILE / 8);  // (t, col, 8-row group)
    for (int w = threadIdx.x; w < chunks; w += 256) {
        const int g8 = w & 7, cc = (w >> 3) & (SC_TILE - 1), t = w >> 9;
        const int c = c0 + cc, r = r0 + 8 * g8;
        if (c >= cols || r >= lds) continue;  // rows in [rows, lds) are the zero padding
        const uint32_t* src = reinterpret_cast<const uint32_t*>(&tile[(t * SC_TILE + cc) * SC_PITCH + 8 * g8]);
        const uint32_t lo = src[0], hi = src[1];
        int8_t d[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            d[i] = (int8_t)(lo >> (8 * i));
            d[i + 4] = (int8_t)(hi >> (8 * i));
        }
        T* dst = S + t * plane + (int64_t)c * lds + r;
        if (vec_out && r + 8 <= lds) {
            *reinterpret_cast<typename Pack8<T>::type*>(dst) = Pack8<T>::make(d);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (r + i < lds) dst[i] = digit_out<T>(d[i]);
        }
    }
}

// sentinel keys -> exponents: an all-zero column gets 0, a non-finite one 0 and the flag
__global__ void col_finish_kernel(int32_t* e_out, int cols) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= cols) return;
    const int k = e_out[j];
    if (k == KEY_NONFINITE) {
        raise_status(DEV_NONFINITE);
        e_out[j] = 0;
    } else if (k == KEY_ZERO) {
        e_out[j] = 0;
    }
}

template <typename X, typename T>
cudaError_t rows_launch(const X* Xm, int64_t ldx, int rows, int cols, int nslices, T* S, int64_t lds, int32_t* e,
                        cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    slice_rows_kernel<X, T><<<rows, SROW_THREADS, 0, s>>>(Xm, ldx, rows, cols, nslices, S, lds, e);
    return cudaGetLastError();
}

template <typename X, typename T>
cudaError_t cols_launch(const X* Xm, int64_t ldx, int rows, int cols, int nslices, T* S, int64_t lds, int32_t* e,
                        cudaStream_t s) {
    if (cols == 0) return cudaSuccess;
    cudaError_t err = cudaMemsetAsync(e, 0x80, (size_t)cols * sizeof(int32_t), s);  // KEY_ZERO
    if (err != cudaSuccess) return err;
    if (rows > 0) {
        dim3 g1((cols + 31) / 32, (rows + CM_ROWS - 1) / CM_ROWS);
        col_key_kernel<X><<<g1, dim3(32, 8), 0, s>>>(Xm, ldx, rows, cols, e);
    }
    const int smem = nslices * SC_TILE * SC_PITCH;
    if (smem > 48 * 1024) {
        err = cudaFuncSetAttribute(slice_cols_kernel<X, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
    }
    dim3 g2((cols + SC_TILE - 1) / SC_TILE, (int)((lds + SC_TILE - 1) / SC_TILE));
    if (lds > 0) slice_cols_kernel<X, T><<<g2, 256, smem, s>>>(Xm, ldx, rows, cols, nslices, e, S, lds);
    col_finish_kernel<<<(cols + 255) / 256, 256, 0, s>>>(e, cols);
    return cudaGetLastError();
}

}  // namespace

cudaError_t slice_rows_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, int8_t* S, int64_t lds,
                              int32_t* e, cudaStream_t s) {
    return rows_launch<float, int8_t>(X, ldx, rows, cols, nslices, S, lds, e, s);
}

cudaError_t slice_cols_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, int8_t* S, int64_t lds,
                              int32_t* e, cudaStream_t s) {
    return cols_launch<float, int8_t>(X, ldx, rows, cols, nslices, S, lds, e, s);
}

cudaError_t slice_rows_f16_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, void* S, int64_t lds,
                                  int32_t* e, cudaStream_t s) {
    return rows_launch<float, __half>(X, ldx, rows, cols, nslices, reinterpret_cast<__half*>(S), lds, e, s);
}

cudaError_t slice_cols_f16_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, void* S, int64_t lds,
                                  int32_t* e, cudaStream_t s) {
    return cols_launch<float, __half>(X, ldx, rows, cols, nslices, reinterpret_cast<__half*>(S), lds, e, s);
}

cudaError_t slice_f64_launch(const double* X, int64_t ldx, int rows, int cols, int axis, int nslices, int8_t* S,
                             int64_t lds, int32_t* e, cudaStream_t s) {
    if (axis == 0) return rows_launch<double, int8_t>(X, ldx, rows, cols, nslices, S, lds, e, s);
    return cols_launch<double, int8_t>(X, ldx, rows, cols, nslices, S, lds, e, s);
}

cudaError_t slice_f64_f16_launch(const double* X, int64_t ldx, int rows, int cols, int axis, int nslices, void* S,
                                 int64_t lds, int32_t* e, cudaStream_t s) {
    if (axis == 0)
        return rows_launch<double, __half>(X, ldx, rows, cols, nslices, reinterpret_cast<__half*>(S), lds, e, s);
    return cols_launch<double, __half>(X, ldx, rows, cols, nslices, reinterpret_cast<__half*>(S), lds, e, s);
}

DETGEMM_STATUS_ACCESSOR(slice_take_status)

}  // namespace detgemm
