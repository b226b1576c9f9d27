// Ozaki slicing — "GPU Mechanism", §3 "Method", Interventions (a) ExactGEMM: each
// operand is cut into 7-bit integer slices scaled by powers of two from frexp.
//
// One exponent per line (row of A, column of B): e = frexp exponent of the line's max
// |x|, so max|x| < 2^e. A value's digits are the signed base-128 digits of
//     R = trunc(|x| * 2^(7 n - e))            (n = nslices, R < 2^(7n))
// most significant first; this equals the iteration d_t = trunc(128 r),
// r <- 128 r - d_t on r = x 2^-e, because truncation toward zero is sign-symmetric.
// R is formed with integer shifts of the fp32 significand, so it is exact.
//
// Rows: one CTA per row, two passes (max, then digits), eight columns per thread.
// Columns: a column-max kernel (atomicMax over row chunks), an exponent kernel, then a
// 64 x 64 tiled transpose that writes every digit plane K-major ([t][col][row]).
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace detgemm {

namespace {

constexpr int SROW_THREADS = 256;

// frexp exponent from the fp32 bits of max|x| (0 for zero)
__device__ __forceinline__ int line_exponent(uint32_t amax) {
    uint32_t M;
    int p;
    if (!f32_normalise(amax, M, p)) return 0;
    return p + 1;
}

// R = trunc(|x| 2^(7n - e)) for fp32 bits xb
__device__ __forceinline__ unsigned long long digits_of(uint32_t xb, int e, int n) {
    uint32_t M;
    int p;
    if (!f32_normalise(xb & 0x7FFFFFFFu, M, p)) return 0ull;
    int sh = p - 23 + 7 * n - e;
    if (sh >= 0) return (unsigned long long)M << sh;
    int r = -sh;
    return r >= 32 ? 0ull : (unsigned long long)(M >> r);
}

__device__ __forceinline__ int8_t digit(unsigned long long R, int t, int n, bool neg) {
    int d = (int)((R >> (7 * (n - 1 - t))) & 127ull);
    return (int8_t)(neg ? -d : d);
}

// digit planes are stored as int8 (the public slicer) or as exact fp16 values (the
// operand planes of the tensor-core engine)
template <typename T>
__device__ __forceinline__ T digit_out(int8_t d);
template <>
__device__ __forceinline__ int8_t digit_out<int8_t>(int8_t d) {
    return d;
}
template <>
__device__ __forceinline__ __half digit_out<__half>(int8_t d) {
    return __int2half_rn((int)d);
}

// One CTA per row, 8 consecutive columns per thread: pass 1 reduces the row's max |x|
// (fp32 bits), pass 2 re-reads the row (cache resident) and writes each plane's eight
// digits with one store (when the plane's row stride allows it).
template <typename T>
__global__ void __launch_bounds__(SROW_THREADS) slice_rows_kernel(const float* __restrict__ X, int64_t ldx, int rows,
                                                                  int cols, int nslices, T* __restrict__ S,
                                                                  int64_t lds, int32_t* __restrict__ e_out) {
    __shared__ uint32_t red[SROW_THREADS / 32];
    const int64_t row = blockIdx.x;
    const uint32_t* x = reinterpret_cast<const uint32_t*>(X + row * ldx);
    const bool vec_in = (ldx % 4) == 0 && (reinterpret_cast<uintptr_t>(X) & 15u) == 0;
    auto load8 = [&](int j0, uint32_t (&v)[8]) {
        if (vec_in && j0 + 8 <= cols) {
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(x + j0));
            const uint4 b = __ldg(reinterpret_cast<const uint4*>(x + j0 + 4));
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = j0 + i < cols ? x[j0 + i] : 0u;
        }
    };
    uint32_t amax = 0;
    for (int j0 = threadIdx.x * 8; j0 < cols; j0 += SROW_THREADS * 8) {
        uint32_t v[8];
        load8(j0, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = max(amax, v[i] & 0x7FFFFFFFu);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < SROW_THREADS / 32; ++w) amax = max(amax, red[w]);
    const int64_t plane = (int64_t)rows * lds;
    T* srow = S + row * lds;
    const bool bad = amax >= 0x7F800000u;  // inf or NaN in the row: digits written as zero
    const int e = bad ? 0 : line_exponent(amax);
    if (threadIdx.x == 0) {
        if (bad) raise_status(DEV_NONFINITE);
        e_out[row] = e;
    }
    const bool vec_out = (lds % 8) == 0 && (reinterpret_cast<uintptr_t>(S) & 15u) == 0;
    for (int j0 = threadIdx.x * 8; j0 < lds; j0 += SROW_THREADS * 8) {
        uint32_t v[8];
        load8(j0, v);  // zero beyond cols: the padding up to lds gets zero digits
        unsigned long long R[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) R[i] = bad ? 0ull : digits_of(v[i], e, nslices);
        for (int t = 0; t < nslices; ++t) {
            int8_t d[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) d[i] = digit(R[i], t, nslices, v[i] >> 31);
            T* dst = srow + t * plane + j0;
            if (vec_out) {
                *reinterpret_cast<typename Pack8<T>::type*>(dst) = Pack8<T>::make(d);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (j0 + i < lds) dst[i] = digit_out<T>(d[i]);
            }
        }
    }
}

// column max of |x| bits: block (32 columns) x (8 row lanes), one chunk of rows per blockIdx.y
constexpr int CM_ROWS = 256;

__global__ void col_absmax_kernel(const float* __restrict__ X, int64_t ldx, int rows, int cols,
                                  uint32_t* __restrict__ colmax) {
    __shared__ uint32_t red[8][32];
    const int j = blockIdx.x * 32 + threadIdx.x;
    const int r0 = blockIdx.y * CM_ROWS;
    const int r1 = min(rows, r0 + CM_ROWS);
    uint32_t m = 0;
    if (j < cols) {
        const uint32_t* x = reinterpret_cast<const uint32_t*>(X);
        for (int r = r0 + threadIdx.y; r < r1; r += 8) m = max(m, x[(int64_t)r * ldx + j] & 0x7FFFFFFFu);
    }
    red[threadIdx.y][threadIdx.x] = m;
    __syncthreads();
    if (threadIdx.y == 0 && j < cols) {
#pragma unroll
        for (int y = 1; y < 8; ++y) m = max(m, red[y][threadIdx.x]);
        atomicMax(colmax + j, m);
    }
}

// colmax bits -> exponents (in place into e_out), non-finite columns flagged
__global__ void col_exponent_kernel(const uint32_t* colmax, int cols, int32_t* e_out) {  // colmax aliases e_out
    int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= cols) return;
    uint32_t m = colmax[j];
    if (m >= 0x7F800000u) {
        raise_status(DEV_NONFINITE);
        e_out[j] = INT32_MIN;  // marks the column: its digits are written as zero
        return;
    }
    e_out[j] = line_exponent(m);
}

// 64 x 64 tile of X (rows r0.., columns c0..), 256 threads: each thread loads four
// columns of four rows (16-byte loads), its digits go to a shared tile [t][col][row],
// then each plane is written K-major, S[t][col][row], eight rows per store (each
// column's 64 rows are 128 contiguous bytes of fp16).
constexpr int SC_TILE = 64;
constexpr int SC_PITCH = SC_TILE + 4;  // bytes per (t, col) line of the shared tile

template <typename T>
__global__ void __launch_bounds__(256) slice_cols_kernel(const float* __restrict__ X, int64_t ldx, int rows, int cols,
                                                         int nslices, const int32_t* __restrict__ e_col,
                                                         T* __restrict__ S, int64_t lds) {
    __shared__ __align__(16) int8_t tile[9][SC_TILE][SC_PITCH];
    const int r0 = blockIdx.y * SC_TILE, c0 = blockIdx.x * SC_TILE;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 column quads x 16 row lanes
    const bool vec_in = (ldx % 4) == 0 && (reinterpret_cast<uintptr_t>(X) & 15u) == 0;
    const int cq = c0 + 4 * tx;
    int ecol[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) ecol[q] = cq + q < cols ? e_col[cq + q] : INT32_MIN;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int rr = ty + 16 * i, r = r0 + rr;
        uint32_t v[4] = {0u, 0u, 0u, 0u};
        if (r < rows) {
            const uint32_t* xr = reinterpret_cast<const uint32_t*>(X) + (int64_t)r * ldx;
            if (vec_in && cq + 4 <= cols) {
                const uint4 a = __ldg(reinterpret_cast<const uint4*>(xr + cq));
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) v[q] = cq + q < cols ? xr[cq + q] : 0u;
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // a column marked non-finite (INT32_MIN) or outside the matrix gets zero digits
            const unsigned long long R = ecol[q] == INT32_MIN ? 0ull : digits_of(v[q], ecol[q], nslices);
            for (int t = 0; t < nslices; ++t) tile[t][4 * tx + q][rr] = digit(R, t, nslices, v[q] >> 31);
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
        const uint32_t* src = reinterpret_cast<const uint32_t*>(&tile[t][cc][8 * g8]);
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

__global__ void fix_nonfinite_cols_kernel(int32_t* e_out, int cols) {
    int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j < cols && e_out[j] == INT32_MIN) e_out[j] = 0;
}

template <typename T>
cudaError_t rows_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, T* S, int64_t lds, int32_t* e,
                        cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    slice_rows_kernel<T><<<rows, SROW_THREADS, 0, s>>>(X, ldx, rows, cols, nslices, S, lds, e);
    return cudaGetLastError();
}

template <typename T>
cudaError_t cols_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, T* S, int64_t lds, int32_t* e,
                        cudaStream_t s) {
    if (cols == 0) return cudaSuccess;
    uint32_t* colmax = reinterpret_cast<uint32_t*>(e);  // reused: max bits, then exponents
    cudaError_t err = cudaMemsetAsync(colmax, 0, (size_t)cols * sizeof(uint32_t), s);
    if (err != cudaSuccess) return err;
    if (rows > 0) {
        dim3 g1((cols + 31) / 32, (rows + CM_ROWS - 1) / CM_ROWS);
        col_absmax_kernel<<<g1, dim3(32, 8), 0, s>>>(X, ldx, rows, cols, colmax);
    }
    col_exponent_kernel<<<(cols + 255) / 256, 256, 0, s>>>(colmax, cols, e);
    dim3 g2((cols + SC_TILE - 1) / SC_TILE, (int)((lds + SC_TILE - 1) / SC_TILE));
    if (lds > 0) slice_cols_kernel<T><<<g2, 256, 0, s>>>(X, ldx, rows, cols, nslices, e, S, lds);
    fix_nonfinite_cols_kernel<<<(cols + 255) / 256, 256, 0, s>>>(e, cols);
    return cudaGetLastError();
}

}  // namespace

cudaError_t slice_rows_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, int8_t* S, int64_t lds,
                              int32_t* e, cudaStream_t s) {
    return rows_launch<int8_t>(X, ldx, rows, cols, nslices, S, lds, e, s);
}

cudaError_t slice_cols_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, int8_t* S, int64_t lds,
                              int32_t* e, cudaStream_t s) {
    return cols_launch<int8_t>(X, ldx, rows, cols, nslices, S, lds, e, s);
}

cudaError_t slice_rows_f16_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, void* S, int64_t lds,
                                  int32_t* e, cudaStream_t s) {
    return rows_launch<__half>(X, ldx, rows, cols, nslices, reinterpret_cast<__half*>(S), lds, e, s);
}

cudaError_t slice_cols_f16_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, void* S, int64_t lds,
                                  int32_t* e, cudaStream_t s) {
    return cols_launch<__half>(X, ldx, rows, cols, nslices, reinterpret_cast<__half*>(S), lds, e, s);
}

DETGEMM_STATUS_ACCESSOR(slice_take_status)

}  // namespace detgemm
