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
// Rows: one CTA per row, two passes (max, then digits). Columns: a column-max kernel
// (atomicMax over row chunks), an exponent kernel, then a 32x32 tiled transpose that
// writes every digit plane K-major ([t][col][row]).
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

template <typename T>
__global__ void __launch_bounds__(SROW_THREADS) slice_rows_kernel(const float* __restrict__ X, int64_t ldx, int rows,
                                                                  int cols, int nslices, T* __restrict__ S,
                                                                  int64_t lds, int32_t* __restrict__ e_out) {
    __shared__ uint32_t red[SROW_THREADS / 32];
    const int64_t row = blockIdx.x;
    const uint32_t* x = reinterpret_cast<const uint32_t*>(X + row * ldx);
    uint32_t amax = 0;
    for (int j = threadIdx.x; j < cols; j += SROW_THREADS) amax = max(amax, x[j] & 0x7FFFFFFFu);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < SROW_THREADS / 32; ++w) amax = max(amax, red[w]);
    const int64_t plane = (int64_t)rows * lds;
    T* s = S + row * lds;
    const bool bad = amax >= 0x7F800000u;  // inf or NaN in the row: digits written as zero
    const int e = bad ? 0 : line_exponent(amax);
    if (threadIdx.x == 0) {
        if (bad) raise_status(DEV_NONFINITE);
        e_out[row] = e;
    }
    for (int j = threadIdx.x; j < lds; j += SROW_THREADS) {
        uint32_t xb = (j < cols && !bad) ? x[j] : 0u;
        unsigned long long R = digits_of(xb, e, nslices);
        bool neg = xb >> 31;
        for (int t = 0; t < nslices; ++t) s[t * plane + j] = digit_out<T>(digit(R, t, nslices, neg));
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

// 32 x 32 tile: rows r0.., columns c0..; digits written to S[t][col][row]
template <typename T>
__global__ void slice_cols_kernel(const float* __restrict__ X, int64_t ldx, int rows, int cols, int nslices,
                                  const int32_t* __restrict__ e_col, T* __restrict__ S, int64_t lds) {
    __shared__ int8_t tile[9][32][33];
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
    for (int yy = ty; yy < 32; yy += 8) {
        int r = r0 + yy, c = c0 + tx;
        unsigned long long R = 0;
        bool neg = false;
        if (r < rows && c < cols) {
            uint32_t xb = reinterpret_cast<const uint32_t*>(X)[(int64_t)r * ldx + c];
            int e = e_col[c];
            if (e != INT32_MIN) {
                R = digits_of(xb, e, nslices);
                neg = xb >> 31;
            }
        }
        for (int t = 0; t < nslices; ++t) tile[t][tx][yy] = digit(R, t, nslices, neg);
    }
    __syncthreads();
    const int64_t plane = (int64_t)cols * lds;
    for (int yy = ty; yy < 32; yy += 8) {
        int c = c0 + yy, r = r0 + tx;
        if (c < cols && r < lds)  // rows in [rows, lds) are the zero padding
            for (int t = 0; t < nslices; ++t) S[t * plane + (int64_t)c * lds + r] = digit_out<T>(tile[t][yy][tx]);
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
    dim3 g2((cols + 31) / 32, (int)((lds + 31) / 32));
    if (lds > 0) slice_cols_kernel<T><<<g2, dim3(32, 8), 0, s>>>(X, ldx, rows, cols, nslices, e, S, lds);
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
