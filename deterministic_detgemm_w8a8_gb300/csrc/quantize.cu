// Power-of-two row quantizer — "Deterministic LLM Inference Across GPU Kernels:
// Power-of-Two INT8 Quantization Scales ...", §V (scales requantized to a power of two
// and the int8 values requantized under it) and §V.C (nearest arm vs ceiling arm).
//
// Per row: a = max|x|, s = a/127; CEIL picks the smallest e with 2^e >= s, NEAREST the
// integer nearest to log2(s); q = clamp(rne(x * 2^-e), -127, 127). Everything after the
// load is integer arithmetic on the fp32 bit pattern, so the exponent choice and every
// rounding are exact (no division, no log, no scaled intermediate).
//
// One CTA per row: pass 1 reduces the row's largest |x| as fp32 bits (for non-negative
// floats the bit order is the value order), pass 2 re-reads the row (L1/L2 resident)
// and writes int8. HBM traffic per element: read 2 B (bf16) or 4 B (fp32), write 1 B.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace detgemm {

namespace {

constexpr int QTHREADS = 256;

template <int DT>
__device__ __forceinline__ uint32_t load_bits(const void* X, int64_t idx) {
    if (DT == DETGEMM_DTYPE_BF16) return (uint32_t)(reinterpret_cast<const uint16_t*>(X)[idx]) << 16;
    return reinterpret_cast<const uint32_t*>(X)[idx];
}

// Exponent of the power-of-two scale from the row's max |x| (fp32 bits, finite, > 0).
// With a = M 2^(p-23), M in [2^23, 2^24):
//   127 * 2^(p-6) = 1.984375 * 2^p, so a <= 127 * 2^(p-6)  <=>  M <= 127 * 2^17,
//   hence ceil exponent ec = p - 6 or p - 5;
//   nearest keeps ec iff a^2 >= 127^2 * 2^(2 ec - 1)  <=>  M^2 >= 16129 * 2^(2 (ec - p) + 45).
__device__ __forceinline__ int pow2_exponent(uint32_t amax, int mode) {
    uint32_t M;
    int p;
    if (!f32_normalise(amax, M, p)) return 0;
    int ec = (M <= (127u << 17)) ? p - 6 : p - 5;
    if (mode == DETGEMM_POW2_NEAREST) {
        int d = ec - p;
        unsigned long long lhs = (unsigned long long)M * M;
        unsigned long long rhs = 16129ull << (2 * d + 45);
        if (lhs < rhs) ec -= 1;
    }
    return ec;
}

// clamp(rne(x * 2^-e), -127, 127) from the fp32 bits of x.
__device__ __forceinline__ int8_t quantize_one(uint32_t xb, int e) {
    uint32_t M;
    int p;
    if (!f32_normalise(xb & 0x7FFFFFFFu, M, p)) return 0;
    int sh = p - 23 - e;  // |x| 2^-e = M 2^sh
    int q;
    if (sh >= 0) {
        q = 127;  // >= 2^23
    } else {
        int r = -sh;
        if (r >= 25) {
            q = 0;  // < 2^24 / 2^25 = 1/2
        } else {
            uint32_t qq = M >> r;
            uint32_t rem = M & ((1u << r) - 1u);
            uint32_t half = 1u << (r - 1);
            if (rem > half || (rem == half && (qq & 1u))) qq += 1;
            q = qq > 127u ? 127 : (int)qq;
        }
    }
    return (int8_t)((xb >> 31) ? -q : q);
}

template <int DT>
__global__ void __launch_bounds__(QTHREADS) quantize_pow2_kernel(const void* __restrict__ X, int64_t ldx, int cols,
                                                                  int mode, int8_t* __restrict__ Q, int64_t ldq,
                                                                  int32_t* __restrict__ e_out) {
    __shared__ uint32_t red[QTHREADS / 32];
    const int64_t row = blockIdx.x;
    const int64_t xoff = row * ldx;
    uint32_t amax = 0;
    for (int j = threadIdx.x; j < cols; j += QTHREADS) amax = max(amax, load_bits<DT>(X, xoff + j) & 0x7FFFFFFFu);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < QTHREADS / 32; ++w) amax = max(amax, red[w]);

    int8_t* q = Q + row * ldq;
    if (amax >= 0x7F800000u) {  // inf or NaN somewhere in the row
        if (threadIdx.x == 0) {
            raise_status(DEV_NONFINITE);
            e_out[row] = 0;
        }
        for (int j = threadIdx.x; j < cols; j += QTHREADS) q[j] = 0;
        return;
    }
    const int e = pow2_exponent(amax, mode);
    if (threadIdx.x == 0) e_out[row] = e;
    for (int j = threadIdx.x; j < cols; j += QTHREADS) q[j] = quantize_one(load_bits<DT>(X, xoff + j), e);
}

}  // namespace

cudaError_t quantize_pow2_launch(const void* X, int x_dtype, int64_t ldx, int rows, int cols, int mode, int8_t* Q,
                                 int64_t ldq, int32_t* e, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    if (x_dtype == DETGEMM_DTYPE_BF16)
        quantize_pow2_kernel<DETGEMM_DTYPE_BF16><<<rows, QTHREADS, 0, s>>>(X, ldx, cols, mode, Q, ldq, e);
    else
        quantize_pow2_kernel<DETGEMM_DTYPE_F32><<<rows, QTHREADS, 0, s>>>(X, ldx, cols, mode, Q, ldq, e);
    return cudaGetLastError();
}

DETGEMM_STATUS_ACCESSOR(quantize_take_status)

}  // namespace detgemm
