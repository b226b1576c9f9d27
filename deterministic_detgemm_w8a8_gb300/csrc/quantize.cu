// Power-of-two row quantizer — "Deterministic LLM Inference Across GPU Kernels:
// Power-of-Two INT8 Quantization Scales ...", §V (scales requantized to a power of two
// and the int8 values requantized under it) and §V.C (nearest arm vs ceiling arm).
//
// Per row: a = max|x|, s = a/127; CEIL picks the smallest e with 2^e >= s, NEAREST the
// integer nearest to log2(s); q = clamp(rne(x * 2^-e), -127, 127). Everything after the
// load is integer arithmetic on the fp32 bit pattern, so the exponent choice and every
// rounding are exact (no division, no log, no scaled intermediate).
//
// One CTA per row, eight columns per thread: pass 1 reduces the row's largest |x| as
// fp32 bits (for non-negative floats the bit order is the value order), pass 2 re-reads
// the row (L1/L2 resident) and writes int8 — or, for the fused linear layer, the same
// integers as exact fp16 values. HBM traffic per element: read 2 B (bf16) or 4 B (fp32),
// write 1 B (int8) or 2 B (fp16).
#include <cuda_fp16.h>
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

// Eight consecutive inputs as fp32 bit patterns (zero beyond cols): one 16-byte load of
// bf16 or two of fp32 when the row allows it.
template <int DT>
__device__ __forceinline__ void load8_bits(const void* X, int64_t xoff, int j0, int cols, bool vec, uint32_t (&v)[8]) {
    if (vec && j0 + 8 <= cols) {
        if (DT == DETGEMM_DTYPE_BF16) {
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(X) + xoff + j0));
            const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = w[i] << 16;
                v[2 * i + 1] = w[i] & 0xFFFF0000u;
            }
        } else {
            const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const uint32_t*>(X) + xoff + j0);
            const uint4 a = __ldg(p), b = __ldg(p + 1);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = j0 + i < cols ? load_bits<DT>(X, xoff + j0 + i) : 0u;
    }
}

// One CTA per row, eight columns per thread. The values are written as int8 (the public
// quantizer) or as exact fp16 values with zeros up to the padded row length qcols (the
// activation operand of the tensor-core GEMM, written directly in its carrier format).
template <int DT, typename OutT>
__global__ void __launch_bounds__(QTHREADS) quantize_pow2_kernel(const void* __restrict__ X, int64_t ldx, int cols,
                                                                  int mode, OutT* __restrict__ Q, int64_t ldq,
                                                                  int qcols, int32_t* __restrict__ e_out) {
    __shared__ uint32_t red[QTHREADS / 32];
    const int64_t row = blockIdx.x;
    const int64_t xoff = row * ldx;
    const int xs = DT == DETGEMM_DTYPE_BF16 ? 2 : 4;
    const bool vec_in = ((ldx * xs) % 16) == 0 && (reinterpret_cast<uintptr_t>(X) & 15u) == 0;
    uint32_t amax = 0;
    for (int j0 = threadIdx.x * 8; j0 < cols; j0 += QTHREADS * 8) {
        uint32_t v[8];
        load8_bits<DT>(X, xoff, j0, cols, vec_in, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = max(amax, v[i] & 0x7FFFFFFFu);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < QTHREADS / 32; ++w) amax = max(amax, red[w]);

    // inf or NaN somewhere in the row: e = 0 and zeros
    const bool bad = amax >= 0x7F800000u;
    const int e = bad ? 0 : pow2_exponent(amax, mode);
    if (threadIdx.x == 0) {
        if (bad) raise_status(DEV_NONFINITE);
        e_out[row] = e;
    }
    OutT* q = Q + row * ldq;
    const bool vec_out = (ldq % 8) == 0 && (reinterpret_cast<uintptr_t>(Q) & 15u) == 0;
    for (int j0 = threadIdx.x * 8; j0 < qcols; j0 += QTHREADS * 8) {
        uint32_t v[8];
        load8_bits<DT>(X, xoff, j0, cols, vec_in, v);
        int8_t d[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) d[i] = bad ? (int8_t)0 : quantize_one(v[i], e);
        if (vec_out && j0 + 8 <= qcols) {
            *reinterpret_cast<typename Pack8<OutT>::type*>(q + j0) = Pack8<OutT>::make(d);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (j0 + i < qcols) q[j0 + i] = Pack8<OutT>::one(d[i]);
        }
    }
}

template <typename OutT>
cudaError_t launch(const void* X, int x_dtype, int64_t ldx, int rows, int cols, int mode, OutT* Q, int64_t ldq,
                   int qcols, int32_t* e, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    if (x_dtype == DETGEMM_DTYPE_BF16)
        quantize_pow2_kernel<DETGEMM_DTYPE_BF16, OutT><<<rows, QTHREADS, 0, s>>>(X, ldx, cols, mode, Q, ldq, qcols, e);
    else
        quantize_pow2_kernel<DETGEMM_DTYPE_F32, OutT><<<rows, QTHREADS, 0, s>>>(X, ldx, cols, mode, Q, ldq, qcols, e);
    return cudaGetLastError();
}

}  // namespace

cudaError_t quantize_pow2_launch(const void* X, int x_dtype, int64_t ldx, int rows, int cols, int mode, int8_t* Q,
                                 int64_t ldq, int32_t* e, cudaStream_t s) {
    return launch<int8_t>(X, x_dtype, ldx, rows, cols, mode, Q, ldq, cols, e, s);
}

cudaError_t quantize_pow2_f16_launch(const void* X, int x_dtype, int64_t ldx, int rows, int cols, int mode, void* Q16,
                                     int64_t ldq, int32_t* e, cudaStream_t s) {
    return launch<__half>(X, x_dtype, ldx, rows, cols, mode, reinterpret_cast<__half*>(Q16), ldq, (int)ldq, e, s);
}

DETGEMM_STATUS_ACCESSOR(quantize_take_status)

}  // namespace detgemm
