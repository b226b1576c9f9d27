// Ozaki recombination — "GPU Mechanism", §3 "Method", Interventions (a) ExactGEMM:
// the exact diagonal sums are recombined in a fixed order in fp64 and rounded once.
//
//   acc = 0.0;  for g = max_diag .. 2:  acc = acc + T_g * 2^(-7g);
//   C_ij = fp32_rne(acc * 2^(e_i + f_j)).
//
// One thread per output element; T is [max_diag - 1][M][ldT] int32, plane d holding the
// diagonal g = max_diag - d. The
// loads of each plane are coalesced along N. Traffic per element: 4 (max_diag - 1) B
// read + 4 B written; fp64 work: max_diag - 1 multiply-adds, issued as separate
// round-to-nearest multiply and add (the multiply by a power of two is exact).
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace detgemm {

namespace {

__global__ void ozaki_combine_kernel(const int32_t* __restrict__ T, int64_t ldT, int max_diag,
                                     const int32_t* __restrict__ e, const int32_t* __restrict__ f,
                                     float* __restrict__ C, int64_t ldc, int M, int N) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    const int i = blockIdx.y;
    if (j >= N) return;
    const int64_t plane = (int64_t)M * ldT;
    const int64_t idx = (int64_t)i * ldT + j;
    int32_t t[19];
#pragma unroll
    for (int g = 0; g < 19; ++g) t[g] = 0;
    for (int g = 2; g <= max_diag; ++g) t[g] = __ldg(T + (int64_t)(max_diag - g) * plane + idx);
    C[(int64_t)i * ldc + j] = ozaki_combine(t, max_diag, e[i], f[j]);
}

}  // namespace

cudaError_t ozaki_combine_launch(const int32_t* T, int64_t ldT, int max_diag, const int32_t* e, const int32_t* f,
                                 float* C, int64_t ldc, int M, int N, cudaStream_t s) {
    if (M == 0 || N == 0) return cudaSuccess;
    dim3 grid((N + 255) / 256, M);
    ozaki_combine_kernel<<<grid, 256, 0, s>>>(T, ldT, max_diag, e, f, C, ldc, M, N);
    return cudaGetLastError();
}

}  // namespace detgemm
