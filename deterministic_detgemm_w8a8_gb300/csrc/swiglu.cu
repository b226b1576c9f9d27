// Gated-linear-unit epilogue on exact accumulators: C = rne_bf16(SiLU(G * 2^(ea+ewg)) *
// U * 2^(ea+ewu)), element by element, rounded once (bf16_silu_mul in silu.cuh). The fused
// W8A8 form runs the same function in the tensor-core engine's epilogue.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/detgemm.h"
#include "common.cuh"
#include "internal.h"
#include "silu.cuh"

namespace detgemm {
namespace {

struct SwArgs {
    const int32_t* G;
    int64_t ldg;
    const int32_t* U;
    int64_t ldu;
    const int32_t* ea;
    const int32_t* ewg;
    const int32_t* ewu;
    uint16_t* C;
    int64_t ldc;
    int M, N;
};

__global__ void swiglu_epilogue_kernel(const SwArgs p) {
    const int64_t total = (int64_t)p.M * p.N;
    bool bad = false;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(idx / p.N), j = (int)(idx - (int64_t)i * p.N);
        const long long ea = p.ea[i];
        p.C[(int64_t)i * p.ldc + j] =
            bf16_silu_mul(p.G[(int64_t)i * p.ldg + j], p.U[(int64_t)i * p.ldu + j], ea + p.ewg[j], ea + p.ewu[j], bad);
    }
    if (bad) raise_status(DEV_RANGE);
}

}  // namespace

cudaError_t swiglu_epilogue_launch(const int32_t* G, int64_t ldg, const int32_t* U, int64_t ldu, const int32_t* ea,
                                   const int32_t* ewg, const int32_t* ewu, uint16_t* C, int64_t ldc, int M, int N,
                                   cudaStream_t s) {
    SwArgs a = {G, ldg, U, ldu, ea, ewg, ewu, C, ldc, M, N};
    const int64_t total = (int64_t)M * N;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    swiglu_epilogue_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

DETGEMM_STATUS_ACCESSOR(swiglu_take_status)

}  // namespace detgemm
