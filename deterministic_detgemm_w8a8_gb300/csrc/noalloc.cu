// detgemm_w8a8_noalloc: the W8A8 GEMM for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a scratch buffer: a plugin inside an
// inference server that is given only its input and output tensors, or a serving loop
// that forbids cudaMalloc on its hot path because an allocation can synchronize the
// whole device and stall other streams. For them this entry point keeps its split-K
// scratch in a fixed array compiled into the library (DETGEMM_NOALLOC_SCRATCH_BYTES),
// which every GPU that loads the library holds until the process exits.
//
// Problems of at most 64 rows run on the decode kernels (the same as detgemm_w8a8); larger
// ones on the int8 warp-MMA tile kernel (mma.sync m16n8k32, exact int32 accumulation, about
// 147 TOPS on the FFN down GEMM), not on the tcgen05 engine, whose fp16 operand copies would
// need tens of MB of scratch: same bits, far lower throughput at large M.
//
// The array's name is only a host-side stand-in in host code, so its device address is
// fetched once per device with cudaGetSymbolAddress (with that device current) and
// cached; the first call on each device does that set-up. Every call clears the part of
// the array it uses before its kernel runs; calls that overlap on the GPU share the
// array and therefore race. Nothing here allocates: no cudaMalloc, cudaFree or
// allocating library routine is called.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/detgemm.h"
#include "common.cuh"
#include "internal.h"

namespace detgemm {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[DETGEMM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDev];  // device address of the array, per device
int g_noalloc_cc[kMaxDev];     // compute capability, per device

// Device address of the scratch array on the current device (set up on first use).
detgemm_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return DETGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_cc[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return DETGEMM_ERR_UNSUPPORTED_DEVICE;
        g_noalloc_cc[dev] = 10 * major + minor;
    }
    if (g_noalloc_cc[dev] != 103) return DETGEMM_ERR_UNSUPPORTED_DEVICE;
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return DETGEMM_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return DETGEMM_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace detgemm

using namespace detgemm;

extern "C" DETGEMM_API size_t detgemm_w8a8_noalloc_scratch_size(int M, int N, int K, int split_k) {
    if (M <= 0 || N <= 0 || K <= 0 || split_k < 1) return 0;
    return igemm_workspace_bytes(M, N, K, split_k);
}

extern "C" DETGEMM_API detgemm_status detgemm_w8a8_noalloc(const int8_t* A, int64_t lda, const int8_t* W,
                                                            int64_t ldw, const int32_t* ea, const int32_t* ew,
                                                            uint16_t* C, int64_t ldc, int M, int N, int K,
                                                            int split_k, detgemm_stream_t stream) {
    // the checks of detgemm_w8a8, in its order; the scratch-size refusal comes last
    if (M < 0 || N < 0 || K < 1) return DETGEMM_ERR_INVALID_ARG;
    if (K > DETGEMM_MAX_K) return DETGEMM_ERR_PRECONDITION;
    if (split_k < 1 || split_k > (K + 63) / 64) return DETGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DETGEMM_OK;
    if (!A || !W || !C) return DETGEMM_ERR_INVALID_ARG;
    if (lda < K || ldw < K || ldc < N) return DETGEMM_ERR_INVALID_ARG;
    if (!al16(A) || !al16(W) || !al16(C)) return DETGEMM_ERR_ALIGNMENT;
    if ((lda % 16) != 0 || (ldw % 16) != 0 || ((ldc * 2) % 16) != 0) return DETGEMM_ERR_ALIGNMENT;
    if (!ea || !ew) return DETGEMM_ERR_INVALID_ARG;
    if (!al4(ea) || !al4(ew)) return DETGEMM_ERR_ALIGNMENT;
    void* scratch = nullptr;
    detgemm_status st = noalloc_scratch(&scratch);  // the device check, then the array's address
    if (st != DETGEMM_OK) return st;
    if (detgemm_w8a8_noalloc_scratch_size(M, N, K, split_k) > (size_t)DETGEMM_NOALLOC_SCRATCH_BYTES)
        return DETGEMM_ERR_WORKSPACE;  // the problem needs more scratch than the fixed array holds
    IGemmArgs a = {};
    a.seg[0] = Seg{A, W};
    a.nseg = 1;
    a.lda = lda;
    a.ldw = ldw;
    a.M = M;
    a.N = N;
    a.K = K;
    a.split = split_k;
    a.mode = EPI_BF16_POW2;
    a.ea = ea;
    a.ew = ew;
    a.C = C;
    a.ldc = ldc;
    return igemm_launch(a, scratch, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? DETGEMM_OK
                                                                                            : DETGEMM_ERR_CUDA;
}
