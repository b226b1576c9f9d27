// Exact int8 -> fp16 widening of GEMM operands, zero-filling K up to the padded row length.
//
// The tensor-core W8A8 path carries int8 values in fp16 (every integer in [-2048, 2048]
// is an fp16 value, so the copy is exact); these kernels write that fp16 copy. The
// conversion is done with byte permutes: b + 128 (the byte with its top bit flipped) is
// placed as the mantissa under the fp16 exponent of 1024, which gives 1024 + b + 128
// exactly, and 1152 is subtracted in fp16 (exact, since the result is an integer of
// magnitude <= 128).
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"

namespace detgemm {

namespace {

__device__ __forceinline__ void widen4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t x = w ^ 0x80808080u;
    const uint32_t l = __byte_perm(x, 0x64646464u, 0x4140);
    const uint32_t h = __byte_perm(x, 0x64646464u, 0x4342);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const __half2 rl = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
    const __half2 rh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
    lo = *reinterpret_cast<const uint32_t*>(&rl);
    hi = *reinterpret_cast<const uint32_t*>(&rh);
}

struct WidenPair {
    const int8_t* X[2];
    int64_t ldx[2];
    int rows[2];
    int K[2];
    __half* Y[2];
    int64_t Kp[2];  // multiples of 16
};

// Both operands of a GEMM in one launch (the second may have zero rows): each thread step
// loads two 16-byte groups of int8 (one grid stride apart) before converting and storing
// 2 x 32 bytes of fp16, which keeps enough reads in flight at 3 blocks per SM. The loads
// bypass L1; the stores are plain so that the GEMM that follows finds the most recently
// written part of its operands in L2.
__device__ __forceinline__ uint4* widen_locate(const WidenPair& p, int64_t nv0, int64_t v, const int8_t*& x, int& kk,
                                               int& m) {
    m = v < nv0 ? 0 : 1;
    const int64_t vm = m == 0 ? v : v - nv0;
    const int64_t nvec = p.Kp[m] / 16;
    const int64_t r = vm / nvec;
    kk = (int)((vm - r * nvec) * 16);
    x = p.X[m] + r * p.ldx[m] + kk;
    return reinterpret_cast<uint4*>(p.Y[m] + r * p.Kp[m] + kk);
}

__device__ __forceinline__ uint4 widen_load16(const int8_t* x, int k, int K) {
    uint4 w;
    if (k + 16 <= K) {
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                     : "l"(x));
    } else {
        uint64_t lo = 0, hi = 0;
        for (int i = 0; i < 16 && k + i < K; ++i) {
            const uint64_t b = (uint64_t)(uint8_t)x[i] << (8 * (i & 7));
            if (i < 8) lo |= b; else hi |= b;
        }
        w = make_uint4((uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32));
    }
    return w;
}

__device__ __forceinline__ void widen_store32(uint4* y, uint4 w) {
    uint4 o0, o1;
    widen4(w.x, o0.x, o0.y);
    widen4(w.y, o0.z, o0.w);
    widen4(w.z, o1.x, o1.y);
    widen4(w.w, o1.z, o1.w);
    y[0] = o0;
    y[1] = o1;
}

// Both kernels are launched as programmatic dependents of the kernel before them on the
// stream: they wait for its completion (which may have produced X) before reading, then let
// the next kernel (the GEMM, which waits for them in turn) be scheduled at once: its blocks
// need an SM's shared memory, so they start as these blocks leave, with their setup done
// by the time the widened operands are complete.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__global__ void __launch_bounds__(256) widen_pair_kernel(const __grid_constant__ WidenPair p) {
    pdl_enter();
    const int64_t nv0 = (int64_t)p.rows[0] * (p.Kp[0] / 16);
    const int64_t total = nv0 + (int64_t)p.rows[1] * (p.Kp[1] / 16);
    const int64_t nt = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += 2 * nt) {
        const int8_t *x0, *x1;
        int k0, k1, m0, m1;
        uint4* y0 = widen_locate(p, nv0, v, x0, k0, m0);
        const uint4 w0 = widen_load16(x0, k0, p.K[m0]);
        const bool two = v + nt < total;
        uint4* y1 = nullptr;
        uint4 w1 = make_uint4(0, 0, 0, 0);
        if (two) {
            y1 = widen_locate(p, nv0, v + nt, x1, k1, m1);
            w1 = widen_load16(x1, k1, p.K[m1]);
        }
        widen_store32(y0, w0);
        if (two) widen_store32(y1, w1);
    }
}

// One matrix whose output row stride is a multiple of 8 (not of 16): 8 int8 per step.
__global__ void __launch_bounds__(256) widen8_kernel(const int8_t* __restrict__ X, int64_t ldx, int rows, int K,
                                                     __half* __restrict__ Y, int64_t Kp) {
    pdl_enter();
    const int64_t nvec = Kp / 8;
    const int64_t total = (int64_t)rows * nvec;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = v / nvec;
        const int k = (int)((v - r * nvec) * 8);
        const int8_t* x = X + r * ldx + k;
        uint2 w;
        if (k + 8 <= K) {
            w = *reinterpret_cast<const uint2*>(x);
        } else {
            uint64_t t = 0;
            for (int i = 0; i < 8 && k + i < K; ++i) t |= (uint64_t)(uint8_t)x[i] << (8 * i);
            w = make_uint2((uint32_t)t, (uint32_t)(t >> 32));
        }
        uint4 o;
        widen4(w.x, o.x, o.y);
        widen4(w.y, o.z, o.w);
        *reinterpret_cast<uint4*>(Y + r * Kp + k) = o;
    }
}

std::mutex g_widen_mutex;
int g_widen_sms[64];

int widen_num_sms() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(g_widen_mutex);
    if (g_widen_sms[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_widen_sms[dev] = n > 0 ? n : 148;
    }
    return g_widen_sms[dev];
}

// 256-thread launch with the programmatic-stream-serialization attribute
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), unsigned blocks, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

unsigned widen_blocks(int64_t total, int per_sm) {
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)widen_num_sms() * per_sm;
    return (unsigned)(blocks > cap ? cap : blocks);
}

}  // namespace

cudaError_t widen_pair_launch(const int8_t* X0, int64_t ldx0, int rows0, int K0, void* Y0, int64_t Kp0,
                              const int8_t* X1, int64_t ldx1, int rows1, int K1, void* Y1, int64_t Kp1,
                              cudaStream_t s) {
    WidenPair p;
    p.X[0] = X0; p.ldx[0] = ldx0; p.rows[0] = rows0; p.K[0] = K0; p.Y[0] = reinterpret_cast<__half*>(Y0); p.Kp[0] = Kp0;
    p.X[1] = X1; p.ldx[1] = ldx1; p.rows[1] = rows1; p.K[1] = K1; p.Y[1] = reinterpret_cast<__half*>(Y1); p.Kp[1] = Kp1;
    const int64_t total = (int64_t)rows0 * (Kp0 / 16) + (int64_t)rows1 * (Kp1 / 16);
    if (total == 0) return cudaSuccess;
    // 3 blocks per SM measured fastest (2, 4, 6, 8 slower)
    return launch_dependent(widen_pair_kernel, widen_blocks(total, 3), s, p);
}

cudaError_t widen_i8_f16_launch(const int8_t* X, int64_t ldx, int rows, int K, void* Y, int64_t Kp, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    if (Kp % 16 == 0) return widen_pair_launch(X, ldx, rows, K, Y, Kp, nullptr, 0, 0, 0, nullptr, 0, s);
    return launch_dependent(widen8_kernel, widen_blocks((int64_t)rows * (Kp / 8), 8), s, X, ldx, rows, K,
                            reinterpret_cast<__half*>(Y), Kp);
}

}  // namespace detgemm
