// Decode-shaped exact int8 GEMM (M <= 64): HBM-bound streaming of W.
//
// acc_ij = sum_k A_ik * W_jk exactly ("Deterministic LLM Inference Across GPU Kernels
// ...", §II "Pipeline and alibi"), then the bf16 pow2 epilogue. With M <= 64 there are
// at most 128 multiply-adds per W byte, so the kernel is bound by reading W once from
// HBM; its job is to keep enough bytes in flight.
//
// One CTA per (128-row block of W, split part). Warp 0, lane 0, is a TMA producer: for
// each 128-wide K block it loads the int8 boxes W[128 x 128] and A[16 MT x 128] (128-byte
// swizzle, one full cache line per row; rows past M or N and columns past K arrive as
// zeros) into a 6-stage ring; two CTAs per SM keep ~200 KB of W in flight per SM.
// Warps 1-4 each own 32 rows of W: they read 16-byte fragments from shared memory, widen
// int8 to fp16 exactly in registers and run the fp16 warp MMA (m16n8k16, fp32
// accumulate; this part's int8 warp MMA is about four times slower). Every partial sum of
// at most 1024 products of magnitude <= 2^14 is an integer below 2^24, so
// the fp32 accumulators are exact; they are drained into int32 registers every 1024 K.
// Split-K parts meet through int32 atomics; the warp that arrives last at its 32-row
// sub-block finishes it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace detgemm {

namespace {

using namespace sm100;

constexpr int SK_ROWS = 128;       // W rows per CTA
constexpr int SK_BK = 128;         // K per stage: one 128-byte line per W row (128-byte swizzle)
constexpr int SK_STAGES = 6;
constexpr int SK_CONSUMERS = 4;
constexpr int SK_THREADS = 32 * (1 + SK_CONSUMERS);
constexpr int SK_W_BYTES = SK_ROWS * SK_BK;  // 16 KB

__host__ __device__ constexpr int sk_stage_bytes(int MT) { return SK_W_BYTES + 16 * MT * SK_BK; }
__host__ __device__ constexpr int sk_smem_bytes(int MT) { return SK_STAGES * sk_stage_bytes(MT) + 1024 + 512; }

struct SkArgs {
    int M, N, K;
    int nblocks;        // 128-row blocks of W
    const int32_t* ea;
    const int32_t* ew;
    uint16_t* C;
    int64_t ldc;
    int mode;           // EPI_BF16_POW2 or EPI_STORE_I32
    int32_t* ws_acc;    // [M x N] exact partial sums
    uint32_t* ws_cnt;   // [n blocks x 4] arrivals
};

// byte offset of the 16-byte chunk c of row r in a box of 128-byte rows, 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// The memory clobber keeps these reads between the stage's full-barrier wait and its
// release (the compiler may not move them across either).
__device__ __forceinline__ uint4 lds16(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::
            "r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_addr(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Exact int8x4 -> two fp16x2 words: b + 128 is placed under the fp16 exponent of 1024
// (giving 1024 + b + 128) and 1152 is subtracted.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t x = w ^ 0x80808080u;
    const uint32_t l = __byte_perm(x, 0x64646464u, 0x4140);
    const uint32_t h = __byte_perm(x, 0x64646464u, 0x4342);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const __half2 rl = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
    const __half2 rh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
    lo = *reinterpret_cast<const uint32_t*>(&rl);
    hi = *reinterpret_cast<const uint32_t*>(&rh);
}

__device__ __forceinline__ void i8x16_to_f16x16(const uint4& v, uint32_t (&h)[8]) {
    i8x4_to_f16x4(v.x, h[0], h[1]);
    i8x4_to_f16x4(v.y, h[2], h[3]);
    i8x4_to_f16x4(v.z, h[4], h[5]);
    i8x4_to_f16x4(v.w, h[6], h[7]);
}

__device__ __forceinline__ void store_pair(const SkArgs& p, int row, int col, int32_t v0, int32_t v1) {
    if (row >= p.M || col >= p.N) return;
    const bool two = col + 1 < p.N;
    if (p.mode == EPI_BF16_POW2) {
        const int32_t ea = p.ea[row];
        uint16_t* C = p.C + (int64_t)row * p.ldc + col;
        const uint16_t h0 = bf16_from_acc_pow2(v0, ea, p.ew[col]);
        if (two) {
            const uint16_t h1 = bf16_from_acc_pow2(v1, ea, p.ew[col + 1]);
            *reinterpret_cast<uint32_t*>(C) = (uint32_t)h0 | ((uint32_t)h1 << 16);
        } else {
            C[0] = h0;
        }
    } else {
        int32_t* C = reinterpret_cast<int32_t*>(p.C) + (int64_t)row * p.ldc + col;
        if (two) *reinterpret_cast<int2*>(C) = make_int2(v0, v1);
        else C[0] = v0;
    }
}

// CTA that owns flattened K block f when F blocks are cut into P equal contiguous ranges
// (range i is [i F / P, (i + 1) F / P))
__device__ __forceinline__ int owner_of(long long f, long long F, long long P) { return (int)(((f + 1) * P - 1) / F); }

template <int MT>
__global__ void __launch_bounds__(SK_THREADS) skinny_kernel(const __grid_constant__ CUtensorMap tmW,
                                                            const __grid_constant__ CUtensorMap tmA,
                                                            const __grid_constant__ SkArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int STAGE = sk_stage_bytes(MT);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SK_STAGES * STAGE);
    uint64_t* empty = full + SK_STAGES;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + SK_STAGES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kbr = (p.K + SK_BK - 1) / SK_BK;  // K blocks per row block
    const long long F = (long long)p.nblocks * kbr;
    const long long P = gridDim.x;
    const int f0 = (int)(((long long)blockIdx.x * F) / P);
    const int f1 = (int)(((long long)(blockIdx.x + 1) * F) / P);

    if (threadIdx.x == 0) {
        for (int s = 0; s < SK_STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, SK_CONSUMERS);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tmW);
            prefetch_tmap(&tmA);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0;
            bool ok = true;
            for (int f = f0; f < f1; ++f) {
                if (!mbar_wait(empty + stage, phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const int nb = f / kbr, kb = f - nb * kbr;
                uint8_t* st = smem + stage * STAGE;
                mbar_arrive_expect_tx(full + stage, STAGE);
                tma_load_2d(st, &tmW, full + stage, kb * SK_BK, nb * SK_ROWS);
                tma_load_2d(st + SK_W_BYTES, &tmA, full + stage, kb * SK_BK, 0);
                ++issued;
                if (++stage == SK_STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                uint32_t n = issued < SK_STAGES ? issued : SK_STAGES;
                int s = stage;
                uint32_t ph = phase;
                for (uint32_t i = 0; i < n; ++i) {
                    if (--s < 0) {
                        s = SK_STAGES - 1;
                        ph ^= 1u;
                    }
                    mbar_wait_drain(full + s, ph);
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1;         // rows [32 cw, 32 cw + 32) of the row block
    const int g = lane >> 2, t = lane & 3;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    const uint32_t sbase = smem_addr(smem);
    int f = f0;
    while (f < f1 && ok) {
        // one segment: this CTA's K blocks inside row block nb
        const int nb = f / kbr;
        const int fend = min(f1, (nb + 1) * kbr);
        int32_t acc[MT][4][4];
        float accf[MT][4][4];
#pragma unroll
        for (int a = 0; a < MT; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    acc[a][b][c] = 0;
                    accf[a][b][c] = 0.f;
                }
        int since = 0;
        for (; f < fend; ++f) {
            // lane 0 polls; after it has seen the phase complete, every lane confirms with one
            // try_wait of its own (the acquire that makes the TMA-written bytes visible to it)
            bool got = lane == 0 ? mbar_wait(full + stage, phase, abort_flag) : true;
            got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
            if (!got) {
                ok = false;
                break;
            }
            for (int spin = 0; !mbar_try_wait(smem_addr(full + stage), phase); ++spin) {
                if (spin > (1 << 20)) {  // cannot happen once lane 0 saw the phase; bounded anyway
                    *abort_flag = 1;
                    break;
                }
            }
            const uint32_t wb = sbase + stage * STAGE;
            const uint32_t ab = wb + SK_W_BYTES;
            // lane (g, t) takes the 16-byte chunks t and t + 4 of each 128-byte row: 32 k values
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int c = t + 4 * half;
                uint32_t hw[4][8];
#pragma unroll
                for (int j = 0; j < 4; ++j) i8x16_to_f16x16(lds16(wb + sw128(32 * cw + 8 * j + g, c)), hw[j]);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t h0[8], h1[8];
                    i8x16_to_f16x16(lds16(ab + sw128(16 * mt + g, c)), h0);
                    i8x16_to_f16x16(lds16(ab + sw128(16 * mt + g + 8, c)), h1);
                    // the chunk's 16 k values feed four k16 MMAs with the same k slots for A and
                    // W: logical (2t + j) <- 4q + j, (2t + 8 + j) <- 4q + 2 + j within the chunk
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t a[4] = {h0[2 * q], h1[2 * q], h0[2 * q + 1], h1[2 * q + 1]};
#pragma unroll
                        for (int j = 0; j < 4; ++j) mma_f16(accf[mt][j], a, hw[j][2 * q], hw[j][2 * q + 1]);
                    }
                }
            }
            // The next write into this stage is a TMA copy (async proxy) while the reads above
            // went through the generic proxy: a proxy fence orders them before the release.
            // Without it the refill could land while a lane was still reading (observed as
            // whole columns off by one K block's contribution, only under load).
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + stage);
            if (++stage == SK_STAGES) {
                stage = 0;
                phase ^= 1u;
            }
            if (++since == 1024 / SK_BK) {  // 1024 products per accumulator since the last drain
#pragma unroll
                for (int a = 0; a < MT; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b)
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            acc[a][b][c] += __float2int_rn(accf[a][b][c]);
                            accf[a][b][c] = 0.f;
                        }
                since = 0;
            }
        }
        if (!ok) break;
#pragma unroll
        for (int a = 0; a < MT; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[a][b][c] += __float2int_rn(accf[a][b][c]);

        // exact partial of this segment -> workspace; the warp that completes the row block's
        // count (one arrival per CTA whose range touches it) finishes it.
        // accumulator (mt, j, e): row 16 mt + g (+8 for e >= 2), column 128 nb + 32 cw + 8 j + 2 t (+1 odd e)
        const int nc = nb * SK_ROWS + 32 * cw;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = 16 * mt + g + 8 * (e >> 1), col = nc + 8 * j + 2 * t + (e & 1);
                    if (row < p.M && col < p.N) atomicAdd(p.ws_acc + (int64_t)row * p.N + col, acc[mt][j][e]);
                }
        __threadfence();
        __syncwarp();
        const int expected = owner_of((long long)(nb + 1) * kbr - 1, F, P) - owner_of((long long)nb * kbr, F, P) + 1;
        unsigned prev = 0;
        if (lane == 0) prev = atomicAdd(p.ws_cnt + nb * SK_CONSUMERS + cw, 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev != (unsigned)(expected - 1)) continue;
        __threadfence();
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = 16 * mt + g + 8 * h, col = nc + 8 * j + 2 * t;
                    int32_t v0 = 0, v1 = 0;
                    if (row < p.M && col < p.N) {
                        v0 = __ldcg(p.ws_acc + (int64_t)row * p.N + col);
                        if (col + 1 < p.N) v1 = __ldcg(p.ws_acc + (int64_t)row * p.N + col + 1);
                    }
                    store_pair(p, row, col, v0, v1);
                }
    }
    if (!ok) {
        // let loads already issued into the ring land before the CTA's shared memory goes away
        if (lane == 0) {
            int s = stage;
            uint32_t ph = phase;
            const int n = (f1 - f0) < SK_STAGES ? (f1 - f0) : SK_STAGES;
            for (int i = 0; i < n; ++i) {
                mbar_wait_drain(full + s, ph, kDrainLimitNs);
                if (++s == SK_STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    }
}

std::mutex g_sk_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_sk_encode = nullptr;

cudaError_t sk_map(CUtensorMap* m, const void* base, int K, int64_t ld, int rows, int box_rows) {
    {
        std::lock_guard<std::mutex> lock(g_sk_mutex);
        if (!g_sk_encode) {
            void* f = nullptr;
            cudaDriverEntryPointQueryResult q;
            cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f) return e != cudaSuccess ? e : cudaErrorUnknown;
            g_sk_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        }
    }
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {(cuuint32_t)SK_BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_sk_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int g_sk_sms[64];

int sk_num_sms() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(g_sk_mutex);
    if (g_sk_sms[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sk_sms[dev] = n > 0 ? n : 148;
    }
    return g_sk_sms[dev];
}

template <int MT>
cudaError_t sk_launch_mt(const CUtensorMap& tmW, const CUtensorMap& tmA, const SkArgs& a, cudaStream_t s) {
    const int smem = sk_smem_bytes(MT);
    cudaError_t e = cudaFuncSetAttribute(skinny_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // two CTAs per SM (the shared-memory ring allows two), each streaming an equal share
    const long long blocks = (long long)a.nblocks * ((a.K + SK_BK - 1) / SK_BK);
    long long grid = 2LL * sk_num_sms();
    if (grid > blocks) grid = blocks;
    skinny_kernel<MT><<<(unsigned)grid, SK_THREADS, smem, s>>>(tmW, tmA, a);
    return cudaGetLastError();
}

}  // namespace

size_t skinny_workspace_bytes(int M, int N, int split) {
    (void)split;
    if (M == 0 || N == 0) return 0;
    size_t acc = ((size_t)M * N * sizeof(int32_t) + 255) & ~(size_t)255;
    return acc + (size_t)((N + SK_ROWS - 1) / SK_ROWS) * SK_CONSUMERS * sizeof(uint32_t);
}

cudaError_t skinny_launch(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw, const int32_t* ea,
                          const int32_t* ew, void* C, int64_t ldc, int mode, int M, int N, int K, int split, void* ws,
                          cudaStream_t s) {
    (void)split;  // the kernel divides K among the SMs itself; the bits never depend on it
    if (M == 0 || N == 0) return cudaSuccess;
    const int MT = (M + 15) / 16;
    SkArgs a = {};
    a.M = M;
    a.N = N;
    a.K = K;
    a.nblocks = (N + SK_ROWS - 1) / SK_ROWS;
    a.ea = ea;
    a.ew = ew;
    a.C = reinterpret_cast<uint16_t*>(C);
    a.ldc = ldc;
    a.mode = mode;
    CUtensorMap tmW, tmA;
    cudaError_t e = sk_map(&tmW, W, K, ldw, N, SK_ROWS);
    if (e == cudaSuccess) e = sk_map(&tmA, A, K, lda, M, 16 * MT);
    if (e != cudaSuccess) return e;
    size_t accb = (((size_t)M * N * sizeof(int32_t)) + 255) & ~(size_t)255;
    a.ws_acc = reinterpret_cast<int32_t*>(ws);
    a.ws_cnt = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(ws) + accb);
    e = cudaMemsetAsync(ws, 0, skinny_workspace_bytes(M, N, 1), s);
    if (e != cudaSuccess) return e;
    switch (MT) {
        case 1: return sk_launch_mt<1>(tmW, tmA, a, s);
        case 2: return sk_launch_mt<2>(tmW, tmA, a, s);
        case 3: return sk_launch_mt<3>(tmW, tmA, a, s);
        default: return sk_launch_mt<4>(tmW, tmA, a, s);
    }
}

DETGEMM_STATUS_ACCESSOR(skinny_take_status)

}  // namespace detgemm
