// Exact integer GEMM on the Blackwell tensor cores (tcgen05, sm_103a).
//
// sm_103a has no integer tcgen05.mma (kind::i8 is rejected), so int8 operands are
// carried exactly in fp16 (every integer in [-2048, 2048] is an fp16 value) and
// multiplied with kind::f16 into fp32 TMEM accumulators. Each product is an integer of
// magnitude <= 128^2 = 2^14, and every partial sum of a chunk of at most 1024 K values
// is an integer of magnitude <= 2^24, which fp32 holds exactly; one MMA instruction sums
// its 16 products exactly and rounds once ("Taming Bitwise Behavior in GPU Kernels with
// Tensor Core", §3.2.1), so no rounding ever changes a value. After each chunk the fp32
// accumulator is drained into int32 registers, which sum the chunks exactly. The
// resulting int32 accumulator is therefore the exact integer dot product, independent
// of tiling, chunking and split-K ("Deterministic LLM Inference Across GPU Kernels ...",
// §II "Pipeline and alibi").
//
// Kernel layout (one CTA per SM, persistent over work units):
//   warp 0   TMA producer: 128x64 A and 256x64 B fp16 boxes (128-byte swizzle) into a
//            4-stage shared-memory ring, one mbarrier pair per stage.
//   warp 1   TMEM owner and MMA issuer: tcgen05.mma M=128 N=256 K=16, four per 64-wide
//            K block, into one of two 256-column fp32 TMEM buffers; one chunk per buffer.
//   warps 2-9  epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 and column half
//            (w - 2) / 4, converts each fp32 chunk to int32 and adds it to 128 int32
//            registers per thread; after the unit's last chunk it applies the epilogue
//            (bf16 pow2 rounding, or int32 store) or, under split-K, adds the partial
//            into an int32 workspace with atomics and the last-arriving CTA finishes.
// A work unit is (plane group d, output tile, split part). Operands are fp16 planes
// [plane][rows][Kp] addressed through 3-D tensor maps; a unit walks a list of
// (A plane, B plane) segments, which is one segment for W8A8 and one per slice pair for
// an Ozaki diagonal.
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

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr int CHUNK_KB = 16;  // 16 blocks of 64 = 1024 K values per exact fp32 chunk
constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*alignment slack*/ + 256 /*barriers*/;

struct Unit {
    int d, tm, tn, z;
};

__device__ __forceinline__ Unit unit_of(const TcArgs& p, int u) {
    Unit r;
    const int per_d = p.tiles_m * p.tiles_n * p.split;
    r.d = u / per_d;
    int rem = u - r.d * per_d;
    int t = rem / p.split;
    r.z = rem - t * p.split;
    // grouped raster: p.group_m tile rows walk together across N for L2 reuse of B
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int gsize = min(p.tiles_m - first_m, p.group_m);
    const int in = t - g * per_group;
    r.tm = first_m + in % gsize;
    r.tn = in / gsize;
    return r;
}

__device__ __forceinline__ void kb_range(const TcArgs& p, const Unit& u, int& f0, int& f1) {
    const int F = p.diag_nseg[u.d] * p.nkb;
    f0 = (int)(((long long)u.z * F) / p.split);
    f1 = (int)(((long long)(u.z + 1) * F) / p.split);
}

// Epilogue of 128 consecutive columns of one output row held by one thread.
__device__ __forceinline__ void finish_row(const TcArgs& p, int d, int row, int col0, const int32_t (&acc)[128]) {
    if (row >= p.M) return;
    if (p.mode == EPI_BF16_POW2) {
        const int32_t ea = p.ea[row];
        uint16_t* C = reinterpret_cast<uint16_t*>(p.C) + (int64_t)row * p.ldc;
#pragma unroll
        for (int j = 0; j < 128; j += 8) {
            const int col = col0 + j;
            if (col + 8 <= p.N) {
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t lo = bf16_from_acc_pow2(acc[j + 2 * i], ea, __ldg(p.ew + col + 2 * i));
                    uint32_t hi = bf16_from_acc_pow2(acc[j + 2 * i + 1], ea, __ldg(p.ew + col + 2 * i + 1));
                    w[i] = lo | (hi << 16);
                }
                *reinterpret_cast<uint4*>(C + col) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (col + i < p.N) C[col + i] = bf16_from_acc_pow2(acc[j + i], ea, __ldg(p.ew + col + i));
            }
        }
    } else {
        int32_t* C = reinterpret_cast<int32_t*>(p.C) + (int64_t)d * p.c_plane + (int64_t)row * p.ldc;
#pragma unroll
        for (int j = 0; j < 128; j += 4) {
            const int col = col0 + j;
            if (col + 4 <= p.N) {
                *reinterpret_cast<int4*>(C + col) = make_int4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (col + i < p.N) C[col + i] = acc[j + i];
            }
        }
    }
}

__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ TcArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* mdone = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdone + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull + b, 1);
            mbar_init(tempty + b, EPI_WARPS);
        }
        mbar_init(mdone, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = p.ndiag * p.tiles_m * p.tiles_n * p.split;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
                const Unit un = unit_of(p, u);
                int f0, f1;
                kb_range(p, un, f0, f1);
                for (int f = f0; f < f1; ++f) {
                    if (!mbar_wait(empty + stage, phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int sidx = f / p.nkb;
                    const int seg = p.diag_first[un.d] + sidx;
                    const int kx = (f - sidx * p.nkb) * BK;
                    uint8_t* sa = smem + stage * STAGE_BYTES;
                    mbar_arrive_expect_tx(full + stage, STAGE_BYTES);
                    tma_load_3d(sa, &tmA, full + stage, kx, un.tm * BM, p.segA[seg]);
                    tma_load_3d(sa + A_BYTES, &tmB, full + stage, kx, un.tn * BN, p.segB[seg]);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let the copies already in flight land before shared memory goes away
                uint32_t n = issued < STAGES ? issued : STAGES;
                int s = stage;
                uint32_t ph = phase;
                for (uint32_t i = 0; i < n; ++i) {
                    if (--s < 0) {
                        s = STAGES - 1;
                        ph ^= 1u;
                    }
                    mbar_wait_drain(full + s, ph);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t tphase = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
                const Unit un = unit_of(p, u);
                int f0, f1;
                kb_range(p, un, f0, f1);
                for (int c0 = f0; c0 < f1 && ok; c0 += CHUNK_KB) {
                    const int c1 = min(f1, c0 + CHUNK_KB);
                    if (!mbar_wait(tempty + buf, tphase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dt = tmem_base + (uint32_t)(buf * BN);
                    for (int f = c0; f < c1; ++f) {
                        if (!mbar_wait(full + stage, phase, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = smem_addr(smem + stage * STAGE_BYTES);
                        const uint64_t ad = sdesc_sw128_kmajor(sa);
                        const uint64_t bd = sdesc_sw128_kmajor(sa + A_BYTES);
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            mma_f16(dt, ad + 2 * k, bd + 2 * k, IDESC, (f > c0 || k > 0) ? 1u : 0u);
                        mma_commit(empty + stage);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    mma_commit(tfull + buf);
                    if (++buf == 2) {
                        buf = 0;
                        tphase ^= 1u;
                    }
                }
            }
            mma_commit(mdone);
            mbar_wait_drain(mdone, 0);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int ew = warp - 2;
        const int q = warp & 3;        // TMEM lane quarter this warp may access
        const int h = ew >> 2;         // column half of the 256-wide tile
        int buf = 0;
        uint32_t tphase = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
            const Unit un = unit_of(p, u);
            int f0, f1;
            kb_range(p, un, f0, f1);
            int32_t acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0;
            for (int c0 = f0; c0 < f1; c0 += CHUNK_KB) {
                // every lane waits, and the warp proceeds only if all saw the phase: the
                // TMEM loads below must be executed by the whole warp or not at all
                const bool got = mbar_wait(tfull + buf, tphase, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + h * 128);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t r[32];
                    tmem_ld32(ta + 32 * j, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[32 * j + i] += __float2int_rn(__uint_as_float(r[i]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty + buf);
                if (++buf == 2) {
                    buf = 0;
                    tphase ^= 1u;
                }
            }
            if (!ok) break;
            const int row = un.tm * BM + q * 32 + lane;
            const int col0 = un.tn * BN + h * 128;
            if (p.split == 1) {
                finish_row(p, un.d, row, col0, acc);
                continue;
            }
            // split-K: exact int32 partial sums meet in the workspace. Each warp owns a
            // 32-row x 128-column sub-block with its own arrival counter; the warp that
            // arrives last (in whichever CTA) reads the full sums and finishes it. No
            // barrier spans more than one warp, so an aborted wait cannot strand others.
            int32_t* ws = p.ws_acc + (int64_t)un.d * p.M * p.N;
            if (row < p.M) {
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (col0 + i < p.N) atomicAdd(ws + (int64_t)row * p.N + col0 + i, acc[i]);
            }
            __threadfence();
            __syncwarp();
            unsigned prev = 0;
            if (lane == 0) {
                const int tile = (un.d * p.tiles_m + un.tm) * p.tiles_n + un.tn;
                prev = atomicAdd(p.ws_cnt + (int64_t)tile * EPI_WARPS + ew, 1u);
            }
            prev = __shfl_sync(0xffffffffu, prev, 0);
            if (prev != (unsigned)(p.split - 1)) continue;
            __threadfence();
            if (row < p.M) {
#pragma unroll
                for (int i = 0; i < 128; ++i) acc[i] = (col0 + i < p.N) ? __ldcg(ws + (int64_t)row * p.N + col0 + i) : 0;
            }
            finish_row(p, un.d, row, col0, acc);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ------------------------------------------------------------------------------------
// int8 -> fp16 widening (exact), zero-filling K up to Kp.  X [rows x K] (ldx) -> Y [rows x Kp]
// ------------------------------------------------------------------------------------
__global__ void widen_i8_f16_kernel(const int8_t* __restrict__ X, int64_t ldx, int rows, int K,
                                    __half* __restrict__ Y, int64_t Kp) {
    const int64_t nvec = Kp / 8;  // 8 outputs (16 bytes) per thread step
    const int64_t total = (int64_t)rows * nvec;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = v / nvec;
        const int k = (int)((v - r * nvec) * 8);
        const int8_t* x = X + r * ldx + k;
        int8_t b[8];
        if (k + 8 <= K) {
            uint2 w = *reinterpret_cast<const uint2*>(x);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                b[i] = (int8_t)(w.x >> (8 * i));
                b[4 + i] = (int8_t)(w.y >> (8 * i));
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) b[i] = (k + i < K) ? x[i] : (int8_t)0;
        }
        __half2 h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __halves2half2(__int2half_rn(b[2 * i]), __int2half_rn(b[2 * i + 1]));
        *reinterpret_cast<uint4*>(Y + r * Kp + k) = *reinterpret_cast<uint4*>(h);
    }
}

// ------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------
std::mutex g_tc_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
int g_num_sms[64];

cudaError_t get_encode(PFN_cuTensorMapEncodeTiled_v12000* fn) {
    std::lock_guard<std::mutex> lock(g_tc_mutex);
    if (!g_encode) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f) return e != cudaSuccess ? e : cudaErrorUnknown;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    *fn = g_encode;
    return cudaSuccess;
}

int num_sms() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(g_tc_mutex);
    if (g_num_sms[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_num_sms[dev] = n > 0 ? n : 148;
    }
    return g_num_sms[dev];
}

// 3-D map over fp16 planes [planes][rows][Kp], box {64, box_rows, 1}, 128-byte swizzle
cudaError_t make_map(CUtensorMap* m, const void* base, int64_t Kp, int rows, int planes, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    cudaError_t e = get_encode(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[3] = {(cuuint64_t)Kp, (cuuint64_t)rows, (cuuint64_t)planes};
    cuuint64_t strides[2] = {(cuuint64_t)Kp * 2, (cuuint64_t)Kp * 2 * (cuuint64_t)rows};
    cuuint32_t box[3] = {(cuuint32_t)BK, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

int64_t tc_padded_k(int K) { return ((int64_t)K + BK - 1) / BK * BK; }

cudaError_t widen_i8_f16_launch(const int8_t* X, int64_t ldx, int rows, int K, void* Y, int64_t Kp, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int64_t total = (int64_t)rows * (Kp / 8);
    int blocks = (int)((total + 255) / 256);
    const int cap = num_sms() * 8;
    if (blocks > cap) blocks = cap;
    widen_i8_f16_kernel<<<blocks, 256, 0, s>>>(X, ldx, rows, K, reinterpret_cast<__half*>(Y), Kp);
    return cudaGetLastError();
}

size_t tc_split_bytes(int ndiag, int M, int N, int split) {
    if (split <= 1) return 0;
    const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    size_t acc = ((size_t)ndiag * M * N * sizeof(int32_t) + 255) & ~(size_t)255;
    return acc + (size_t)ndiag * tiles * EPI_WARPS * sizeof(uint32_t);
}

cudaError_t tc_gemm_launch(const TcArgs& a_in, const void* A16, int a_planes, const void* B16, int b_planes,
                           int64_t Kp, void* ws_split, cudaStream_t s) {
    TcArgs a = a_in;
    if (a.M == 0 || a.N == 0) return cudaSuccess;
    a.tiles_m = (a.M + BM - 1) / BM;
    a.tiles_n = (a.N + BN - 1) / BN;
    a.nkb = (int)(Kp / BK);
    if (a.group_m <= 0) a.group_m = 8;
    CUtensorMap tmA, tmB;
    cudaError_t e = make_map(&tmA, A16, Kp, a.M, a_planes, BM);
    if (e == cudaSuccess) e = make_map(&tmB, B16, Kp, a.N, b_planes, BN);
    if (e != cudaSuccess) return e;
    if (a.split > 1) {
        size_t accb = (((size_t)a.ndiag * a.M * a.N * sizeof(int32_t)) + 255) & ~(size_t)255;
        a.ws_acc = reinterpret_cast<int32_t*>(ws_split);
        a.ws_cnt = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(ws_split) + accb);
        e = cudaMemsetAsync(ws_split, 0, tc_split_bytes(a.ndiag, a.M, a.N, a.split), s);
        if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int total = a.ndiag * a.tiles_m * a.tiles_n * a.split;
    const int grid = total < num_sms() ? total : num_sms();
    tc_gemm_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(tmA, tmB, a);
    return cudaGetLastError();
}

DETGEMM_STATUS_ACCESSOR(tc_take_status)

}  // namespace detgemm
