// Exact integer GEMM on the warp-level int8 tensor-core path (mma.sync m16n8k32 s8).
//
// acc_ij = sum over segments and k of A_seg[i,k] * W_seg[j,k], accumulated in int32 by
// the tensor core itself: integer multiply-add has no rounding, so every order of the
// sum gives the same bits (the argument of "Deterministic LLM Inference Across GPU
// Kernels ...", §II "Pipeline and alibi", that the int32 accumulator cannot depend on
// tiling or on how K is split). Split-K ("Taming Bitwise Behavior in GPU Kernels with Tensor
// Core", §3.2.2) cuts the flattened K range into `split` contiguous parts; the parts
// meet in an int32 workspace through atomic adds (exact, order-free) and the last CTA
// to arrive at a tile applies the epilogue.
//
// Two kernels:
//  * igemm_tile_kernel   — 128x128x64 CTA tile, 8 warps, 4-stage cp.async ring,
//                          XOR-swizzled shared memory and ldmatrix fragments.
//  (decode-shaped problems, decode_path(M, K), go to the TMA-fed kernels in gemm_skinny.cu)
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace detgemm {

namespace {

constexpr int TBM = 128, TBN = 128, TBK = 64, TSTAGES = 4, TTHREADS = 256;

__device__ __forceinline__ void mma_s8(int32_t (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(uint32_t smem, const void* gptr, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem), "l"(gptr), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t smem) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// byte offset of 16-byte chunk c of row r in a [rows x 64 B] tile, XOR-swizzled so
// that the 8 rows an ldmatrix reads fall into 8 distinct bank groups
__device__ __forceinline__ int swz(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) << 4); }

// flattened K-block range [f0, f1) of split part z over F blocks
__device__ __forceinline__ void split_range(int F, int split, int z, int& f0, int& f1) {
    f0 = (int)(((long long)z * F) / split);
    f1 = (int)(((long long)(z + 1) * F) / split);
}

// Epilogue for one pair of horizontally adjacent accumulators (row, col), (row, col+1).
__device__ __forceinline__ void store_pair(const IGemmArgs& p, int row, int col, int32_t v0, int32_t v1) {
    if (row >= p.M || col >= p.N) return;
    bool two = col + 1 < p.N;
    if (p.mode != EPI_STORE_I32) {
        int32_t ea = p.ea[row];
        const bool bias = p.mode == EPI_BF16_POW2_BIAS;
        uint16_t h0 = bias ? bf16_from_acc_pow2_bias(v0, ea, p.ew[col], p.bias[col])
                           : bf16_from_acc_pow2(v0, ea, p.ew[col]);
        uint16_t* C = reinterpret_cast<uint16_t*>(p.C) + (int64_t)row * p.ldc + col;
        if (two) {
            uint16_t h1 = bias ? bf16_from_acc_pow2_bias(v1, ea, p.ew[col + 1], p.bias[col + 1])
                               : bf16_from_acc_pow2(v1, ea, p.ew[col + 1]);
            *reinterpret_cast<uint32_t*>(C) = (uint32_t)h0 | ((uint32_t)h1 << 16);
        } else {
            C[0] = h0;
        }
    } else {
        int32_t* C = reinterpret_cast<int32_t*>(p.C) + (int64_t)row * p.ldc + col;
        if (two) {
            *reinterpret_cast<int2*>(C) = make_int2(v0, v1);
        } else {
            C[0] = v0;
        }
    }
}

__device__ __forceinline__ void add_pair(const IGemmArgs& p, int row, int col, int32_t v0, int32_t v1) {
    if (row >= p.M || col >= p.N) return;
    int32_t* w = p.ws_acc + (int64_t)row * p.N + col;
    atomicAdd(w, v0);
    if (col + 1 < p.N) atomicAdd(w + 1, v1);
}

__device__ __forceinline__ void load_pair(const IGemmArgs& p, int row, int col, int32_t& v0, int32_t& v1) {
    v0 = v1 = 0;
    if (row >= p.M || col >= p.N) return;
    const int32_t* w = p.ws_acc + (int64_t)row * p.N + col;
    v0 = __ldcg(w);
    if (col + 1 < p.N) v1 = __ldcg(w + 1);
}

// Arrival at a split tile: returns true in every thread of the last CTA to arrive.
__device__ __forceinline__ bool arrive_last(const IGemmArgs& p, int tile) {
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned prev = atomicAdd(p.ws_cnt + tile, 1u);
        s_last = (prev == (unsigned)(p.split - 1));
    }
    __syncthreads();
    if (s_last) __threadfence();
    return s_last;
}

// ------------------------------------------------------------------------------------
// 128x128 tile kernel
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(TTHREADS) igemm_tile_kernel(const __grid_constant__ IGemmArgs p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = warp >> 2, wn = warp & 3;  // 2 x 4 warps, warp tile 64 x 32
    const int m0 = blockIdx.y * TBM, n0 = blockIdx.x * TBN;
    const int nkb = (p.K + TBK - 1) / TBK;
    const int F = nkb * p.nseg;
    int f0, f1;
    split_range(F, p.split, blockIdx.z, f0, f1);
    const int nf = f1 - f0;

    uint8_t* As = smem;
    uint8_t* Bs = smem + TSTAGES * TBM * TBK;
    const uint32_t As_u = smem_u32(As), Bs_u = smem_u32(Bs);

    auto load_stage = [&](int f, int stage) {
        int s = f / nkb, kb = f - s * nkb;
        int k0 = kb * TBK;
        const int8_t* A = p.seg[s].A;
        const int8_t* W = p.seg[s].W;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            int idx = tid + i * TTHREADS;
            int r = idx >> 2, c = idx & 3;
            int kk = k0 + c * 16;
            int kb_valid = p.K - kk;
            kb_valid = kb_valid < 0 ? 0 : (kb_valid > 16 ? 16 : kb_valid);
            int ra = m0 + r, rb = n0 + r;
            const int8_t* ga = A + (int64_t)(ra < p.M ? ra : 0) * p.lda + (kb_valid ? kk : 0);
            const int8_t* gb = W + (int64_t)(rb < p.N ? rb : 0) * p.ldw + (kb_valid ? kk : 0);
            cp_async16(As_u + stage * TBM * TBK + swz(r, c), ga, ra < p.M ? kb_valid : 0);
            cp_async16(Bs_u + stage * TBN * TBK + swz(r, c), gb, rb < p.N ? kb_valid : 0);
        }
    };

    int32_t acc[4][4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][b][c] = 0;

#pragma unroll
    for (int s = 0; s < TSTAGES - 1; ++s) {
        if (s < nf) load_stage(f0 + s, s);
        cp_async_commit();
    }

    for (int it = 0; it < nf; ++it) {
        cp_async_wait<TSTAGES - 2>();
        __syncthreads();
        {
            int nxt = it + TSTAGES - 1;
            if (nxt < nf) load_stage(f0 + nxt, nxt % TSTAGES);
            cp_async_commit();
        }
        const int stage = it % TSTAGES;
        const uint32_t a_base = As_u + stage * TBM * TBK;
        const uint32_t b_base = Bs_u + stage * TBN * TBK;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            uint32_t af[4][4], bf[2][4];
#pragma unroll
            for (int mi = 0; mi < 4; ++mi) {
                int r = wm * 64 + mi * 16 + (lane & 15);
                int c = ks * 2 + (lane >> 4);
                ldmatrix_x4(af[mi], a_base + swz(r, c));
            }
#pragma unroll
            for (int nj = 0; nj < 2; ++nj) {
                int mi = lane >> 3;
                int r = wn * 32 + nj * 16 + ((mi >> 1) << 3) + (lane & 7);
                int c = ks * 2 + (mi & 1);
                ldmatrix_x4(bf[nj], b_base + swz(r, c));
            }
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int ni = 0; ni < 4; ++ni)
                    mma_s8(acc[mi][ni], af[mi], bf[ni >> 1][(ni & 1) * 2], bf[ni >> 1][(ni & 1) * 2 + 1]);
        }
    }
    cp_async_wait<0>();

    const int g = lane >> 2, t = lane & 3;
    if (p.split == 1) {
#pragma unroll
        for (int mi = 0; mi < 4; ++mi)
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                int row = m0 + wm * 64 + mi * 16 + g;
                int col = n0 + wn * 32 + ni * 8 + 2 * t;
                store_pair(p, row, col, acc[mi][ni][0], acc[mi][ni][1]);
                store_pair(p, row + 8, col, acc[mi][ni][2], acc[mi][ni][3]);
            }
        return;
    }
#pragma unroll
    for (int mi = 0; mi < 4; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            int row = m0 + wm * 64 + mi * 16 + g;
            int col = n0 + wn * 32 + ni * 8 + 2 * t;
            add_pair(p, row, col, acc[mi][ni][0], acc[mi][ni][1]);
            add_pair(p, row + 8, col, acc[mi][ni][2], acc[mi][ni][3]);
        }
    if (!arrive_last(p, blockIdx.y * gridDim.x + blockIdx.x)) return;
#pragma unroll
    for (int mi = 0; mi < 4; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            int row = m0 + wm * 64 + mi * 16 + g;
            int col = n0 + wn * 32 + ni * 8 + 2 * t;
            int32_t v0, v1;
            load_pair(p, row, col, v0, v1);
            store_pair(p, row, col, v0, v1);
            load_pair(p, row + 8, col, v0, v1);
            store_pair(p, row + 8, col, v0, v1);
        }
}

bool use_skinny(int M, int K) { return decode_path(M, K); }

int n_tiles(int M, int N) { return ((N + TBN - 1) / TBN) * ((M + TBM - 1) / TBM); }

}  // namespace

size_t igemm_workspace_bytes(int M, int N, int K, int split) {
    if (M == 0 || N == 0) return 0;
    if (use_skinny(M, K)) return skinny_workspace_bytes(M, N, K, split);  // needed at any split
    if (split <= 1) return 0;
    size_t acc = (size_t)M * (size_t)N * sizeof(int32_t);
    acc = (acc + 255) & ~(size_t)255;
    return acc + (size_t)n_tiles(M, N) * sizeof(uint32_t);
}

cudaError_t igemm_launch(const IGemmArgs& a_in, void* ws, cudaStream_t s) {
    IGemmArgs a = a_in;
    if (a.M == 0 || a.N == 0) return cudaSuccess;
    if (use_skinny(a.M, a.K)) {
        if (a.nseg != 1) return cudaErrorInvalidValue;
        return skinny_launch(a.seg[0].A, a.lda, a.seg[0].W, a.ldw, a.ea, a.ew, a.bias, a.C, a.ldc, a.mode, a.M, a.N,
                             a.K, a.split, ws, s);
    }
    if (a.split > 1) {
        size_t accb = (((size_t)a.M * a.N * sizeof(int32_t)) + 255) & ~(size_t)255;
        a.ws_acc = reinterpret_cast<int32_t*>(ws);
        a.ws_cnt = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(ws) + accb);
        cudaError_t e = cudaMemsetAsync(ws, 0, igemm_workspace_bytes(a.M, a.N, a.K, a.split), s);
        if (e != cudaSuccess) return e;
    }
    const int smem = TSTAGES * (TBM + TBN) * TBK;
    cudaError_t e = cudaFuncSetAttribute(igemm_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.N + TBN - 1) / TBN, (a.M + TBM - 1) / TBM, a.split);
    igemm_tile_kernel<<<grid, TTHREADS, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace detgemm
