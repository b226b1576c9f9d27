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
//  * igemm_skinny_kernel — M <= 64: each warp streams 32 rows of W straight from
//                          global memory with 16-byte loads; the int8 values are widened
//                          exactly to fp16 in registers for the fp16 warp MMA (fp32
//                          partials drained to int32 every <= 1024 K). W is read exactly
//                          once per split part.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace detgemm {

namespace {

constexpr int TBM = 128, TBN = 128, TBK = 64, TSTAGES = 4, TTHREADS = 256;
constexpr int SKN = 128;  // W rows per skinny CTA (4 warps x 32)

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
    if (p.mode == EPI_BF16_POW2) {
        int32_t ea = p.ea[row];
        uint16_t h0 = bf16_from_acc_pow2(v0, ea, p.ew[col]);
        uint16_t* C = reinterpret_cast<uint16_t*>(p.C) + (int64_t)row * p.ldc + col;
        if (two) {
            uint16_t h1 = bf16_from_acc_pow2(v1, ea, p.ew[col + 1]);
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

// ------------------------------------------------------------------------------------
// Skinny kernel (M <= 16 * MT)
//
// Lane (g, t) of a warp loads bytes [16t, 16t + 16) of a 64-wide K block for W row g of
// each of its four 8-row groups, and the same bytes of A rows g and g + 8 of each 16-row
// tile. The k positions a lane holds are assigned to mma fragment slots identically for
// A and W, so the product covers every k of the block exactly once (the dot product is
// an exact integer sum, hence indifferent to the order of its k).
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg_nc16(const int8_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg16(const int8_t* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// 16 bytes at p where only `valid` (0..16) bytes lie inside the matrix; the rest read as 0
__device__ __forceinline__ uint4 ld16_partial(const int8_t* p, int valid) {
    uint32_t w[4] = {0, 0, 0, 0};
    for (int b = 0; b < valid; ++b) w[b >> 2] |= (uint32_t)(uint8_t)p[b] << (8 * (b & 3));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint32_t u4_get(const uint4& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// fp16 warp MMA: D (fp32) += A (16x16 fp16) * B (16x8 fp16)
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Exact int8x4 -> two fp16x2 (bytes 0,1 -> lo; bytes 2,3 -> hi): b + 128 is placed under
// the fp16 exponent of 1024, giving 1024 + (b + 128), and 1152 is subtracted.
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

// 16 int8 values (a uint4) -> 8 fp16x2 words, in k order
__device__ __forceinline__ void i8x16_to_f16x16(const uint4& v, uint32_t (&h)[8]) {
    i8x4_to_f16x4(v.x, h[0], h[1]);
    i8x4_to_f16x4(v.y, h[2], h[3]);
    i8x4_to_f16x4(v.z, h[4], h[5]);
    i8x4_to_f16x4(v.w, h[6], h[7]);
}

// The skinny kernel runs on the fp16 warp MMA (this part's int8 warp MMA is about four
// times slower): int8 values are widened exactly in registers, products accumulate in
// fp32 exactly (integers below 2^24) for at most 16 blocks of 64 K values per thread,
// and every such chunk is drained into int32 registers.
template <int MT, int U>
__global__ void __launch_bounds__(128) igemm_skinny_kernel(const __grid_constant__ IGemmArgs p) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int nw = blockIdx.x * SKN + warp * 32;
    const int nkb = (p.K + 63) / 64;
    const int F = nkb * p.nseg;
    int f0, f1;
    split_range(F, p.split, blockIdx.y, f0, f1);

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
    static_assert(16 % U == 0, "a drain must fall on an iteration boundary");
    int since = 0;  // 64-wide K blocks accumulated in accf since the last drain

    for (int fb = f0; fb < f1; fb += U) {
        uint4 wv[U][4], av[U][MT][2];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            int f = fb + u;
            bool live = f < f1;
            int s = live ? f / nkb : 0;
            int kb = live ? f - s * nkb : 0;
            int kk = kb * 64 + 16 * t;
            int valid = live ? p.K - kk : 0;
            valid = valid < 0 ? 0 : (valid > 16 ? 16 : valid);
            const int8_t* W = p.seg[s].W;
            const int8_t* A = p.seg[s].A;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                int n = nw + 8 * j + g;
                if (n < p.N && valid == 16) wv[u][j] = ldg_nc16(W + (int64_t)n * p.ldw + kk);
                else if (n < p.N && valid > 0) wv[u][j] = ld16_partial(W + (int64_t)n * p.ldw + kk, valid);
                else wv[u][j] = make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    int m = mt * 16 + h * 8 + g;
                    if (m < p.M && valid == 16) av[u][mt][h] = ldg16(A + (int64_t)m * p.lda + kk);
                    else if (m < p.M && valid > 0) av[u][mt][h] = ld16_partial(A + (int64_t)m * p.lda + kk, valid);
                    else av[u][mt][h] = make_uint4(0, 0, 0, 0);
                }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint32_t hw[4][8];
#pragma unroll
            for (int j = 0; j < 4; ++j) i8x16_to_f16x16(wv[u][j], hw[j]);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t h0[8], h1[8];
                i8x16_to_f16x16(av[u][mt][0], h0);
                i8x16_to_f16x16(av[u][mt][1], h1);
                // the lane's 16 k values kk .. kk+15 feed four k16 MMAs, the same k slots
                // for A and W: logical (2t + j) <- kk + 4q + j, (2t + 8 + j) <- kk + 4q + 2 + j
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t a[4] = {h0[2 * q], h1[2 * q], h0[2 * q + 1], h1[2 * q + 1]};
#pragma unroll
                    for (int j = 0; j < 4; ++j) mma_f16(accf[mt][j], a, hw[j][2 * q], hw[j][2 * q + 1]);
                }
            }
        }
        since += U;
        if (since == 16) {
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
#pragma unroll
    for (int a = 0; a < MT; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][b][c] += __float2int_rn(accf[a][b][c]);

    if (p.split == 1) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                int col = nw + 8 * j + 2 * t;
                store_pair(p, mt * 16 + g, col, acc[mt][j][0], acc[mt][j][1]);
                store_pair(p, mt * 16 + g + 8, col, acc[mt][j][2], acc[mt][j][3]);
            }
        return;
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int col = nw + 8 * j + 2 * t;
            add_pair(p, mt * 16 + g, col, acc[mt][j][0], acc[mt][j][1]);
            add_pair(p, mt * 16 + g + 8, col, acc[mt][j][2], acc[mt][j][3]);
        }
    if (!arrive_last(p, blockIdx.x)) return;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int col = nw + 8 * j + 2 * t;
            int32_t v0, v1;
            load_pair(p, mt * 16 + g, col, v0, v1);
            store_pair(p, mt * 16 + g, col, v0, v1);
            load_pair(p, mt * 16 + g + 8, col, v0, v1);
            store_pair(p, mt * 16 + g + 8, col, v0, v1);
        }
}

bool use_skinny(int M) { return M <= 64; }

int n_tiles(int M, int N) {
    if (use_skinny(M)) return (N + SKN - 1) / SKN;
    return ((N + TBN - 1) / TBN) * ((M + TBM - 1) / TBM);
}

}  // namespace

size_t igemm_workspace_bytes(int M, int N, int split) {
    if (split <= 1 || M == 0 || N == 0) return 0;
    size_t acc = (size_t)M * (size_t)N * sizeof(int32_t);
    acc = (acc + 255) & ~(size_t)255;
    return acc + (size_t)n_tiles(M, N) * sizeof(uint32_t);
}

cudaError_t igemm_launch(const IGemmArgs& a_in, void* ws, cudaStream_t s) {
    IGemmArgs a = a_in;
    if (a.M == 0 || a.N == 0) return cudaSuccess;
    if (a.split > 1) {
        size_t accb = (((size_t)a.M * a.N * sizeof(int32_t)) + 255) & ~(size_t)255;
        a.ws_acc = reinterpret_cast<int32_t*>(ws);
        a.ws_cnt = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(ws) + accb);
        cudaError_t e = cudaMemsetAsync(ws, 0, igemm_workspace_bytes(a.M, a.N, a.split), s);
        if (e != cudaSuccess) return e;
    }
    if (use_skinny(a.M)) {
        dim3 grid((a.N + SKN - 1) / SKN, a.split);
        int mt = (a.M + 15) / 16;
        switch (mt) {
            case 1: igemm_skinny_kernel<1, 4><<<grid, 128, 0, s>>>(a); break;
            case 2: igemm_skinny_kernel<2, 2><<<grid, 128, 0, s>>>(a); break;
            case 3: igemm_skinny_kernel<3, 2><<<grid, 128, 0, s>>>(a); break;
            default: igemm_skinny_kernel<4, 1><<<grid, 128, 0, s>>>(a); break;
        }
        return cudaGetLastError();
    }
    const int smem = TSTAGES * (TBM + TBN) * TBK;
    cudaError_t e = cudaFuncSetAttribute(igemm_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.N + TBN - 1) / TBN, (a.M + TBM - 1) / TBM, a.split);
    igemm_tile_kernel<<<grid, TTHREADS, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace detgemm
