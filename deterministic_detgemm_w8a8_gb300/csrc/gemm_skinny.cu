// Decode-shaped exact int8 GEMM (M <= 64): HBM-bound streaming of W.
//
// acc_ij = sum_k A_ik * W_jk exactly ("Deterministic LLM Inference Across GPU Kernels
// ...", §II "Pipeline and alibi"), then the bf16 pow2 epilogue. With M <= 64 there are
// at most 128 multiply-adds per W byte, so the kernel is bound by reading W once from
// HBM; its job is to keep enough bytes in flight and to spend few instructions per byte.
// K <= 4096 runs in one launch (skinny_wk_kernel, below: whole rows of W per CTA); longer K
// takes the split form:
//
// Three launches per call, chained by programmatic dependent launch (each starts while
// its predecessor runs and waits for it with griddepcontrol.wait where it needs its data):
//   prep    zeroes the int32 accumulator workspace and writes an exact fp16 copy of A
//           (tiny: M x K) into it, so that the main kernel converts only W;
//   main    streams W and adds its exact partial sums into the workspace with int32
//           atomics; its TMA producer starts on W before prep has finished and waits for
//           prep only before its first A load;
//   finish  once main has completed (all partial sums performed), rounds each sum to bf16
//           (or stores it as int32).
// Main kernel: persistent (two CTAs per SM up to 32 tokens, else one), each CTA owning an
// equal contiguous range of the flattened (128-row block of W, 128-wide K block) space.
// Warp 0, lane 0, is the TMA producer: per K block it loads the int8 box W[128 x 128]
// (evict-first L2 policy: W is read exactly once) and the fp16 boxes A[16 MT x 64] x 2
// (128-byte swizzle; rows past M or N and columns past K arrive as zeros) into a ring of
// stages. The consumer warps each own 128 / SK_CONSUMERS rows of W: they read 16-byte
// fragments from shared memory, widen the int8 W bytes to fp16 exactly in registers and
// run the fp16 warp MMA (m16n8k16, fp32 accumulate; this part's int8 warp MMA is about
// four times slower). Every partial sum of at most 1024 products of magnitude <= 2^14 is
// an integer below 2^24, so the fp32 accumulators are exact; they are drained into int32
// registers every 1024 K. The CTAs meet through int32 atomics in the workspace (integer
// addition: the order in which they land cannot change the sum).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace detgemm {

namespace {

using namespace sm100;

constexpr int SK_ROWS = 128;       // W rows per row block
constexpr int SK_BK = 128;         // K per stage: one 128-byte line per W row (128-byte swizzle)
constexpr int SK_CONSUMERS = 8;    // consumer warps per CTA
constexpr int SK_RPW = SK_ROWS / SK_CONSUMERS;  // W rows per consumer warp
constexpr int SK_NJ = SK_RPW / 8;               // n8 MMA column groups per consumer warp
constexpr int SK_THREADS = 32 * (1 + SK_CONSUMERS);
constexpr int SK_W_BYTES = SK_ROWS * SK_BK;  // 16 KB

// Up to 32 tokens two CTAs share an SM (registers and shared memory allow it); above,
// the accumulators need the registers of one CTA per SM, which then gets a deeper ring.
__host__ __device__ constexpr int sk_ctas_per_sm(int MT) { return MT <= 2 ? 2 : 1; }
__host__ __device__ constexpr int sk_smem_budget(int MT) { return sk_ctas_per_sm(MT) == 2 ? 110 * 1024 : 220 * 1024; }
__host__ __device__ constexpr int sk_a_box_bytes(int MT) { return 16 * MT * 128; }  // 16 MT rows x 64 fp16
__host__ __device__ constexpr int sk_stage_bytes(int MT) { return SK_W_BYTES + 2 * sk_a_box_bytes(MT); }
__host__ __device__ constexpr int sk_stages(int MT) {
    return (sk_smem_budget(MT) - 1280) / sk_stage_bytes(MT) > 6 ? 6 : (sk_smem_budget(MT) - 1280) / sk_stage_bytes(MT);
}
__host__ __device__ constexpr int sk_smem_bytes(int MT) { return sk_stages(MT) * sk_stage_bytes(MT) + 1024 + 256; }

struct SkArgs {
    int M, N, K;
    int nblocks;        // 128-row blocks of W
    const int32_t* ea;
    const int32_t* ew;
    const uint16_t* bias;  // [N] bf16 bits (EPI_BF16_POW2_BIAS)
    uint16_t* C;
    int64_t ldc;
    int mode;           // EPI_BF16_POW2, EPI_BF16_POW2_BIAS or EPI_STORE_I32
    int32_t* ws_acc;    // [N x M] exact sums (token-contiguous: one warp atomic covers 8
                        // consecutive tokens of 4 columns)
    int parts;          // 0: each CTA takes an equal share of the flattened (row block, K block)
                        // space; > 0: exactly `parts` contiguous K parts per row block, CTA b
                        // taking part b % parts of row block b / parts (the tensor-core decode
                        // kernel: the cluster size)
};

// Workspace: [acc: N x M int32][A16: M x lda16 fp16], each part 256-byte aligned.
struct SkLayout {
    size_t acc, a16, total;
    int64_t lda16;
};

SkLayout sk_layout(int M, int N, int K) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    SkLayout L;
    L.lda16 = ((int64_t)K + 7) / 8 * 8;
    L.acc = 0;
    L.a16 = up((size_t)M * N * sizeof(int32_t));
    L.total = L.a16 + up((size_t)M * L.lda16 * 2);
    return L;
}

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

// L2 policy for the W stream, which nothing re-reads: its lines are evicted first (measured
// on GB300: a TMA stream of these boxes reaches ~5.5 TB/s with it, ~4.6 TB/s without)
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// tma_load_2d with an L2 cache policy
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
        "%4}], [%2], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_addr(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// L2 prefetch of the box at (x, y): a hint that moves no data into shared memory, so it may be
// issued before the wait on the prerequisite grid (any write that grid makes to the same lines
// lands in L2 before the real loads after the wait read them)
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* m, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(m)),
                 "r"(x), "r"(y)
                 : "memory");
}

// programmatic dependent launch: let the dependent grid start / wait for the prerequisite
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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

// rne_bf16(acc * 2^ea * 2^ew) for ea, ew in [-60, 40]: acc truncated to 24 significant bits
// with the last kept bit set when anything was dropped (rounding to odd), scaled exactly by
// the two powers of two, then rounded to nearest-even: odd rounding at 24 >= 8 + 2 bits
// followed by one nearest rounding at 8 bits equals one nearest rounding, so the bits are
// those of the integer construction bf16_from_acc_pow2.
__device__ __forceinline__ uint16_t bf16_pow2_fast(int32_t acc, int32_t ea, int32_t ew) {
    const float x = __int2float_rz(acc);
    const uint32_t xb = __float_as_uint(x) | (uint32_t)(__float2int_rz(x) != acc);
    const float y = __fmul_rn(__fmul_rn(__uint_as_float(xb), __uint_as_float((uint32_t)(ea + 127) << 23)),
                              __uint_as_float((uint32_t)(ew + 127) << 23));
    return __bfloat16_as_ushort(__float2bfloat16_rn(y));
}

__device__ __forceinline__ void sts16(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// store_pair with the exponents (and bias bits) already at hand, for rows < p.M, cols < p.N
__device__ __forceinline__ void store_pair_pre(const SkArgs& p, int row, int col, int32_t v0, int32_t v1, int32_t ea,
                                               int32_t ew0, int32_t ew1, uint32_t b0, uint32_t b1) {
    if (row >= p.M || col >= p.N) return;
    const bool two = col + 1 < p.N;
    if (p.mode == EPI_STORE_I32) {
        int32_t* C = reinterpret_cast<int32_t*>(p.C) + (int64_t)row * p.ldc + col;
        if (two) *reinterpret_cast<int2*>(C) = make_int2(v0, v1);
        else C[0] = v0;
        return;
    }
    uint16_t h0, h1;
    if (p.mode == EPI_BF16_POW2_BIAS) {
        h0 = bf16_from_acc_pow2_bias(v0, ea, ew0, b0);
        h1 = bf16_from_acc_pow2_bias(v1, ea, ew1, b1);
    } else if (__all_sync(__activemask(), ea >= -60 && ea <= 40 && ew0 >= -60 && ew0 <= 40 && ew1 >= -60 && ew1 <= 40)) {
        // a warp-uniform branch, not a select: the integer form is evaluated only where needed
        h0 = bf16_pow2_fast(v0, ea, ew0);
        h1 = bf16_pow2_fast(v1, ea, ew1);
    } else {
        h0 = bf16_from_acc_pow2(v0, ea, ew0);
        h1 = bf16_from_acc_pow2(v1, ea, ew1);
    }
    uint16_t* C = p.C + (int64_t)row * p.ldc + col;
    if (two) *reinterpret_cast<uint32_t*>(C) = (uint32_t)h0 | ((uint32_t)h1 << 16);
    else C[0] = h0;
}

__device__ __forceinline__ void store_pair(const SkArgs& p, int row, int col, int32_t v0, int32_t v1) {
    if (row >= p.M || col >= p.N) return;
    const bool two = col + 1 < p.N;
    if (p.mode != EPI_STORE_I32) {
        const int32_t ea = p.ea[row];
        uint16_t* C = p.C + (int64_t)row * p.ldc + col;
        const bool bias = p.mode == EPI_BF16_POW2_BIAS;
        const uint16_t h0 = bias ? bf16_from_acc_pow2_bias(v0, ea, p.ew[col], p.bias[col])
                                 : bf16_from_acc_pow2(v0, ea, p.ew[col]);
        if (two) {
            const uint16_t h1 = bias ? bf16_from_acc_pow2_bias(v1, ea, p.ew[col + 1], p.bias[col + 1])
                                     : bf16_from_acc_pow2(v1, ea, p.ew[col + 1]);
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


// ---------------------------------------------------------------------------- prep
// Zeroes `zero_words` 16-byte words at Z and writes Y[r][k] = (fp16) X[r][k] for k < K,
// zero for K <= k < ldy (ldy a multiple of 8).
__global__ void __launch_bounds__(256) skinny_prep_kernel(uint4* __restrict__ Z, int64_t zero_words,
                                                          const int8_t* __restrict__ X, int64_t ldx, int rows, int K,
                                                          __half* __restrict__ Y, int64_t ldy) {
    pdl_launch_dependents();
    const int64_t nt = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t i = tid; i < zero_words; i += nt) Z[i] = make_uint4(0, 0, 0, 0);
    const int64_t nvec = ldy / 8;
    for (int64_t v = tid; v < (int64_t)rows * nvec; v += nt) {
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
        i8x4_to_f16x4(w.x, o.x, o.y);
        i8x4_to_f16x4(w.y, o.z, o.w);
        *reinterpret_cast<uint4*>(Y + r * ldy + k) = o;
    }
}

// ---------------------------------------------------------------------------- main
template <int MT>
__global__ void __launch_bounds__(SK_THREADS, sk_ctas_per_sm(MT)) skinny_kernel(const __grid_constant__ CUtensorMap tmW,
                                                               const __grid_constant__ CUtensorMap tmA,
                                                               const __grid_constant__ SkArgs p) {
    constexpr int STAGES = sk_stages(MT);
    constexpr int STAGE = sk_stage_bytes(MT);
    constexpr int ABOX = sk_a_box_bytes(MT);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE);
    uint64_t* empty = full + STAGES;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STAGES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kbr = (p.K + SK_BK - 1) / SK_BK;  // K blocks per row block
    int f0, f1;  // this CTA's range of the flattened (row block, K block) space
    if (p.parts > 0) {
        const int nb = (int)blockIdx.x / p.parts, z = (int)blockIdx.x - nb * p.parts;
        f0 = nb * kbr + (int)(((long long)z * kbr) / p.parts);
        f1 = nb * kbr + (int)(((long long)(z + 1) * kbr) / p.parts);
    } else {
        const long long F = (long long)p.nblocks * kbr;
        const long long P = gridDim.x;
        f0 = (int)(((long long)blockIdx.x * F) / P);
        f1 = (int)(((long long)(blockIdx.x + 1) * F) / P);
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, SK_CONSUMERS);
        }
        *abort_flag = 0;
        fence_mbar_init();
        pdl_launch_dependents();  // the finish kernel may be scheduled; it waits for this grid
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tmW);
            prefetch_tmap(&tmA);
            const uint64_t stream_policy = l2_policy_evict_first();
            // W does not depend on the prep kernel: the first ring's worth of W boxes is
            // issued before waiting for it, their A boxes after
            const int pre = (f1 - f0) < STAGES ? (f1 - f0) : STAGES;
            for (int i = 0; i < pre; ++i) {
                const int f = f0 + i;
                const int nb = f / kbr, kb = f - nb * kbr;
                mbar_arrive_expect_tx(full + i, STAGE);
                tma_load_2d_hint(smem + i * STAGE, &tmW, full + i, kb * SK_BK, nb * SK_ROWS, stream_policy);
            }
            pdl_wait();
            for (int i = 0; i < pre; ++i) {
                const int kb = (f0 + i) % kbr;
                uint8_t* a = smem + i * STAGE + SK_W_BYTES;
                tma_load_2d(a, &tmA, full + i, kb * SK_BK, 0);
                tma_load_2d(a + ABOX, &tmA, full + i, kb * SK_BK + 64, 0);
            }
            int stage = pre == STAGES ? 0 : pre;
            uint32_t phase = pre == STAGES ? 1u : 0u;
            uint32_t issued = pre;
            bool ok = true;
            for (int f = f0 + pre; f < f1; ++f) {
                if (!mbar_wait(empty + stage, phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const int nb = f / kbr, kb = f - nb * kbr;
                uint8_t* st = smem + stage * STAGE;
                mbar_arrive_expect_tx(full + stage, STAGE);
                tma_load_2d_hint(st, &tmW, full + stage, kb * SK_BK, nb * SK_ROWS, stream_policy);
                tma_load_2d(st + SK_W_BYTES, &tmA, full + stage, kb * SK_BK, 0);
                tma_load_2d(st + SK_W_BYTES + ABOX, &tmA, full + stage, kb * SK_BK + 64, 0);
                ++issued;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                uint32_t n = issued < (uint32_t)STAGES ? issued : (uint32_t)STAGES;
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
        return;
    }

    // ---------------------------------------------------------------- consumers
    pdl_wait();                      // the workspace is zeroed before any atomic below
    const int cw = warp - 1;         // rows [SK_RPW cw, +SK_RPW) of the row block
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
        int32_t acc[MT][SK_NJ][4];
        float accf[MT][SK_NJ][4];
#pragma unroll
        for (int a = 0; a < MT; ++a)
#pragma unroll
            for (int b = 0; b < SK_NJ; ++b)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    acc[a][b][c] = 0;
                    accf[a][b][c] = 0.f;
                }
        int since = 0;
        for (; f < fend; ++f) {
            // every lane waits (and so acquires the TMA-written bytes) itself
            const bool got = __all_sync(0xffffffffu, mbar_wait(full + stage, phase, abort_flag));
            if (!got) {
                ok = false;
                break;
            }
            const uint32_t wb = sbase + stage * STAGE;
            const uint32_t ab = wb + SK_W_BYTES;
            // lane (g, t) takes the 16-byte W chunks t and t + 4 of each 128-byte row (16 k
            // values each); the matching 16 k of A are the fp16 chunks 2t, 2t + 1 of A box `half`
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int c = t + 4 * half;
                uint32_t hw[SK_NJ][8];
#pragma unroll
                for (int j = 0; j < SK_NJ; ++j) i8x16_to_f16x16(lds16(wb + sw128(SK_RPW * cw + 8 * j + g, c)), hw[j]);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const uint32_t abox = ab + half * ABOX;
                    const uint4 x0 = lds16(abox + sw128(16 * mt + g, 2 * t));
                    const uint4 x1 = lds16(abox + sw128(16 * mt + g, 2 * t + 1));
                    const uint4 y0 = lds16(abox + sw128(16 * mt + g + 8, 2 * t));
                    const uint4 y1 = lds16(abox + sw128(16 * mt + g + 8, 2 * t + 1));
                    const uint32_t h0[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                    const uint32_t h1[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
                    // the chunk's 16 k values feed four k16 MMAs with the same k slots for A and
                    // W: logical (2t + j) <- 4q + j, (2t + 8 + j) <- 4q + 2 + j within the chunk
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t a[4] = {h0[2 * q], h1[2 * q], h0[2 * q + 1], h1[2 * q + 1]};
#pragma unroll
                        for (int j = 0; j < SK_NJ; ++j) mma_f16(accf[mt][j], a, hw[j][2 * q], hw[j][2 * q + 1]);
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
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
            if (++since == 1024 / SK_BK) {  // 1024 products per accumulator since the last drain
#pragma unroll
                for (int a = 0; a < MT; ++a)
#pragma unroll
                    for (int b = 0; b < SK_NJ; ++b)
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
            for (int b = 0; b < SK_NJ; ++b)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[a][b][c] += __float2int_rn(accf[a][b][c]);

        // exact partial of this segment -> workspace
        // accumulator (mt, j, e): row 16 mt + g (+8 for e >= 2), column 128 nb + SK_RPW cw + 8 j + 2 t (+1 odd e)
        const int nc = nb * SK_ROWS + SK_RPW * cw;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int j = 0; j < SK_NJ; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = 16 * mt + g + 8 * (e >> 1), col = nc + 8 * j + 2 * t + (e & 1);
                    if (row < p.M && col < p.N) atomicAdd(p.ws_acc + (int64_t)col * p.M + row, acc[mt][j][e]);
                }
    }
    if (!ok) {
        // let loads already issued into the ring land before the CTA's shared memory goes away
        if (lane == 0) {
            int s = stage;
            uint32_t ph = phase;
            const int n = (f1 - f0) < STAGES ? (f1 - f0) : STAGES;
            for (int i = 0; i < n; ++i) {
                mbar_wait_drain(full + s, ph, kDrainLimitNs);
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------- finish
// C from the exact sums once the main kernel has completed. A block takes 32 columns: their
// sums are 32 M consecutive words of the token-contiguous workspace (read coalesced into
// shared memory), then each thread rounds two columns of one row (written coalesced).
constexpr int SKF_COLS = 32;

__global__ void __launch_bounds__(256) skinny_finish_kernel(const __grid_constant__ SkArgs p) {
    __shared__ int32_t tile[SKF_COLS][64 + 1];  // [column][token], M <= 64
    pdl_wait();
    const int c0 = blockIdx.x * SKF_COLS;
    const int ncols = min(SKF_COLS, p.N - c0);
    const int words = ncols * p.M;
    const int32_t* src = p.ws_acc + (int64_t)c0 * p.M;
    for (int i = threadIdx.x; i < words; i += blockDim.x) {
        const int c = i / p.M;
        tile[c][i - c * p.M] = __ldcg(src + i);
    }
    __syncthreads();
    const int pairs = SKF_COLS / 2;
    for (int i = threadIdx.x; i < p.M * pairs; i += blockDim.x) {
        const int row = i / pairs;
        const int c = 2 * (i - row * pairs);
        if (c < ncols) store_pair(p, row, c0 + c, tile[c][row], c + 1 < ncols ? tile[c + 1][row] : 0);
    }
}

// ---------------------------------------------------------------------------- whole K
// Decode-shaped problems with a short K and at most 16 tokens (one launch, no workspace):
// CTA b owns W rows [R b, R b + R) over the whole of K (R = 16 as launched), so its sums are
// complete inside the CTA. Warp 0, lane 0, streams per 128-wide K block one int8 box W[R x 128]
// (evict-first) and one int8 box A[M x 128] of the real token rows (128-byte swizzle, zero
// fill past N and K; the tile's rows M .. 15 are zeroed in shared memory once) into a ring
// of 16 stages (the whole of a K = 2048 problem in flight). The exponents the rounding needs
// are loaded into registers while W streams. The consumer warps are R / 16 row groups (16 W
// rows each; one group of 8 rows for R = 8) times four K groups: K group kg takes the K blocks
// kb = kg mod 4 (their stages, kb mod WK_STAGES, are released by its row-group warps). Both
// operands are widened to fp16 in registers and multiplied with the fp16 warp MMA into fp32
// accumulators. With K <= WK_MAX_K = 4096 a warp's K blocks hold at most 1024 k values, so
// every partial sum is an integer of magnitude <= 2^24, exact in fp32, and no int32 drain is
// needed on the way. At the end the four K groups' partials, converted to int32, meet in
// shared memory (integer sums, exact) and each row group's first warp rounds and stores them.
constexpr int WK_KG = 4;
constexpr int WK_MAX_K = WK_KG * 1024;  // longer K goes to the split kernel (all SMs share K)
constexpr int WK_STAGES = 16;           // the whole of a K = 2048 problem in flight

// Geometry by the number of W rows per CTA (32, 16 or 8): RG row groups of consumer warps,
// each over NJ 8-row MMA tiles, times WK_KG K groups.
template <int ROWS>
struct WkGeo {
    static_assert(ROWS == 32 || ROWS == 16 || ROWS == 8, "rows per CTA");
    static constexpr int RG = ROWS >= 16 ? ROWS / 16 : 1;
    static constexpr int NJ = ROWS >= 16 ? 2 : 1;
    static constexpr int CONSUMERS = RG * WK_KG;
    static constexpr int THREADS = 32 * (1 + CONSUMERS);
    static constexpr int W_BYTES = ROWS * 128;
    static constexpr int A_BYTES = 16 * 128;  // one 16-token tile
    static constexpr int STAGE = W_BYTES + A_BYTES;
    static constexpr int RED_BYTES = CONSUMERS * 32 * NJ * 4 * 4;
    static constexpr int SMEM = (WK_STAGES * STAGE > RED_BYTES ? WK_STAGES * STAGE : RED_BYTES) + 1024 + 512;
    static constexpr int PER_SM = 227 * 1024 / SMEM < 8 ? 227 * 1024 / SMEM : 8;
};

template <int ROWS>
__global__ void __launch_bounds__(WkGeo<ROWS>::THREADS, WkGeo<ROWS>::PER_SM)
    skinny_wk_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ SkArgs p) {
    using G = WkGeo<ROWS>;
    constexpr int STAGE = G::STAGE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (G::SMEM - 1024 - 512));
    uint64_t* empty = full + WK_STAGES;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + WK_STAGES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkb = (p.K + 127) / 128;
    const int row0 = blockIdx.x * ROWS;
    if (threadIdx.x == 0) {
        for (int s = 0; s < WK_STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, G::RG);  // the row-group warps of the stage's K group
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    // The CTA's W rows go to L2 at once (DRAM latency paid once, not per ring refill), and the
    // next call may be scheduled now: it runs this same prologue while this grid works, so
    // that back-to-back calls keep HBM busy across the launch boundary.
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmW);
        for (int kb = 0; kb < nkb; ++kb) tma_prefetch_2d(&tmW, kb * 128, row0);
        pdl_launch_dependents();
    }
    // the A box holds the M real token rows only, so the tile's rows M .. 15 of every stage
    // are zeroed once here and never written by the TMA
    const int a_rows = p.M;
    if (a_rows < 16) {
        const int words = (16 - a_rows) * 8;  // 16-byte words of one stage's unused rows
        for (int i = threadIdx.x; i < WK_STAGES * words; i += G::THREADS) {
            const int st = i / words, w = i - st * words;
            sts16(smem_addr(smem + st * STAGE + G::W_BYTES + a_rows * 128) + 16u * (uint32_t)w, 0u, 0u, 0u, 0u);
        }
    }
    __syncthreads();
    // launched as a programmatic dependent of the kernel before it: apart from the L2 hints
    // above, nothing below touches global memory before that kernel has completed
    pdl_wait();

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tmA);
            const uint64_t stream_policy = l2_policy_evict_first();
            bool ok = true;
            int kb = 0;
            for (; kb < nkb; ++kb) {
                const int st = kb % WK_STAGES;
                if (kb >= WK_STAGES && !mbar_wait(empty + st, ((kb / WK_STAGES) - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                uint8_t* d = smem + st * STAGE;
                mbar_arrive_expect_tx(full + st, G::W_BYTES + a_rows * 128);
                tma_load_2d_hint(d, &tmW, full + st, kb * 128, row0, stream_policy);
                tma_load_2d(d + G::W_BYTES, &tmA, full + st, kb * 128, 0);
            }
            if (!ok) {
                // let the loads already issued land before the CTA's shared memory goes away
                for (int i = kb - 1; i >= 0 && i >= kb - WK_STAGES; --i)
                    mbar_wait_drain(full + i % WK_STAGES, (i / WK_STAGES) & 1u, kDrainLimitNs);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int rg = cw % G::RG, kg = cw / G::RG;
    const int g = lane >> 2, t = lane & 3;
    const int wr0 = 8 * G::NJ * rg;  // this row group's first W row in the CTA
    // the epilogue's operands, loaded now by the warps that store (K group 0) so that their
    // latency hides behind the main loop: the exponents of this lane's token rows and W columns
    // (and the bias bits)
    int32_t pre_ea[2], pre_ew[G::NJ][2];
    uint32_t pre_b[G::NJ][2];
    if (kg == 0) {
        const bool bf = p.mode != EPI_STORE_I32, bi = p.mode == EPI_BF16_POW2_BIAS;
#pragma unroll
        for (int h = 0; h < 2; ++h) pre_ea[h] = bf && g + 8 * h < p.M ? __ldg(p.ea + g + 8 * h) : 0;
#pragma unroll
        for (int j = 0; j < G::NJ; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int c = row0 + wr0 + 8 * j + 2 * t + e;
                pre_ew[j][e] = bf && c < p.N ? __ldg(p.ew + c) : 0;
                pre_b[j][e] = bi && c < p.N ? (uint32_t)__ldg(p.bias + c) : 0u;
            }
    }
    const uint32_t sbase = smem_addr(smem);
    float accf[G::NJ][4];
#pragma unroll
    for (int b = 0; b < G::NJ; ++b)
#pragma unroll
        for (int c = 0; c < 4; ++c) accf[b][c] = 0.f;
    bool ok = true;
    for (int kb = kg; kb < nkb; kb += WK_KG) {
        const int st = kb % WK_STAGES;
        const bool got = __all_sync(0xffffffffu, mbar_wait(full + st, (kb / WK_STAGES) & 1u, abort_flag));
        if (!got) {
            ok = false;
            break;
        }
        const uint32_t wb = sbase + st * STAGE;
        const uint32_t ab = wb + G::W_BYTES;
        // lane (g, t) takes the 16-byte chunks t and t + 4 of each 128-byte row (16 k values
        // each) of W and of A alike, so both operands see the same k order
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int c = t + 4 * half;
            uint32_t hw[G::NJ][8];
#pragma unroll
            for (int j = 0; j < G::NJ; ++j) i8x16_to_f16x16(lds16(wb + sw128(wr0 + 8 * j + g, c)), hw[j]);
            uint32_t h0[8], h1[8];
            i8x16_to_f16x16(lds16(ab + sw128(g, c)), h0);
            i8x16_to_f16x16(lds16(ab + sw128(g + 8, c)), h1);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t a[4] = {h0[2 * q], h1[2 * q], h0[2 * q + 1], h1[2 * q + 1]};
#pragma unroll
                for (int j = 0; j < G::NJ; ++j) mma_f16(accf[j], a, hw[j][2 * q], hw[j][2 * q + 1]);
            }
        }
        // generic-proxy reads of the stage ordered before its release to the TMA refill
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + st);
    }

    // The K groups' partials meet in the ring: every consumer is past its last stage, so
    // every load into it has landed (unless a wait gave up, which raised the abort flag and
    // the device status; then nothing is stored). Layout [warp][element][lane].
    asm volatile("bar.sync 1, %0;" ::"r"(G::CONSUMERS * 32) : "memory");
    int32_t* red = reinterpret_cast<int32_t*>(smem);
#pragma unroll
    for (int j = 0; j < G::NJ; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) red[(cw * (G::NJ * 4) + j * 4 + c) * 32 + lane] = __float2int_rn(accf[j][c]);
    asm volatile("bar.sync 1, %0;" ::"r"(G::CONSUMERS * 32) : "memory");
    if (kg != 0 || !ok || *abort_flag) return;
    // accumulator (j, c): token g (+8 for c >= 2), W row wr0 + 8 j + 2 t (+1 for odd c)
#pragma unroll
    for (int j = 0; j < G::NJ; ++j) {
        int32_t v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int e = j * 4 + c;
            int32_t sum = 0;
#pragma unroll
            for (int k = 0; k < WK_KG; ++k) sum += red[((rg + G::RG * k) * (G::NJ * 4) + e) * 32 + lane];
            v[c] = sum;
        }
        const int col = row0 + wr0 + 8 * j + 2 * t;
        store_pair_pre(p, g, col, v[0], v[1], pre_ea[0], pre_ew[j][0], pre_ew[j][1], pre_b[j][0], pre_b[j][1]);
        store_pair_pre(p, g + 8, col, v[2], v[3], pre_ea[1], pre_ew[j][0], pre_ew[j][1], pre_b[j][0], pre_b[j][1]);
    }
}
// launch with the programmatic-stream-serialization attribute (may overlap the kernel before)
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

std::mutex g_sk_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_sk_encode = nullptr;

// 2-D map over a row-major matrix [rows x cols] of `esize`-byte elements with row stride
// `ld` elements; box {128 bytes, box_rows}, 128-byte swizzle, zero fill out of bounds
cudaError_t sk_map(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, int cols, int64_t ld,
                   int rows, int box_rows) {
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
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * (cuuint64_t)esize};
    cuuint32_t box[2] = {(cuuint32_t)(128 / esize), (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_sk_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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

int g_sk_per_sm[64][5];  // resident CTAs per SM of skinny_kernel<MT>, per device (0 = not set up)

template <int MT>
cudaError_t sk_launch_mt(const CUtensorMap& tmW, const CUtensorMap& tmA, const SkArgs& a, cudaStream_t s) {
    const int smem = sk_smem_bytes(MT);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int per_sm;
    {
        // set up once per device: the shared-memory opt-in and the resident CTAs per SM
        std::lock_guard<std::mutex> lock(g_sk_mutex);
        per_sm = g_sk_per_sm[dev][MT];
        if (per_sm == 0) {
            e = cudaFuncSetAttribute(skinny_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            // persistent: every CTA resident at once (sk_ctas_per_sm per SM), each streaming an equal share
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, skinny_kernel<MT>, SK_THREADS, (size_t)smem);
            if (e != cudaSuccess) return e;
            if (per_sm < 1) return cudaErrorInvalidConfiguration;
            if (per_sm > sk_ctas_per_sm(MT)) per_sm = sk_ctas_per_sm(MT);
            g_sk_per_sm[dev][MT] = per_sm;
        }
    }
    const long long blocks = (long long)a.nblocks * ((a.K + SK_BK - 1) / SK_BK);
    long long grid = (long long)per_sm * sk_num_sms();
    if (grid > blocks) grid = blocks;
    if (a.parts > 0) grid = (long long)a.nblocks * a.parts;  // one CTA per (row block, K part)
    e = launch_pdl(skinny_kernel<MT>, dim3((unsigned)grid), dim3(SK_THREADS), (size_t)smem, s, tmW, tmA, a);
    if (e != cudaSuccess) return e;
    const unsigned fblocks = (unsigned)((a.N + SKF_COLS - 1) / SKF_COLS);
    return launch_pdl(skinny_finish_kernel, dim3(fblocks), dim3(256), 0, s, a);
}

int g_wk_set[64][3];  // skinny_wk_kernel<ROWS> opted into its shared memory, per device

template <int ROWS>
cudaError_t wk_launch_rows(const CUtensorMap& tmW, const CUtensorMap& tmA, const SkArgs& a, cudaStream_t s) {
    using G = WkGeo<ROWS>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const int gi = ROWS == 32 ? 0 : (ROWS == 16 ? 1 : 2);
    {
        std::lock_guard<std::mutex> lock(g_sk_mutex);
        if (!g_wk_set[dev][gi]) {
            e = cudaFuncSetAttribute(skinny_wk_kernel<ROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
            if (e != cudaSuccess) return e;
            g_wk_set[dev][gi] = 1;
        }
    }
    cudaError_t le = launch_pdl(skinny_wk_kernel<ROWS>, dim3((unsigned)((a.N + ROWS - 1) / ROWS)), dim3(G::THREADS),
                                (size_t)G::SMEM, s, tmW, tmA, a);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}


// ---------------------------------------------------------------------------- tensor-core decode
// Decode-shaped problems with K <= DT_MAX_K on the fifth-generation tensor cores. The W rows
// are the 128-row operand of tcgen05.mma (M = 128) and the tokens the narrow one (N = 16 MT),
// so even one token wastes no multiply-add lanes on W: D[128 x 16 MT] += W[128 x 16] T[16 MT x 16]^T,
// fp16 operands (exact for int8), fp32 accumulation in TMEM. Every partial sum of at most 1024
// products of magnitude <= 2^14 is an integer below 2^24, so each 1024-K chunk accumulates
// exactly in its own TMEM columns and the chunks are added as int32 at the end.
// The widened W operand lives in tensor memory (the MMA reads A from TMEM): thread r of a
// converter warp owns W row r, which is TMEM lane r, and stores its widened row there, so W
// crosses shared memory once (its int8 TMA stage) instead of three times; shared memory
// bandwidth, not HBM, bounded the form that staged fp16 W tiles in shared memory.
// The K blocks (128 wide) of each 128-row block of W are cut into `parts` contiguous ranges,
// one per CTA of a thread-block cluster of `parts` CTAs. Every CTA writes its int32 partial
// sums into its shared memory; CTA z then reads, through distributed shared memory, the
// partials of its slice of the 128 rows from every CTA of the cluster (16 bytes at a time),
// adds them (integer addition: the order cannot change the sum) and rounds.
// Roles (576 threads, one CTA per SM):
//   warp 0     lane 0 streams, per K block, the int8 boxes W[128 x 128] (evict-first: W is
//              read once) and T[16 MT x 128] (128-byte swizzle; zeros past N, M and K) into a
//              ring of dt_s8(MT) stages;
//   warp 1     allocates TMEM; lane 0 issues the MMAs (eight K = 16 steps per K block, A from
//              TMEM, B from shared memory) and commits each stage back to the converters;
//   warps 2-17 widen each stage exactly to fp16: warp w takes W rows 32 (w mod 4) .. +31 (its
//              TMEM lanes) over K quarter (w - 2) / 4 into one of DT_SW TMEM stages, and one
//              16-byte chunk of the token box per thread into a shared-memory tcgen05 operand
//              tile (K-major, 128-byte swizzle: chunk c of row r at c ^ (r mod 8)). They stage
//              the exponents of the outputs in shared memory while the stream runs; once the
//              MMAs are done, warp w drains lanes 32 (w mod 4) .. +31 for token quarter (w - 2) / 4.
constexpr int DT_CONV_WARPS = 16;
constexpr int DT_THREADS = 64 + 32 * DT_CONV_WARPS;
constexpr int DT_MAX_K = 4096;
constexpr int DT_SW = 4;                // widened stages (W in TMEM, tokens in shared memory)
constexpr uint32_t DT_TMEM_COLS = 512;  // W stages: columns [0, 64 DT_SW); accumulators above
constexpr uint32_t DT_ACC_COL = 64 * DT_SW;
constexpr int DT_W8 = 128 * 128;  // int8 W box bytes
__host__ __device__ constexpr int dt_s8(int MT) { return MT <= 2 ? 7 : 6; }
__host__ __device__ constexpr int dt_st8_bytes(int MT) { return DT_W8 + 16 * MT * 128; }
__host__ __device__ constexpr int dt_stt_bytes(int MT) { return 2 * 16 * MT * 128; }  // fp16 token stage
constexpr int DT_EPI_BYTES = 4 * (64 + 128 + 128);  // staged ea, ew and bias of one row block
__host__ __device__ constexpr int dt_smem_bytes(int MT) {
    return dt_s8(MT) * dt_st8_bytes(MT) + DT_SW * dt_stt_bytes(MT) + DT_EPI_BYTES + 1024 + 256;
}
// more than half of an SM's shared memory: one CTA per SM, so the whole TMEM is this CTA's
static_assert(dt_smem_bytes(1) > 116 * 1024 && dt_smem_bytes(4) <= 227 * 1024, "shared memory");
static_assert(DT_ACC_COL + 4 * 64 <= DT_TMEM_COLS, "TMEM: four 1024-K chunks of 64 tokens above the W stages");

__device__ __forceinline__ int4 ld_dsmem_v4(uint32_t cluster_addr) {
    int4 v;
    asm volatile("ld.shared::cluster.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}
// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16: A is M x K with row m in TMEM lane m and
// the K values in pairs per 32-bit column (k = 2c in the low half of column c)
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}


// one output of the decode kernels: row m, column col, with its exponents (and bias) at hand
__device__ __forceinline__ void store_one(const SkArgs& p, int m, int col, int32_t v, int32_t ea, int32_t ew,
                                          uint32_t b) {
    if (p.mode == EPI_STORE_I32) {
        reinterpret_cast<int32_t*>(p.C)[(int64_t)m * p.ldc + col] = v;
        return;
    }
    uint16_t h;
    if (p.mode == EPI_BF16_POW2_BIAS) h = bf16_from_acc_pow2_bias(v, ea, ew, b);
    else if (ea >= -60 && ea <= 40 && ew >= -60 && ew <= 40) h = bf16_pow2_fast(v, ea, ew);
    else h = bf16_from_acc_pow2(v, ea, ew);
    p.C[(int64_t)m * p.ldc + col] = h;
}

template <int MT>
__global__ void __launch_bounds__(DT_THREADS, 1) decode_tc_kernel(const __grid_constant__ CUtensorMap tmW,
                                                                  const __grid_constant__ CUtensorMap tmA,
                                                                  const __grid_constant__ SkArgs p) {
    constexpr int MP = 16 * MT, S8 = dt_s8(MT), ST8 = dt_st8_bytes(MT), STT = dt_stt_bytes(MT);
    constexpr int MQ = MP / 4;  // tokens per epilogue warp
    constexpr uint32_t IDESC = idesc_f16_f32(128, MP);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ringt = smem + S8 * ST8;  // fp16 token stages
    int32_t* sea = reinterpret_cast<int32_t*>(ringt + DT_SW * STT);  // ea[0, 64), ew and bias of the rows
    int32_t* sew = sea + 64;
    uint32_t* sbias = reinterpret_cast<uint32_t*>(sew + 128);
    uint64_t* full8 = reinterpret_cast<uint64_t*>(sbias + 128);
    uint64_t* empty8 = full8 + S8;
    uint64_t* fullw = empty8 + S8;
    uint64_t* emptyw = fullw + DT_SW;
    uint64_t* accf = emptyw + DT_SW;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int P = p.parts;
    const int z = (int)cluster_ctarank();
    const int n0 = (int)(blockIdx.x / P) * 128;
    const int nkb = (p.K + 127) / 128;
    const int f0 = (int)(((long long)z * nkb) / P);
    const int nloc = (int)(((long long)(z + 1) * nkb) / P) - f0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S8; ++s) {
            mbar_init(full8 + s, 1);
            mbar_init(empty8 + s, DT_CONV_WARPS);
        }
        for (int t = 0; t < DT_SW; ++t) {
            mbar_init(fullw + t, DT_CONV_WARPS);
            mbar_init(emptyw + t, 1);  // the MMA commit
        }
        mbar_init(accf, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, DT_TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmA);
        // the CTA's W boxes go to L2 at once (DRAM latency paid once, not per ring refill)
        for (int i = 0; i < nloc; ++i) tma_prefetch_2d(&tmW, (f0 + i) * 128, n0);
        pdl_launch_dependents();  // the next call may be scheduled (it waits for this grid)
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // launched as a programmatic dependent of the kernel before it: the setup above overlaps
    // that kernel's tail; apart from the L2 hints, nothing below touches global memory before
    // it has completed
    pdl_wait();

    const bool epi = warp >= 2;
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;           // W row of this thread: its TMEM lane
    const int qk = (warp - 2) >> 2;           // K quarter of the W stages / token quarter of the drain
    const int mq0 = MQ * qk;                  // first token of this warp's quarter
    const uint32_t lane_base = tmem_base + ((uint32_t)(32 * q4) << 16);
    // the rounding's operands, staged now so that their latency hides behind the stream
    if (epi) {
        const int t = threadIdx.x - 64;
        if (t < 64) sea[t] = t < p.M && p.mode != EPI_STORE_I32 ? __ldg(p.ea + t) : 0;
        if (t < 128) {
            const bool in = n0 + t < p.N && p.mode != EPI_STORE_I32;
            sew[t] = in ? __ldg(p.ew + n0 + t) : 0;
            sbias[t] = in && p.mode == EPI_BF16_POW2_BIAS ? (uint32_t)__ldg(p.bias + n0 + t) : 0u;
        }
    }

    bool ok = true;
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int i = 0;
            for (; i < nloc; ++i) {
                const int s = i % S8;
                if (i >= S8 && !mbar_wait(empty8 + s, (uint32_t)((i / S8) - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                uint8_t* d = smem + s * ST8;
                mbar_arrive_expect_tx(full8 + s, ST8);
                const int kx = (f0 + i) * 128;
                tma_load_2d_hint(d, &tmW, full8 + s, kx, n0, pol);
                tma_load_2d(d + DT_W8, &tmA, full8 + s, kx, 0);
            }
            if (!ok) {
                // let the loads already issued land before the CTA's shared memory goes away
                for (int j = i - 1; j >= 0 && j >= i - S8; --j)
                    mbar_wait_drain(full8 + j % S8, (uint32_t)(j / S8) & 1u, kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            for (int i = 0; i < nloc; ++i) {
                const int t = i % DT_SW;
                if (!mbar_wait(fullw + t, (uint32_t)(i / DT_SW) & 1u, abort_flag)) break;
                tc_fence_after();
                const uint32_t bt = smem_addr(ringt + t * STT);
                const uint32_t d = tmem_base + DT_ACC_COL + (uint32_t)((i >> 3) * MP);  // 1024-K chunk i / 8
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t bd = sdesc_sw128_kmajor(bt + (uint32_t)((k >> 2) * MP * 128)) + 2 * (k & 3);
                    mma_f16_tmem_a(d, tmem_base + (uint32_t)(64 * t + 8 * k), bd, IDESC, ((i & 7) | k) != 0 ? 1u : 0u);
                }
                mma_commit(emptyw + t);
            }
            mma_commit(accf);  // every MMA issued above has completed when this arrives
            mbar_wait_drain(accf, 0);  // ... and before TMEM is freed, even after an abort
        }
    } else {
        // ------------------------------------------------------------ converters
        const int t = threadIdx.x - 64;  // 0 .. 511
        const int sw = row & 7;
        for (int i = 0; i < nloc; ++i) {
            const int s = i % S8, tw = i % DT_SW;
            bool got = mbar_wait(full8 + s, (uint32_t)(i / S8) & 1u, abort_flag);
            if (got && i >= DT_SW) got = mbar_wait(emptyw + tw, (uint32_t)((i / DT_SW) - 1) & 1u, abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t s8 = smem_addr(smem + s * ST8);
            // all of this thread's loads first (one latency), then the widening and the stores
            uint4 wv[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) wv[c] = lds16(s8 + (uint32_t)(row * 128 + (((2 * qk + c) ^ sw) << 4)));
            // token chunk t (row t / 8, chunk t % 8) of the MP * 8 <= 512
            constexpr int TQ = (MP * 8 + 511) / 512;
            uint4 tv[TQ];
#pragma unroll
            for (int j = 0; j < TQ; ++j) {
                const int q = t + 512 * j;
                tv[j] = make_uint4(0, 0, 0, 0);
                if (q < MP * 8) tv[j] = lds16(s8 + (uint32_t)(DT_W8 + (q >> 3) * 128 + (((q & 7) ^ ((q >> 3) & 7)) << 4)));
            }
            uint32_t h[16];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t hh[8];
                i8x16_to_f16x16(wv[c], hh);
#pragma unroll
                for (int e = 0; e < 8; ++e) h[8 * c + e] = hh[e];
            }
            tmem_st16(lane_base + (uint32_t)(64 * tw + 16 * qk), h);
#pragma unroll
            for (int j = 0; j < TQ; ++j) {
                const int q = t + 512 * j;
                const int m = q >> 3, c8 = q & 7, msw = m & 7;
                if (q < MP * 8) {
                    uint32_t hh[8];
                    i8x16_to_f16x16(tv[j], hh);
                    const uint32_t td = smem_addr(ringt + tw * STT) + (uint32_t)((c8 >> 2) * MP * 128 + m * 128);
                    const int cc = 2 * (c8 & 3);
                    sts16(td + (uint32_t)((cc ^ msw) << 4), hh[0], hh[1], hh[2], hh[3]);
                    sts16(td + (uint32_t)(((cc + 1) ^ msw) << 4), hh[4], hh[5], hh[6], hh[7]);
                }
            }
            tmem_wait_st();
            // the TMEM stores, the generic-proxy reads of the int8 stage and writes of the token
            // tile are ordered before the MMA and the TMA refill (async proxy)
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(empty8 + s);
                mbar_arrive(fullw + tw);
            }
        }
        // ------------------------------------------------------------ drain
        const bool done = mbar_wait(accf, 0, abort_flag);
        ok = __all_sync(0xffffffffu, ok && done) && *abort_flag == 0;
    }
    int32_t acc[MQ];
#pragma unroll
    for (int j = 0; j < MQ; ++j) acc[j] = 0;
    if (epi && ok) {
        tc_fence_after();
        const int nchunks = (nloc + 7) / 8;
        for (int ch = 0; ch < nchunks; ++ch) {
            // all of the chunk's loads in flight, then one wait
            uint32_t v[MQ / 4][4];
#pragma unroll
            for (int j = 0; j < MQ / 4; ++j) tmem_ld4(lane_base + DT_ACC_COL + (uint32_t)(ch * MP + mq0 + 4 * j), v[j]);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < MQ / 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[4 * j + e] += __float2int_rn(__uint_as_float(v[j][e]));
        }
    }
    tc_fence_before();
    // [token][W row] partial sums in the token ring: every MMA has completed (accf) and every
    // conversion is done, so the ring is free
    int32_t* red = reinterpret_cast<int32_t*>(ringt);
    if (epi && ok) {
#pragma unroll
        for (int j = 0; j < MQ; ++j) red[(mq0 + j) * 128 + row] = acc[j];
    }
    if (P > 1) cluster_sync();  // every CTA's partials are in place (and every CTA has started)
    else __syncthreads();
    if (epi && ok) {
        // this CTA's slice of the rows, in groups of four (one 16-byte load per CTA of the
        // cluster): rows [4 g0, 4 g1)
        const int g0 = (z * 32) / P, g1 = ((z + 1) * 32) / P, G = g1 - g0;
        const uint32_t rbase = smem_addr(red);
        for (int it = threadIdx.x - 64; it < p.M * G; it += 32 * DT_CONV_WARPS) {
            const int m = it / G, r = 4 * (g0 + it - m * G);
            const uint32_t a = rbase + (uint32_t)((m * 128 + r) * 4);
            int4 v = make_int4(0, 0, 0, 0);
            for (int zz = 0; zz < P; ++zz) {
                const int4 u = P > 1 ? ld_dsmem_v4(mapa(a, (uint32_t)zz)) : *reinterpret_cast<const int4*>(red + m * 128 + r);
                v.x += u.x;
                v.y += u.y;
                v.z += u.z;
                v.w += u.w;
            }
            const int32_t vv[4] = {v.x, v.y, v.z, v.w};
            const int col = n0 + r;
            if (col + 3 < p.N && p.mode != EPI_BF16_POW2_BIAS) {
                // four whole outputs in one store (rows of C are 16-byte aligned, col a multiple of 4)
                if (p.mode == EPI_STORE_I32) {
                    *reinterpret_cast<int4*>(reinterpret_cast<int32_t*>(p.C) + (int64_t)m * p.ldc + col) = v;
                } else {
                    const int32_t ea = sea[m];
                    int32_t ew[4];
                    bool inr = ea >= -60 && ea <= 40;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        ew[e] = sew[r + e];
                        inr = inr && ew[e] >= -60 && ew[e] <= 40;
                    }
                    uint16_t h[4];
                    // a branch, not a select: the integer form is evaluated only where needed
                    if (__all_sync(__activemask(), inr)) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) h[e] = bf16_pow2_fast(vv[e], ea, ew[e]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) h[e] = bf16_from_acc_pow2(vv[e], ea, ew[e]);
                    }
                    *reinterpret_cast<uint2*>(p.C + (int64_t)m * p.ldc + col) =
                        make_uint2((uint32_t)h[0] | ((uint32_t)h[1] << 16), (uint32_t)h[2] | ((uint32_t)h[3] << 16));
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (col + e < p.N) store_one(p, m, col + e, vv[e], sea[m], sew[r + e], sbias[r + e]);
            }
        }
    }
    if (P > 1) cluster_sync();  // no CTA leaves while another may still read its partials
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, DT_TMEM_COLS);
}

int g_dt_set[64][5];      // decode_tc_kernel<MT> opted into its shared memory, per device
int g_dt_clusters[64][5][9];  // active clusters of `parts` CTAs at once, per device and MT (0: not known)

template <int MT>
int dt_active_clusters(int parts) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(g_sk_mutex);
    if (!g_dt_set[dev][MT]) {
        if (cudaFuncSetAttribute(decode_tc_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 dt_smem_bytes(MT)) != cudaSuccess)
            return 0;
        g_dt_set[dev][MT] = 1;
    }
    if (g_dt_clusters[dev][MT][parts] == 0) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = parts;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(parts * 64, 1, 1);
        cfg.blockDim = dim3(DT_THREADS, 1, 1);
        cfg.dynamicSmemBytes = dt_smem_bytes(MT);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel<MT>, &cfg) != cudaSuccess) n = 0;
        g_dt_clusters[dev][MT][parts] = n > 0 ? n : -1;
    }
    return g_dt_clusters[dev][MT][parts];
}

// Cluster size: the largest number of K parts (<= 8, <= the K blocks) with which every row
// block's cluster is resident at once; one part when even that does not fit.
template <int MT>
int dt_parts(int nrb, int nkb) {
    for (int P = nkb < 8 ? nkb : 8; P > 1; --P) {
        const int n = dt_active_clusters<MT>(P);
        if (n > 0 && nrb <= n) return P;
    }
    return 1;
}

template <int MT>
cudaError_t dt_launch_mt(const CUtensorMap& tmW, const CUtensorMap& tmA, SkArgs a, cudaStream_t s) {
    const int nkb = (a.K + 127) / 128;
    if (dt_active_clusters<MT>(1) == 0) return cudaErrorInvalidConfiguration;
    a.parts = dt_parts<MT>(a.nblocks, nkb);
    // every 1024-K chunk of a part has MP accumulator columns above the W stages
    if (((nkb + a.parts - 1) / a.parts + 7) / 8 * 16 * MT > (int)(DT_TMEM_COLS - DT_ACC_COL)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.parts;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)(a.nblocks * a.parts), 1, 1);
    cfg.blockDim = dim3(DT_THREADS, 1, 1);
    cfg.dynamicSmemBytes = dt_smem_bytes(MT);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_tc_kernel<MT>, tmW, tmA, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool decode_path(int M, int K) {
    (void)K;
    return M <= 64;
}

size_t skinny_workspace_bytes(int M, int N, int K, int split) {
    (void)split;
    if (M == 0 || N == 0) return 0;
    return sk_layout(M, N, K).total;
}

int skinny_exact_parts(int K, int split) {
    const int kbr = (K + SK_BK - 1) / SK_BK;
    return split < kbr ? split : kbr;
}

cudaError_t skinny_launch(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw, const int32_t* ea,
                          const int32_t* ew, const uint16_t* bias, void* C, int64_t ldc, int mode, int M, int N, int K,
                          int split, void* ws, cudaStream_t s, bool exact_split) {
    // Without exact_split the kernels choose their own cut (the bits never depend on it);
    // with it, every row block of W is cut into skinny_exact_parts(K, split) contiguous K
    // parts on the split form below, whatever K is.
    if (M == 0 || N == 0) return cudaSuccess;
    if (!decode_path(M, K)) return cudaErrorInvalidValue;
    const int MT = (M + 15) / 16;
    if (K <= DT_MAX_K && MT > 1 && !exact_split) {
        // short K, 17 to 64 tokens: the tensor-core decode kernel (one launch, no workspace)
        SkArgs a = {};
        a.M = M;
        a.N = N;
        a.K = K;
        a.nblocks = (N + 127) / 128;
        a.ea = ea;
        a.ew = ew;
        a.bias = bias;
        a.C = reinterpret_cast<uint16_t*>(C);
        a.ldc = ldc;
        a.mode = mode;
        CUtensorMap tmW, tmA;
        cudaError_t e = sk_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, W, K, ldw, N, 128);
        if (e == cudaSuccess) e = sk_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A, K, lda, M, 16 * MT);
        if (e != cudaSuccess) return e;
        switch (MT) {
            case 2: return dt_launch_mt<2>(tmW, tmA, a, s);
            case 3: return dt_launch_mt<3>(tmW, tmA, a, s);
            default: return dt_launch_mt<4>(tmW, tmA, a, s);
        }
    }
    if (K <= WK_MAX_K && MT == 1 && !exact_split) {
        // short K, at most 16 tokens: one CTA per 32 W rows over the whole of K, int8 A read
        // directly (its one-launch set-up is cheaper than the tensor-core kernel's, which only
        // pays once the warp MMA work grows with the tokens)
        SkArgs a = {};
        a.M = M;
        a.N = N;
        a.K = K;
        a.ea = ea;
        a.ew = ew;
        a.bias = bias;
        a.C = reinterpret_cast<uint16_t*>(C);
        a.ldc = ldc;
        a.mode = mode;
        CUtensorMap tmW, tmA;
        // 16 W rows per CTA (up to three CTAs per SM): measured against 32 rows (two per SM) and
        // 8 rows (four per SM) on back-to-back calls at N = 6144, K = 2048: 5.16 against 5.62
        // and 8.91 us at M = 1, 5.30 against 5.82 and 8.48 us at M = 16
        constexpr int ROWS = 16;
        cudaError_t e = sk_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, W, K, ldw, N, ROWS);
        // the token box holds the M real rows (the tile's other rows stay zero in shared memory)
        if (e == cudaSuccess) e = sk_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A, K, lda, M, M);
        if (e != cudaSuccess) return e;
        return wk_launch_rows<ROWS>(tmW, tmA, a, s);
    }
    const SkLayout L = sk_layout(M, N, K);
    char* base = reinterpret_cast<char*>(ws);
    SkArgs a = {};
    a.M = M;
    a.N = N;
    a.K = K;
    a.nblocks = (N + SK_ROWS - 1) / SK_ROWS;
    a.ea = ea;
    a.ew = ew;
    a.bias = bias;
    a.C = reinterpret_cast<uint16_t*>(C);
    a.ldc = ldc;
    a.mode = mode;
    a.ws_acc = reinterpret_cast<int32_t*>(base + L.acc);
    a.parts = exact_split ? skinny_exact_parts(K, split) : 0;
    __half* A16 = reinterpret_cast<__half*>(base + L.a16);
    CUtensorMap tmW, tmA;
    cudaError_t e = sk_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, W, K, ldw, N, SK_ROWS);
    if (e == cudaSuccess) e = sk_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, A16, K, L.lda16, M, 16 * MT);
    if (e != cudaSuccess) return e;
    // prep: zero the accumulators, widen A into the workspace
    const int64_t zero_words = (int64_t)(L.a16 / 16);
    const int64_t work = zero_words + (int64_t)M * (L.lda16 / 8);
    int64_t blocks = (work + 255) / 256;
    const int64_t cap = (int64_t)sk_num_sms() * 4;
    if (blocks > cap) blocks = cap;
    skinny_prep_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<uint4*>(base), zero_words, A, lda, M, K, A16,
                                                        L.lda16);
    e = cudaGetLastError();
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
