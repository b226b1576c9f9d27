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
// Kernel layout: persistent clusters of two CTAs (one CTA per SM) over work units; a
// unit is (plane group d, 256 x BN output tile, split part), BN = 256, or 192 for an
// unsplit one-plane problem whose tiles all fit in one round of the clusters.
//   warp 0     TMA producer (both CTAs): CTA r loads A rows [256 tm + 128 r, +128) and B
//              rows [BN tn + BN/2 r, +BN/2) of each 64-wide K block, fp16 with the 128-byte
//              swizzle, into a 6-stage ring (32 KB or 28 KB per stage).
//   warp 1     TMEM owner (both CTAs; the pair allocates collectively) and, in the even
//              CTA, the MMA issuer: tcgen05.mma.cta_group::2 M=256 N=BN K=16, four per K
//              block, into one of two BN-column fp32 TMEM buffers, one K chunk per buffer.
//   warps 2..  epilogue (both CTAs; 8 warps of 128 columns for BN = 256, 12 of 64 for 192):
//              warp w reads TMEM lanes 32 (w % 4) .. +31 and column group (w - 2) / 4 of its
//              CTA's 128 rows, converts each fp32 chunk to int32 and adds it to its int32
//              registers; after the unit's last chunk it rounds to bf16 (or keeps int32),
//              stages its block in a 4 KB shared-memory slot and writes it with TMA stores or,
//              under split-K, adds the partial into the tile's int32 slot of the split
//              workspace with TMA reductions; the last-arriving warp reads the sums back and
//              finishes.
// Operands are fp16 planes [plane][rows][Kp] addressed through 3-D tensor maps; a unit
// walks a list of (A plane, B plane) segments: one segment for W8A8, one per slice pair
// for an Ozaki diagonal.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "silu.cuh"
#include "sm100.cuh"

namespace detgemm {

namespace {

using namespace sm100;

constexpr int BK = 64;
constexpr int SPLIT_BN = 256;  // tile width of split-K launches (and of every multi-plane launch)
constexpr uint32_t TMEM_COLS = 512;
constexpr int CHUNK_KB = 16;  // 16 blocks of 64 = 1024 K values per exact fp32 chunk

struct Unit {
    int d, tm, tn, z;  // plane group, tile row, tile column, K part
};

// tile unit j -> (plane group, tile row, tile column)
__device__ __forceinline__ void tile_of(const TcArgs& p, int j, int& d, int& tm, int& tn) {
    const int per_d = p.tiles_m * p.tiles_n;
    d = j / per_d;
    const int t = j - d * per_d;
    // grouped raster: p.group_m tile rows walk together across N for L2 reuse of B
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int gsize = min(p.tiles_m - first_m, p.group_m);
    const int in = t - g * per_group;
    tm = first_m + in % gsize;
    tn = in / gsize;
}

// unit u -> tile unit u / split (plane group major; its slot in the split workspace),
// K part u % split
__device__ __forceinline__ Unit unit_of(const TcArgs& p, int u) {
    Unit r;
    const int j = u / p.split;
    r.z = u - j * p.split;
    tile_of(p, j, r.d, r.tm, r.tn);
    return r;
}

// The i-th unit u of CTA pair cid (false past its last): each plane group in turn, its base
// units, then its leftover unit if it has one (see TcArgs::extra_of). Recomputed from i
// (one step per plane group) so that a role's loop carries one counter.
__device__ __forceinline__ bool unit_at(const TcArgs& p, int cid, int ncl, int i, int& u) {
    const int per_d = p.tiles_m * p.tiles_n * p.split;
    const int nb = per_d / ncl;
    for (int d = 0; d < p.ndiag; ++d) {
        const int x = p.extra_of[d][cid];
        if (i < nb) {
            u = d * per_d + cid + ncl * i;
            return true;
        }
        if (i == nb && x >= 0) {
            u = d * per_d + nb * ncl + x;
            return true;
        }
        i -= nb + (x >= 0);
    }
    return false;
}

__device__ __forceinline__ void kb_range(const TcArgs& p, const Unit& u, int& f0, int& f1) {
    const int F = p.diag_nseg[u.d] * p.nkb;
    f0 = (int)(((long long)u.z * F) / p.split);
    f1 = (int)(((long long)(u.z + 1) * F) / p.split);
}

// rne_bf16(acc * 2^ea * 2^ew) for exponents in [-60, 40] (so that every intermediate is
// a normal fp32 number): acc is truncated to 24 significant bits and the last kept bit is
// set when anything was dropped (rounding to odd), the scaling by powers of two is exact,
// and the final conversion rounds to nearest-even. Rounding to odd at 24 bits followed by
// rounding to nearest at 8 bits equals one rounding to nearest at 8 bits, because 24 >=
// 8 + 2; so the result is bit-identical to the integer construction of
// bf16_from_acc_pow2, at a fraction of its instruction count.
__device__ __forceinline__ float ro24_scaled(int32_t acc, float sa, float sw) {
    const float x = __int2float_rz(acc);
    const uint32_t xb = __float_as_uint(x) | (uint32_t)(__float2int_rz(x) != acc);
    return __fmul_rn(__fmul_rn(__uint_as_float(xb), sa), sw);
}

__device__ __forceinline__ float exp2_f32(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// Epilogue of a warp's 32 rows x COLS columns (COLS = 128 or 64): lane l holds row row0 + l. The results go
// through the warp's 4 KB shared-memory slot, 32 rows x 128 bytes with the 128-byte
// swizzle (16-byte chunk c of row r at c ^ (r % 8), so the eight lanes of each store phase
// hit eight different bank groups), and from there to global memory with one TMA store per
// piece (64 bf16 or 32 int32 columns); the TMA clips rows past M and columns past N. Before
// a piece overwrites the slot, the warp's previous store must have finished reading it.
// The column exponents are loaded once per warp (lane l loads columns PER l .. PER l + PER - 1,
// PER = COLS / 32, coalesced) and broadcast by shuffle.
__device__ __forceinline__ void slot_acquire(bool& pending) {
    if (pending) {
        if ((threadIdx.x & 31) == 0) bulk_wait_read_all();
        __syncwarp();
    }
}

__device__ __forceinline__ void slot_release(const CUtensorMap* tmC, uint8_t* slot, int x, int y, int z, bool live,
                                             bool& pending) {
    fence_proxy_async_smem();
    __syncwarp();
    if (live && (threadIdx.x & 31) == 0) {  // a piece wholly past M or N is not stored
        tma_store_3d(tmC, slot, x, y, z);
        bulk_commit();
    }
    pending = true;
}

__device__ __forceinline__ void st_shared16(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}


template <int COLS, bool kBias>
__device__ __forceinline__ void finish_rows(const TcArgs& p, const CUtensorMap* tmC, uint8_t* slot, int d, int row0,
                                            int col0, const int32_t (&acc)[COLS], bool& pending) {
    constexpr int PER = COLS / 32;
    const int lane = threadIdx.x & 31;
    const int row = row0 + lane;
    const uint32_t sbase = smem_addr(slot) + (uint32_t)lane * 128u;
    const int sw = lane & 7;
    if (p.mode != EPI_STORE_I32) {
        int32_t ewv[PER];
        uint32_t bv[PER];
        bool inrange = true;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int c = col0 + PER * lane + i;
            ewv[i] = c < p.N ? __ldg(p.ew + c) : 0;
            bv[i] = kBias && c < p.N ? (uint32_t)__ldg(p.bias + c) : 0u;
            inrange &= ewv[i] >= -60 && ewv[i] <= 40;
        }
        const int32_t ea = row < p.M ? __ldg(p.ea + row) : 0;
        inrange &= ea >= -60 && ea <= 40;
        const bool fast = __all_sync(0xffffffffu, inrange);  // warp-uniform choice
        float swv[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) swv[i] = exp2_f32(fast ? ewv[i] : 0);
        const float sa = exp2_f32(fast ? ea : 0);
        float bsw[PER];
        float sa_b = 0.0f;
        if constexpr (kBias) {
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const bool ok = ewv[i] >= -60 && ewv[i] <= 40 && ((bv[i] >> 7) & 0xFFu) < 191u;
                bsw[i] = ok ? exp2_f32(ewv[i]) : 0.0f;
            }
            sa_b = ea >= -60 && ea <= 40 ? exp2_f32(ea) : 0.0f;
        }
#pragma unroll
        for (int hh = 0; hh < COLS / 64; ++hh) {
            slot_acquire(pending);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = 64 * hh + 8 * jj;
                uint32_t w[4];
                if constexpr (kBias) {
                    // the fast form where the scale allows it (bsw: the column's 2^ew, or 0
                    // when its exponent or bias needs the general form; sa_b: the row's 2^ea,
                    // or 0), else the general form (its column exponent read again; 0 past N)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int c = j + 2 * i;
                        const float s0 = __shfl_sync(0xffffffffu, bsw[c % PER], c / PER);
                        const float s1 = __shfl_sync(0xffffffffu, bsw[(c + 1) % PER], (c + 1) / PER);
                        const uint32_t b0 = __shfl_sync(0xffffffffu, bv[c % PER], c / PER);
                        const uint32_t b1 = __shfl_sync(0xffffffffu, bv[(c + 1) % PER], (c + 1) / PER);
                        const float sc0 = sa_b * s0, sc1 = sa_b * s1;
                        const uint32_t u0 = acc[c] < 0 ? 0u - (uint32_t)acc[c] : (uint32_t)acc[c];
                        const uint32_t u1 = acc[c + 1] < 0 ? 0u - (uint32_t)acc[c + 1] : (uint32_t)acc[c + 1];
                        uint32_t h0, h1;
                        if (sc0 != 0.0f && u0 < (1u << 24)) {
                            h0 = bf16_from_scaled_bias_ro(acc[c], sc0, b0);
                        } else {
                            const int32_t e = col0 + c < p.N ? __ldg(p.ew + col0 + c) : 0;
                            h0 = bf16_from_acc_pow2_bias_general(acc[c], ea, e, (uint16_t)b0);
                        }
                        if (sc1 != 0.0f && u1 < (1u << 24)) {
                            h1 = bf16_from_scaled_bias_ro(acc[c + 1], sc1, b1);
                        } else {
                            const int32_t e = col0 + c + 1 < p.N ? __ldg(p.ew + col0 + c + 1) : 0;
                            h1 = bf16_from_acc_pow2_bias_general(acc[c + 1], ea, e, (uint16_t)b1);
                        }
                        w[i] = h0 | (h1 << 16);
                    }
                } else if (fast) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int c = j + 2 * i;
                        const float s0 = __shfl_sync(0xffffffffu, swv[c % PER], c / PER);
                        const float s1 = __shfl_sync(0xffffffffu, swv[(c + 1) % PER], (c + 1) / PER);
                        const __nv_bfloat162 h =
                            __floats2bfloat162_rn(ro24_scaled(acc[c], sa, s0), ro24_scaled(acc[c + 1], sa, s1));
                        w[i] = *reinterpret_cast<const uint32_t*>(&h);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int c = j + 2 * i;
                        const int32_t e0 = __shfl_sync(0xffffffffu, ewv[c % PER], c / PER);
                        const int32_t e1 = __shfl_sync(0xffffffffu, ewv[(c + 1) % PER], (c + 1) / PER);
                        w[i] = (uint32_t)bf16_from_acc_pow2(acc[c], ea, e0) |
                               ((uint32_t)bf16_from_acc_pow2(acc[c + 1], ea, e1) << 16);
                    }
                }
                st_shared16(sbase + (uint32_t)((jj ^ sw) << 4), w[0], w[1], w[2], w[3]);
            }
            slot_release(tmC, slot, col0 + 64 * hh, row0, 0, row0 < p.M && col0 + 64 * hh < p.N, pending);
        }
    } else {
#pragma unroll
        for (int pc = 0; pc < COLS / 32; ++pc) {
            slot_acquire(pending);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = 32 * pc + 4 * jj;
                st_shared16(sbase + (uint32_t)((jj ^ sw) << 4), (uint32_t)acc[j], (uint32_t)acc[j + 1],
                            (uint32_t)acc[j + 2], (uint32_t)acc[j + 3]);
            }
            slot_release(tmC, slot, col0 + 32 * pc, row0, d, row0 < p.M && col0 + 32 * pc < p.N, pending);
        }
    }
}

// Gated-linear-unit epilogue of a warp's 32 rows x 64 accumulator columns (the sixteen-warp
// geometry), which hold the gate and up accumulators of 32 outputs in turn (column 2c: gate,
// 2c + 1: up, of output column colo0 + c): each output is rne_bf16(SiLU(g) * u). The exact
// sums sit in the warp's TMEM columns at ta (written there by the caller, whose accumulator
// buffer stays held until this returns), read 16 columns at a time, so that the registers
// are free for the evaluations of eight outputs at once. A first pass takes the call-free
// tiers (bf16_silu_mul_fast) and marks what they leave undecided; a second pass reads the
// marked outputs' operands again for the out-of-line evaluations; release_buffer() hands the
// accumulator buffer back to the MMA once the operands are no longer needed. The warp's 32 x
// 32 bf16 block is staged in its slot (64-byte rows, no swizzle) and written by one TMA store.
template <typename Release>
__device__ __forceinline__ void finish_swiglu(const TcArgs& p, const CUtensorMap* tmC, uint8_t* slot, int row0,
                                              int colo0, uint32_t ta, Release release_buffer, bool& pending) {
    const int lane = threadIdx.x & 31;
    const int row = row0 + lane;
    const uint32_t sbase = smem_addr(slot) + (uint32_t)lane * 64u;
    const int c_own = colo0 + lane;  // lane l loads the exponents of output l
    const int32_t eg_own = c_own < p.N ? __ldg(p.ew + c_own) : 0;
    const int32_t eu_own = c_own < p.N ? __ldg(p.ewu + c_own) : 0;
    const int32_t ea = row < p.M ? __ldg(p.ea + row) : 0;
    // every live pair's exponents ea + ew, ea + ewu in [-60, 40], and each exponent within
    // [-120, 120] (so that 2^ea, 2^ew, 2^ewu and their products are exact fp32 numbers), lets
    // the first pass skip the per-output checks; a warp that holds any other leaves all its
    // outputs to the second pass
    const bool lr = row < p.M, lc = c_own < p.N;
    const int ea_lo = __reduce_min_sync(0xffffffffu, lr ? ea : INT_MAX);
    const int ea_hi = __reduce_max_sync(0xffffffffu, lr ? ea : INT_MIN);
    const int eg_lo = __reduce_min_sync(0xffffffffu, lc ? min(eg_own, eu_own) : INT_MAX);
    const int eg_hi = __reduce_max_sync(0xffffffffu, lc ? max(eg_own, eu_own) : INT_MIN);
    const bool general = (long long)ea_lo + eg_lo < -60 || (long long)ea_hi + eg_hi > 40 || ea_lo < -120 ||
                         ea_hi > 120 || eg_lo < -120 || eg_hi > 120;
    bool bad = false;
    uint32_t undecided = 0;  // bit c: output c is left to the second pass
    slot_acquire(pending);
    if (!general) {
        // the scales 2^ewg and 2^ewu of the warp's 32 output columns, in the slot's upper half
        // (the staged outputs take its first 2 KB), read back as broadcasts
        float* sc = reinterpret_cast<float*>(slot + 2048);
        const bool in = lc && eg_own >= -120 && eg_own <= 120 && eu_own >= -120 && eu_own <= 120;
        sc[lane] = in ? __uint_as_float((uint32_t)(eg_own + 127) << 23) : 1.0f;
        sc[32 + lane] = in ? __uint_as_float((uint32_t)(eu_own + 127) << 23) : 1.0f;
        __syncwarp();
        const float sa = lr ? __uint_as_float((uint32_t)(ea + 127) << 23) : 1.0f;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            uint32_t acc[16];  // columns 16 jj ..: the gate and up sums of outputs 8 jj .. 8 jj + 7
            tmem_ld16(ta + 16u * (uint32_t)jj, acc);
            tmem_wait_ld();
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float y[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int c = 8 * jj + 2 * i + e;
                    const float sg = __fmul_rn(sa, sc[c]);
                    const float su = __fmul_rn(sa, sc[32 + c]);
                    bool zero, ok;  // evaluated for every pair (straight-line code)
                    y[e] = silu_mul_f32_scaled((int32_t)acc[4 * i + 2 * e], (int32_t)acc[4 * i + 2 * e + 1], sg, su,
                                               zero, ok);
                    // an exact zero (g u = 0) is +0, whatever the evaluation gave (-0, or a NaN
                    // from 0 / (1 + e^-g) when e^-g overflows)
                    y[e] = zero ? 0.0f : y[e];
                    undecided |= zero || ok ? 0u : 1u << c;
                }
                // both nearest-even roundings in one conversion (outputs past M or N are computed
                // and staged too; the TMA store writes none of them)
                const __nv_bfloat162 pr = __floats2bfloat162_rn(y[0], y[1]);
                w[i] = *reinterpret_cast<const uint32_t*>(&pr);
            }
            st_shared16(sbase + (uint32_t)(jj << 4), w[0], w[1], w[2], w[3]);
        }
        // only live outputs go to the second pass
        const int live_cols = p.N - colo0;
        undecided &= !lr || live_cols <= 0 ? 0u : live_cols >= 32 ? 0xFFFFFFFFu : (1u << live_cols) - 1u;
    } else {
        const int live_cols = p.N - colo0;
        undecided = row >= p.M || live_cols <= 0 ? 0u : live_cols >= 32 ? 0xFFFFFFFFu : (1u << live_cols) - 1u;
    }
    // second pass, one output column at a time (warp-uniform). Up to four columns (nearly
    // always the case) have their operands copied into registers first, so that the buffer is
    // released before the slower evaluations; more are read from TMEM one at a time, and the
    // buffer is released after them.
    uint32_t cols = __reduce_or_sync(0xffffffffu, undecided);
    if (__popc(cols) <= 4) {
        uint32_t gv[4], uv[4];
        int cv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            cv[k] = cols != 0 ? __ffs(cols) - 1 : -1;
            gv[k] = uv[k] = 0;
            if (cols != 0) tmem_ld2(ta + 2u * (uint32_t)cv[k], gv[k], uv[k]);
            cols &= cols - 1;
        }
        tmem_wait_ld();
        release_buffer();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (cv[k] < 0) break;
            const int c = cv[k];
            const int32_t eg = __shfl_sync(0xffffffffu, eg_own, c);
            const int32_t eu = __shfl_sync(0xffffffffu, eu_own, c);
            if ((undecided >> c) & 1u) {
                const uint32_t r = bf16_silu_mul_any((int32_t)gv[k], (int32_t)uv[k], (long long)ea + eg, (long long)ea + eu);
                bad |= (r >> 16) != 0;
                st_shared_u16(sbase + 2u * (uint32_t)c, (uint16_t)r);
            }
        }
    } else {
        for (; cols != 0; cols &= cols - 1) {
            const int c = __ffs(cols) - 1;
            uint32_t g, u;
            tmem_ld2(ta + 2u * (uint32_t)c, g, u);
            tmem_wait_ld();
            const int32_t eg = __shfl_sync(0xffffffffu, eg_own, c);
            const int32_t eu = __shfl_sync(0xffffffffu, eu_own, c);
            if ((undecided >> c) & 1u) {
                const uint32_t r = bf16_silu_mul_any((int32_t)g, (int32_t)u, (long long)ea + eg, (long long)ea + eu);
                bad |= (r >> 16) != 0;
                st_shared_u16(sbase + 2u * (uint32_t)c, (uint16_t)r);
            }
        }
        release_buffer();
    }
    if (bad) raise_status(DEV_RANGE);
    slot_release(tmC, slot, colo0, row0, 0, row0 < p.M && colo0 < p.N, pending);
}

// A warp's 32 x COLS int32 partial into the split workspace (int32 [tile units x 256][256],
// row-major): 32 x 32 pieces staged in the warp's slot (128-byte swizzle) and added to
// global memory by TMA reductions.
template <int COLS>
__device__ __forceinline__ void reduce_rows(const CUtensorMap* tmS, uint8_t* slot, int wrow, int wcol,
                                            const int32_t (&acc)[COLS], bool& pending) {
    const int lane = threadIdx.x & 31;
    const uint32_t sbase = smem_addr(slot) + (uint32_t)lane * 128u;
    const int sw = lane & 7;
#pragma unroll
    for (int pc = 0; pc < COLS / 32; ++pc) {
        slot_acquire(pending);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            const int j = 32 * pc + 4 * jj;
            st_shared16(sbase + (uint32_t)((jj ^ sw) << 4), (uint32_t)acc[j], (uint32_t)acc[j + 1],
                        (uint32_t)acc[j + 2], (uint32_t)acc[j + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_reduce_add_2d(tmS, slot, wcol + 32 * pc, wrow);
            bulk_commit();
        }
        pending = true;
    }
}

// ------------------------------------------------------------------------------------
// The kernel (tcgen05 cta_group::2): a cluster of two CTAs computes a 256 x 256
// tile. CTA r of the pair holds A rows [256 tm + 128 r, +128) and B rows
// [256 tn + 128 r, +128) of every K block in its own 6-stage ring (32 KB per stage); the
// even CTA issues one M=256 N=256 K=16 MMA that reads both CTAs' halves and writes each
// CTA's 128 rows of the accumulator into that CTA's TMEM. Per SM this halves the B
// operand bytes each multiply-add needs compared with a single-CTA 128 x 256 tile.
// Synchronisation across the pair:
//   full[s]   in the even CTA: its producer arms it with both CTAs' bytes; both CTAs'
//             TMA loads complete on it (.cta_group::2 loads may signal the peer's barrier)
//   empty[s]  in both CTAs: the MMA commit arrives on both (multicast)
//   tfull[b]  in both CTAs: the MMA commit arrives on both (multicast)
//   tempty[b] in the even CTA: all 16 epilogue warps of the pair arrive on it
// ------------------------------------------------------------------------------------
// Tile geometry by tile width BN: 256 (eight epilogue warps of 32 rows x 128 columns) or
// 192 (twelve of 32 x 64), chosen by choose_bn; B rows per CTA are BN / 2. kNarrow: 256-wide
// tiles with sixteen epilogue warps of 32 x 64 and five stages (the same shared memory, 96
// registers a thread): a tile's finish runs on twice the warps, which pays where the finish
// is exposed (short K, few rounds, the biased epilogue) and costs a few per cent of the main
// loop elsewhere.
template <int BNT, bool kNarrow = false>
struct Geo {
    static constexpr int BN = BNT;
    static constexpr int COLS = BNT == 256 && !kNarrow ? 128 : 64;  // columns per epilogue warp
    static constexpr int EPI_WARPS = 4 * BNT / COLS;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int STAGES = EPI_WARPS > 12 ? 5 : 6;
    static constexpr int A_BYTES = 128 * BK * 2;
    static constexpr int B_BYTES = (BNT / 2) * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t IDESC = idesc_f16_f32(256, BNT);
    static constexpr int SLOT_BYTES = 32 * 128;  // one epilogue warp's staging slot
    static constexpr int SMEM_BYTES =
        STAGES * STAGE_BYTES + EPI_WARPS * SLOT_BYTES + 1024 /*alignment slack*/ + 256 /*barriers*/;
};
static_assert(Geo<256>::SMEM_BYTES <= 227 * 1024 && Geo<192>::SMEM_BYTES <= 227 * 1024 &&
                  Geo<256, true>::SMEM_BYTES <= 227 * 1024,
              "shared memory");

static_assert(2 * 256 <= 512 && 2 * 192 <= 512, "two accumulator buffers in TMEM");

// kSplit: the instantiation for split > 1 (the split epilogue's registers stay out of the
// other one); kGroups: several plane groups (the Ozaki diagonals), units assigned through
// TcArgs::extra_of (one group: plain round-robin, with no table walk in the loops); kBias:
// the epilogue adds a bf16 bias per column before its rounding (EPI_BF16_POW2_BIAS; its
// registers stay out of the other instantiations); kNarrow: the 256-wide geometry with
// sixteen epilogue warps; kFloat: the fixed-order floating-point GEMM -- fp16 or bf16
// operands (TcArgs::idesc_fp), the whole K range of a tile accumulated in one TMEM buffer in
// K order (no chunk drains), and the raw fp32 accumulator stored (EPI_STORE_I32 layout);
// kSwiglu: the gated-linear-unit W8A8 GEMM -- B planes 0 (gate) and 1 (up) loaded with their
// rows interleaved, each output rounded once as rne_bf16(SiLU(g) * u) (finish_swiglu; its
// instantiation is the sixteen-warp geometry, whose finish runs on twice the warps)
template <int BNT, bool kSplit, bool kGroups, bool kBias, bool kNarrow, bool kFloat = false, bool kSwiglu = false>
__global__ void __launch_bounds__(Geo<BNT, kNarrow>::THREADS, 1)
    tc2_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmS,
                    const __grid_constant__ TcArgs p) {
    typedef Geo<BNT, kNarrow> G;
    constexpr int BN = G::BN, COLS = G::COLS, EPI_WARPS = G::EPI_WARPS, P_STAGES = G::STAGES;
    constexpr int P_A_BYTES = G::A_BYTES, P_STAGE_BYTES = G::STAGE_BYTES, P_SLOT_BYTES = G::SLOT_BYTES;
    constexpr uint32_t P_IDESC = G::IDESC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* slots = smem + P_STAGES * P_STAGE_BYTES;  // epilogue staging, 1024-byte aligned
    uint64_t* full = reinterpret_cast<uint64_t*>(slots + EPI_WARPS * P_SLOT_BYTES);
    uint64_t* empty = full + P_STAGES;
    uint64_t* tfull = empty + P_STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* mdone = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdone + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cid = (int)cluster_id_x(), ncl = (int)num_clusters_x();
    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull + b, 1);
            mbar_init(tempty + b, 2 * EPI_WARPS);
        }
        mbar_init(mdone, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, TMEM_COLS);  // collective over the pair: both CTAs issue it
        tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers are initialised before any remote arrival
    tc_fence_after();
    // Launched as a programmatic dependent of the kernel before it on the stream: the setup
    // above overlaps that kernel's tail; every thread waits for its completion (and the
    // visibility of its writes: the operands, the exponents) before touching global memory.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t tmem_base = *tmem_slot;
    const int total = p.ndiag * p.tiles_m * p.tiles_n * p.split;  // one plane group: units cid, cid + ncl, ...
    const uint32_t full_lead = mapa(smem_addr(full), 0);
    const uint32_t tempty_lead = mapa(smem_addr(tempty), 0);

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0;
            bool ok = true;
            for (int i = 0, u = cid; ok && (kGroups ? unit_at(p, cid, ncl, i, u) : u < total); ++i, u += ncl) {
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
                    uint8_t* sa = smem + stage * P_STAGE_BYTES;
                    if (rank == 0) mbar_arrive_expect_tx(full + stage, 2 * P_STAGE_BYTES);
                    const uint32_t fb = full_lead + 8u * (uint32_t)stage;
                    tma_load_3d_pair(sa, &tmA, fb, kx, un.tm * 256 + (int)rank * 128, p.segA[seg]);
                    if constexpr (kSwiglu)  // rows j of the gate and up planes, interleaved (map {K, plane, row})
                        tma_load_3d_pair(sa + P_A_BYTES, &tmB, fb, kx, 0, (un.tn * BN + (int)rank * (BN / 2)) / 2);
                    else
                        tma_load_3d_pair(sa + P_A_BYTES, &tmB, fb, kx, un.tn * BN + (int)rank * (BN / 2), p.segB[seg]);
                    ++issued;
                    if (++stage == P_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && rank == 0) {
                // let the copies already in flight land before shared memory goes away
                uint32_t n = issued < P_STAGES ? issued : P_STAGES;
                int s = stage;
                uint32_t ph = phase;
                for (uint32_t i = 0; i < n; ++i) {
                    if (--s < 0) {
                        s = P_STAGES - 1;
                        ph ^= 1u;
                    }
                    mbar_wait_drain(full + s, ph);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------------------ MMA issuer (even CTA)
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t tphase = 0;
            bool ok = true;
            for (int i = 0, u = cid; ok && (kGroups ? unit_at(p, cid, ncl, i, u) : u < total); ++i, u += ncl) {
                const Unit un = unit_of(p, u);
                int f0, f1;
                kb_range(p, un, f0, f1);
                const int chunk = kFloat ? f1 - f0 : CHUNK_KB;  // kFloat: one accumulation over all of K
                for (int c0 = f0; c0 < f1 && ok; c0 += chunk) {
                    const int c1 = min(f1, c0 + chunk);
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
                        const uint32_t sa = smem_addr(smem + stage * P_STAGE_BYTES);
                        const uint64_t ad = sdesc_sw128_kmajor(sa);
                        const uint64_t bd = sdesc_sw128_kmajor(sa + P_A_BYTES);
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            mma_f16_pair(dt, ad + 2 * k, bd + 2 * k, kFloat ? p.idesc_fp : P_IDESC,
                                         (f > c0 || k > 0) ? 1u : 0u);
                        mma_commit_pair_mc(empty + stage, 0x3);
                        if (++stage == P_STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    mma_commit_pair_mc(tfull + buf, 0x3);
                    if (++buf == 2) {
                        buf = 0;
                        tphase ^= 1u;
                    }
                }
            }
            mma_commit_pair_mc(mdone, 0x1);
            mbar_wait_drain(mdone, 0);
        }
    } else {
        // ---------------------------------------------------------------- epilogue (both CTAs)
        const int ew = warp - 2;
        const int q = warp & 3;
        const int h = ew >> 2;
        uint8_t* slot = slots + ew * P_SLOT_BYTES;
        bool pending = false;  // a TMA store from this warp's slot may still be in flight
        int buf = 0;
        uint32_t tphase = 0;
        bool ok = true;
        for (int i = 0, u = cid; ok && (kGroups ? unit_at(p, cid, ncl, i, u) : u < total); ++i, u += ncl) {
            const Unit un = unit_of(p, u);
            int f0, f1;
            kb_range(p, un, f0, f1);
            int32_t acc[COLS];
#pragma unroll
            for (int i = 0; i < COLS; ++i) acc[i] = 0;
            const int chunk = kFloat ? f1 - f0 : CHUNK_KB;
            uint32_t ta_fin = 0;  // kSwiglu: the last chunk's columns, held until the finish
            int buf_fin = 0;
            for (int c0 = f0; c0 < f1; c0 += chunk) {
                const bool got = mbar_wait(tfull + buf, tphase, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + h * COLS);
                // 16 columns per load: the accumulators plus one load's registers stay within
                // the thread's register budget
#pragma unroll
                for (int j = 0; j < COLS / 16; ++j) {
                    uint32_t r[16];
                    tmem_ld16(ta + 16 * j, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        if constexpr (kFloat) acc[16 * j + i] = (int32_t)r[i];  // the fp32 bits as they are
                        else acc[16 * j + i] += __float2int_rn(__uint_as_float(r[i]));
                    }
                }
                if constexpr (kSwiglu) {
                    if (c0 + chunk >= f1) {
                        // the last chunk: the exact sums go back into the buffer's columns for the
                        // finish's second pass, which releases the buffer
                        ta_fin = ta;
                        buf_fin = buf;
#pragma unroll
                        for (int j = 0; j < COLS / 16; ++j) {
                            uint32_t v[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] = (uint32_t)acc[16 * j + i];
                            tmem_st16(ta + 16 * j, v);
                        }
                        tmem_wait_st();
                    }
                }
                if (!kSwiglu || c0 + chunk < f1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(tempty_lead + 8u * (uint32_t)buf);
                }
                if (++buf == 2) {
                    buf = 0;
                    tphase ^= 1u;
                }
            }
            if (!ok) break;
            const int row = un.tm * 256 + (int)rank * 128 + q * 32 + lane;
            const int col0 = un.tn * BN + h * COLS;
            if constexpr (!kSplit) {
                if constexpr (kSwiglu) {
                    const auto release = [&]() {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster(tempty_lead + 8u * (uint32_t)buf_fin);
                    };
                    finish_swiglu(p, &tmC, slot, row - lane, col0 / 2, ta_fin, release, pending);
                } else finish_rows<COLS, kBias>(p, &tmC, slot, un.d, row - lane, col0, acc, pending);
                continue;
            }
            // a K part: add the exact partial into the tile's slot of the split workspace with
            // TMA reductions (integer addition in L2: order-free), then count the arrival; the
            // warp that arrives last reads the complete sums back
            const int sidx = u / p.split;
            const int wrow = sidx * 256 + (int)rank * 128 + q * 32;
            reduce_rows<COLS>(&tmS, slot, wrow, h * COLS, acc, pending);
            unsigned prev = 0;
            if (lane == 0) {
                bulk_wait_all();             // the reductions have been performed
                fence_proxy_async_global();  // ... before the arrival below
                __threadfence();
                prev = atomicAdd(p.ws_cnt + ((int64_t)sidx * 2 + rank) * EPI_WARPS + ew, 1u);
            }
            pending = false;
            prev = __shfl_sync(0xffffffffu, prev, 0);
            if (prev != (unsigned)(p.split - 1)) continue;
            __threadfence();
            // lane l's row: 32 independent 16-byte loads. They go through L1, which holds no
            // copy of these lines (no one reads a slot before its sums are complete, and L1 starts
            // each launch empty), so that the four 16-byte pieces of each 128-byte line that a
            // lane reads in turn come from one L2 request.
            const int4* src = reinterpret_cast<const int4*>(p.ws_acc + (int64_t)(wrow + lane) * BN + h * COLS);
#pragma unroll
            for (int i = 0; i < COLS / 4; ++i) {
                const int4 v = __ldca(src + i);
                acc[4 * i] = v.x;
                acc[4 * i + 1] = v.y;
                acc[4 * i + 2] = v.z;
                acc[4 * i + 3] = v.w;
            }
            finish_rows<COLS, kBias>(p, &tmC, slot, un.d, row - lane, col0, acc, pending);
        }
        // the slot's last stores complete before the CTA's shared memory goes away
        if (pending && lane == 0) bulk_wait_all();
    }

    __syncwarp();
    // the next kernel on the stream may be scheduled once every CTA is here (not earlier:
    // its blocks would wait beside this kernel's and take issue slots)
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tc_fence_before();
    cluster_sync();  // no CTA leaves while its pair may still read its smem or barriers
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// ------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------
std::mutex g_tc_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

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

// 3-D map over fp16 planes [planes][rows][ld] of which the first kext columns are the
// matrix (TMA fills the box beyond kext and beyond rows with zeros), box {64, box_rows, 1},
// 128-byte swizzle
cudaError_t make_map(CUtensorMap* m, const void* base, int64_t kext, int64_t ld, int rows, int planes, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    cudaError_t e = get_encode(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[3] = {(cuuint64_t)kext, (cuuint64_t)rows, (cuuint64_t)planes};
    cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)ld * 2 * (cuuint64_t)rows};
    cuuint32_t box[3] = {(cuuint32_t)BK, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D map over two fp16 planes [2][rows][ld] read with their rows interleaved: dims {kext,
// plane, row}, box {64, 2, 64}, so that a box holds rows j of plane 0, j of plane 1, j + 1 of
// plane 0, ... (128-byte swizzle over the 128 interleaved rows)
cudaError_t make_pair_map(CUtensorMap* m, const void* base, int64_t kext, int64_t ld, int rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    cudaError_t e = get_encode(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[3] = {(cuuint64_t)kext, 2, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)ld * 2 * (cuuint64_t)rows, (cuuint64_t)ld * 2};
    cuuint32_t box[3] = {(cuuint32_t)BK, 2, 64};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D map over the output: bf16 [1][M][ldc] (box 64 x 32) or int32 planes [ndiag][M][ldc]
// spaced c_plane elements apart (box 32 x 32); 128-byte swizzle, the epilogue's slot layout
cudaError_t make_out_map(CUtensorMap* m, const TcArgs& a) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    cudaError_t e = get_encode(&enc);
    if (e != cudaSuccess) return e;
    const bool bf = a.mode != EPI_STORE_I32;
    const cuuint64_t es = bf ? 2 : 4;
    const int planes = bf ? 1 : a.ndiag;
    const cuuint64_t row_bytes = (cuuint64_t)a.ldc * es;
    const cuuint64_t plane_bytes = (planes > 1 ? (cuuint64_t)a.c_plane : (cuuint64_t)a.ldc * (cuuint64_t)a.M) * es;
    cuuint64_t dims[3] = {(cuuint64_t)a.N, (cuuint64_t)a.M, (cuuint64_t)planes};
    cuuint64_t strides[2] = {row_bytes, plane_bytes};
    // the gated-linear-unit epilogue stores 32 x 32 blocks from 64-byte slot rows
    cuuint32_t box[3] = {(cuuint32_t)(a.swiglu ? 32 : 128 / es), 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_INT32, 3, a.C, dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     a.swiglu ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

int64_t tc_padded_k(int K) { return ((int64_t)K + BK - 1) / BK * BK; }


// Split workspace: one 256 x 256 int32 slot per tile unit, then an arrival counter per tile
// unit, CTA and epilogue warp; zeroed by a memset before the engine starts. Split launches
// use 256 x 256 tiles.
constexpr size_t kSlotBytes = (size_t)256 * SPLIT_BN * sizeof(int32_t);

static size_t split_ws_bytes(int cut) {
    if (cut <= 0) return 0;
    return (size_t)cut * kSlotBytes +
           (((size_t)cut * 2 * Geo<SPLIT_BN>::EPI_WARPS * sizeof(uint32_t) + 255) & ~(size_t)255);
}

size_t tc_split_bytes(int ndiag, int M, int N, int split) {
    if (split <= 1) return 0;
    return split_ws_bytes(ndiag * ((M + 255) / 256) * ((N + SPLIT_BN - 1) / SPLIT_BN));
}

// 2-D map over the split workspace's slots: int32 [units x 256][256], box 32 x 32, the
// epilogue's slot layout (128-byte swizzle)
static cudaError_t make_ws_map(CUtensorMap* m, void* base, int cut) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    cudaError_t e = get_encode(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[2] = {SPLIT_BN, (cuuint64_t)cut * 256};
    cuuint64_t strides[1] = {SPLIT_BN * sizeof(int32_t)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {
int g_max_clusters[64][2];  // per device: 256-wide, 192-wide tiles

template <int BNT, bool kSplit, bool kGroups, bool kBias, bool kNarrow, bool kFloat = false, bool kSwiglu = false>
cudaError_t opt_in() {
    return cudaFuncSetAttribute(tc2_gemm_kernel<BNT, kSplit, kGroups, kBias, kNarrow, kFloat, kSwiglu>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, Geo<BNT, kNarrow>::SMEM_BYTES);
}

template <int BNT>
int occupancy_clusters() {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * 76, 1, 1);
    cfg.blockDim = dim3(Geo<BNT>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Geo<BNT>::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc2_gemm_kernel<BNT, false, false, false, false>, &cfg) != cudaSuccess || n <= 0) n = 1;
    return n;
}

// CTA pairs resident at once for tile width bn (256 or 192); also opts the kernels into
// their shared memory, once per device
int max_pair_clusters(int bn) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 1;
    std::lock_guard<std::mutex> lock(g_tc_mutex);
    if (g_max_clusters[dev][0] == 0) {
        if (opt_in<256, false, false, false, false>() != cudaSuccess ||
            opt_in<256, false, false, false, true>() != cudaSuccess ||
            opt_in<256, false, true, false, false>() != cudaSuccess ||
            opt_in<256, true, true, false, false>() != cudaSuccess ||
            opt_in<192, false, false, false, false>() != cudaSuccess ||
            opt_in<256, false, false, true, true>() != cudaSuccess ||
            opt_in<256, true, true, true, false>() != cudaSuccess ||
            opt_in<192, false, false, true, false>() != cudaSuccess ||
            opt_in<256, false, false, false, false, true>() != cudaSuccess ||
            opt_in<256, false, false, false, true, false, true>() != cudaSuccess)
            return 0;
        g_max_clusters[dev][0] = occupancy_clusters<256>();
        g_max_clusters[dev][1] = occupancy_clusters<192>();
    }
    return g_max_clusters[dev][bn == 256 ? 0 : 1];
}
}  // namespace

static void set_tiles(TcArgs& a, int64_t kext, int bn) {
    a.tiles_m = (a.M + 255) / 256;
    a.tiles_n = (a.N + bn - 1) / bn;
    a.nkb = (int)((kext + BK - 1) / BK);
    if (a.group_m <= 0) a.group_m = 8;
}

// Tile width of an unsplit one-plane launch. When every tile fits in one round of the
// clusters, the call takes about one tile's time, which 256 x 192 tiles cut by a quarter if
// they still fit in one round (the 257 x 6144 x 2048 sweep GEMM: 64 tiles of 192 columns on
// 76 pairs, 31 us against 41 us for 48 tiles of 256). Over several rounds the narrower tile
// is no help: on the 8192 x 12288 x 4096 FFN GEMM (27 rounds of 192-wide tiles against 21 of
// 256) it took 581 us against 461, the tensor pipe busy 59% of the time against 74%.
static int choose_bn(const TcArgs& a) {
    if (a.split > 1 || a.ndiag != 1) return 256;
    const int c256 = max_pair_clusters(256), c192 = max_pair_clusters(192);
    if (c256 <= 0 || c192 <= 0) return 256;
    const long long tm = (a.M + 255) / 256;
    const bool one256 = tm * ((a.N + 255) / 256) <= c256;
    const bool one192 = tm * ((a.N + 191) / 192) <= c192;
    return one256 && one192 ? 192 : 256;
}

// Leftover units of each plane group (per_d mod C of them) to CTA pairs: the groups in
// order (the Ozaki diagonals come heaviest first), each leftover to the pair with the least
// work so far (ties: the lowest index), at most one per pair and group. Work is counted in
// segments (a unit of group d reads diag_nseg[d] plane pairs). For a single group this is
// leftover k -> pair k, a plain round-robin.
static void assign_leftovers(TcArgs& a, int C) {
    memset(a.extra_of, -1, sizeof(a.extra_of));
    const int per_d = a.tiles_m * a.tiles_n * a.split;
    const int nb = per_d / C, nx = per_d % C;
    long long load[kTcMaxClusters];
    for (int c = 0; c < C; ++c) load[c] = 0;
    for (int d = 0; d < a.ndiag; ++d) {
        const long long w = a.diag_nseg[d];
        for (int c = 0; c < C; ++c) load[c] += (long long)nb * w;
        for (int k = 0; k < nx; ++k) {
            int best = -1;
            for (int c = 0; c < C; ++c)
                if (a.extra_of[d][c] < 0 && (best < 0 || load[c] < load[best])) best = c;
            a.extra_of[d][best] = (int8_t)k;
            load[best] += w;
        }
    }
}

template <int BNT, bool kSplit, bool kGroups, bool kBias, bool kNarrow, bool kFloat = false, bool kSwiglu = false>
static cudaError_t launch_engine(const TcArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                 const CUtensorMap& tmC, const CUtensorMap& tmS, int clusters, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddepcontrol.wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(Geo<BNT, kNarrow>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Geo<BNT, kNarrow>::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e =
        cudaLaunchKernelEx(&cfg, tc2_gemm_kernel<BNT, kSplit, kGroups, kBias, kNarrow, kFloat, kSwiglu>, tmA, tmB, tmC,
                           tmS, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t tc_gemm_launch(const TcArgs& a0, const void* A16, int64_t lda, int a_planes, const void* B16,
                           int64_t ldb, int b_planes, int64_t kext, void* ws_split, cudaStream_t s, bool exact_split,
                           int* split_run) {
    if (a0.M == 0 || a0.N == 0) return cudaSuccess;
    TcArgs a = a0;
    if (max_pair_clusters(256) <= 0) return cudaErrorInvalidConfiguration;
    const bool bias = a.mode == EPI_BF16_POW2_BIAS;
    if (bias && (a.ndiag != 1 || a.bias == nullptr)) return cudaErrorInvalidValue;
    // split_k is an upper bound (the bits do not depend on it): more parts than fill the CTA
    // pairs once only add rounds of partial tiles, so it is lowered until every part of every
    // tile runs in one round and each part keeps at least 256 K (measured: at 16 tiles and
    // K = 16384, 125 -> 90 us at 4 parts; at 192 tiles and K = 2048, 58 -> 291 us at 8)
    if (a.split > 1 && !exact_split) {
        const long long tiles = (long long)a.ndiag * ((a.M + 255) / 256) * ((a.N + 255) / 256);
        const int c256 = max_pair_clusters(256);
        while (a.split > 1 && (tiles * a.split > c256 || kext / a.split < 256)) --a.split;
    }
    if (split_run) *split_run = a.split;
    if (a.fp_mode && (a.split != 1 || a.ndiag != 1 || a.mode != EPI_STORE_I32)) return cudaErrorInvalidValue;
    if (a.fp_mode)  // kind::f16 with fp16 (mode 1) or bf16 (mode 2) operands, fp32 accumulator
        a.idesc_fp = Geo<256>::IDESC | (a.fp_mode == 2 ? (1u << 7) | (1u << 10) : 0u);
    if (a.swiglu && (a.split != 1 || a.ndiag != 1 || a.mode != EPI_BF16_POW2 || b_planes != 2))
        return cudaErrorInvalidValue;
    const int bn = a.fp_mode || a.swiglu || (bias && a.split > 1) ? 256 : choose_bn(a);
    set_tiles(a, kext, bn);
    if (a.swiglu) a.tiles_n = (a.N + 127) / 128;  // 128 outputs (256 interleaved B rows) per tile
    CUtensorMap tmA, tmB, tmC;
    cudaError_t e = make_map(&tmA, A16, kext, lda, a.M, a_planes, 128);
    if (e == cudaSuccess)
        e = a.swiglu ? make_pair_map(&tmB, B16, kext, ldb, a.N) : make_map(&tmB, B16, kext, ldb, a.N, b_planes, bn / 2);
    if (e == cudaSuccess) e = make_out_map(&tmC, a);
    if (e != cudaSuccess) return e;
    int clusters = max_pair_clusters(bn);
    if (clusters <= 0) return cudaErrorInvalidConfiguration;
    const int total = a.ndiag * a.tiles_m * a.tiles_n * a.split;
    CUtensorMap tmS;
    memset(&tmS, 0, sizeof(tmS));
    if (a.split > 1) {  // every tile unit in `split` K parts, one slot each
        const int cut = a.ndiag * a.tiles_m * a.tiles_n;
        a.ws_acc = reinterpret_cast<int32_t*>(ws_split);
        a.ws_cnt = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(ws_split) + (size_t)cut * kSlotBytes);
        e = make_ws_map(&tmS, ws_split, cut);
        if (e != cudaSuccess) return e;
        e = cudaMemsetAsync(ws_split, 0, split_ws_bytes(cut), s);
        if (e != cudaSuccess) return e;
    }
    if (clusters > total) clusters = total;
    if (clusters > kTcMaxClusters) clusters = kTcMaxClusters;
    assign_leftovers(a, clusters);
    // split launches (and every multi-group launch) walk the assignment table; the one-group
    // unsplit ones keep a plain round-robin (the table walk's registers would spill there)
    // Unsplit one-group launches of 256-wide tiles take the sixteen-warp geometry where a
    // tile's finish is exposed: always for the biased epilogue; otherwise for K <= 1024 (one
    // TMEM chunk per tile) or at most 12288 K-columns per CTA pair in all (rounds x K; measured
    // from 2048 x 4096 x 1024: 38 -> 31 us to 8192 x 6144 x 2048: 158 -> 160 us).
    const long long rounds = (total + clusters - 1) / clusters;
    const bool narrow = kext <= 1024 || rounds * kext <= 12288;
    if (a.fp_mode) return launch_engine<256, false, false, false, false, true>(a, tmA, tmB, tmC, tmS, clusters, s);
    if (a.swiglu)
        return launch_engine<256, false, false, false, true, false, true>(a, tmA, tmB, tmC, tmS, clusters, s);
    if (bias && a.split > 1) return launch_engine<256, true, true, true, false>(a, tmA, tmB, tmC, tmS, clusters, s);
    if (bias && bn == 192) return launch_engine<192, false, false, true, false>(a, tmA, tmB, tmC, tmS, clusters, s);
    if (bias) return launch_engine<256, false, false, true, true>(a, tmA, tmB, tmC, tmS, clusters, s);
    if (a.split > 1) return launch_engine<256, true, true, false, false>(a, tmA, tmB, tmC, tmS, clusters, s);
    if (a.ndiag > 1) return launch_engine<256, false, true, false, false>(a, tmA, tmB, tmC, tmS, clusters, s);
    if (bn == 192) return launch_engine<192, false, false, false, false>(a, tmA, tmB, tmC, tmS, clusters, s);
    if (narrow) return launch_engine<256, false, false, false, true>(a, tmA, tmB, tmC, tmS, clusters, s);
    return launch_engine<256, false, false, false, false>(a, tmA, tmB, tmC, tmS, clusters, s);
}

// Self-check of the bounded waits: one thread waits on an mbarrier that nothing ever
// arrives on, with the given limit; the wait expires, raises DEV_TIMEOUT in this unit's
// status word and the kernel returns normally.
__global__ void selftest_wait_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, limit_ns);
}

cudaError_t selftest_wait_launch(uint64_t limit_ns, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(limit_ns);
    return cudaGetLastError();
}

DETGEMM_STATUS_ACCESSOR(tc_take_status)

}  // namespace detgemm
