// Internal launch interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace detgemm {

// One K segment of an integer GEMM: operand bases for A [rows x K] and W [cols x K].
// The W8A8 GEMM has one segment; an Ozaki diagonal g has g - 1 (one per slice pair).
struct Seg {
    const int8_t* A;
    const int8_t* W;
};

// EPI_BF16_POW2_BIAS: as EPI_BF16_POW2 with a bf16 bias per output column added to the
// exactly scaled accumulator before the one rounding.
enum EpilogueMode : int { EPI_BF16_POW2 = 0, EPI_STORE_I32 = 1, EPI_BF16_POW2_BIAS = 2 };

constexpr int kMaxSeg = 9;  // an Ozaki diagonal holds at most nslices (<= 9) slice pairs

struct IGemmArgs {
    Seg seg[kMaxSeg];
    int nseg;
    int64_t lda, ldw;
    int M, N, K;          // K per segment
    int split;            // number of contiguous parts of the flattened K range
    int mode;             // EpilogueMode
    const int32_t* ea;    // [M] (bf16 mode)
    const int32_t* ew;    // [N] (bf16 mode)
    const uint16_t* bias; // [N] bf16 bits (bias mode)
    void* C;              // bf16 bits or int32
    int64_t ldc;
    int32_t* ws_acc;      // [M x N] int32, zero on entry (split > 1)
    uint32_t* ws_cnt;     // one arrival counter per output tile, zero on entry (split > 1)
};

// Decode-shaped exact int8 GEMM streaming W through a TMA ring (gemm_skinny.cu), for the
// problems decode_path accepts (M <= 64); everything else runs on the tensor-core engine.
bool decode_path(int M, int K);
size_t skinny_workspace_bytes(int M, int N, int K, int split);
// exact_split: cut every 128-row block of W into exactly skinny_exact_parts(K, split)
// contiguous K parts (128-wide K blocks) instead of the kernels' own cut.
cudaError_t skinny_launch(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw, const int32_t* ea,
                          const int32_t* ew, const uint16_t* bias, void* C, int64_t ldc, int mode, int M, int N, int K,
                          int split, void* ws, cudaStream_t s, bool exact_split = false);
int skinny_exact_parts(int K, int split);
cudaError_t skinny_take_status(uint32_t* bits);

// Integer GEMM on the mma.sync int8 path (exact int32 accumulation); decode_path problems
// are routed to skinny_launch.
size_t igemm_workspace_bytes(int M, int N, int K, int split);
cudaError_t igemm_launch(const IGemmArgs& a, void* ws, cudaStream_t s);

// Pow2 quantizer and Ozaki slicer.
cudaError_t quantize_pow2_launch(const void* X, int x_dtype, int64_t ldx, int rows, int cols, int mode,
                                 int8_t* Q, int64_t ldq, int32_t* e, cudaStream_t s);
// the same integers as exact fp16 values, zero for cols <= j < ldq (the padded operand of
// the tensor-core engine; ldq a multiple of 8)
cudaError_t quantize_pow2_f16_launch(const void* X, int x_dtype, int64_t ldx, int rows, int cols, int mode,
                                     void* Q16, int64_t ldq, int32_t* e, cudaStream_t s);
// Digit planes: ROWS -> S[t][row][j] with row stride lds >= cols; COLS -> S[t][col][r] with
// column stride lds >= rows. Padding bytes up to lds are written as zero.
cudaError_t slice_rows_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, int8_t* S,
                              int64_t lds, int32_t* e, cudaStream_t s);
cudaError_t slice_cols_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, int8_t* S,
                              int64_t lds, int32_t* e, cudaStream_t s);
// the same digits as exact fp16 values (operand planes of the tensor-core engine)
cudaError_t slice_rows_f16_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, void* S,
                                  int64_t lds, int32_t* e, cudaStream_t s);
cudaError_t slice_cols_f16_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, void* S,
                                  int64_t lds, int32_t* e, cudaStream_t s);
// fp64 operands: axis 0 = rows, 1 = columns; int8 digits or exact fp16 digit values
cudaError_t slice_f64_launch(const double* X, int64_t ldx, int rows, int cols, int axis, int nslices, int8_t* S,
                             int64_t lds, int32_t* e, cudaStream_t s);
cudaError_t slice_f64_f16_launch(const double* X, int64_t ldx, int rows, int cols, int axis, int nslices, void* S,
                                 int64_t lds, int32_t* e, cudaStream_t s);

// ------------------------------------------------------------------------------------
// tcgen05 engine (gemm_tc.cu): exact int GEMM on fp16-carried operand planes.
// A planes: fp16 [a_planes][M][Kp], B planes: fp16 [b_planes][N][Kp] (Kp multiple of 64).
// Plane group d (an Ozaki diagonal; 0 for W8A8) sums segments diag_first[d] ..
// diag_first[d] + diag_nseg[d] - 1, segment s pairing A plane segA[s] with B plane segB[s].
constexpr int kTcMaxDiag = 18;
constexpr int kTcMaxSeg = 96;
constexpr int kTcMaxClusters = 128;  // CTA pairs of one launch

struct TcArgs {
    int M, N;
    int nkb;                   // 64-wide K blocks per segment (set by the launcher)
    int ndiag;
    int diag_first[kTcMaxDiag];
    int diag_nseg[kTcMaxDiag];
    int16_t segA[kTcMaxSeg];
    int16_t segB[kTcMaxSeg];
    int split;                 // contiguous parts of each group's flattened K-block range; with
                               // split > 1 the parts' exact int32 partials meet in the split
                               // workspace (one 256 x 256 slot per tile unit) and the warp that
                               // arrives last at its counter rounds the sums
    int tiles_m, tiles_n;      // set by the launcher
    // Work assignment (set by the launcher): plane group d has per_d = tiles * split units;
    // CTA pair c takes units c, c + C, ... below C * (per_d / C) (C pairs launched), and
    // the leftover unit C * (per_d / C) + extra_of[d][c] when that is >= 0 (the leftovers of
    // the groups, heaviest group first, go to the least-loaded pairs).
    int8_t extra_of[kTcMaxDiag][kTcMaxClusters];
    int group_m;               // tile rows per raster group (0: default)
    int mode;                  // EpilogueMode
    const int32_t* ea;
    const int32_t* ew;
    const uint16_t* bias;      // [N] bf16 bits (EPI_BF16_POW2_BIAS)
    void* C;                   // bf16 [M x ldc], or int32 planes [ndiag][c_plane]
    int64_t ldc;
    int64_t c_plane;           // elements between int32 output planes
    int32_t* ws_acc;           // set by the launcher (split > 1): [tile units][256][256] sums
    uint32_t* ws_cnt;          // [tile units][2 CTAs][epilogue warps] arrival counters
    int fp_mode;               // 1 / 2: the fixed-order floating-point GEMM on fp16 / bf16
                               // operands (one group, split 1, EPI_STORE_I32 layout holding fp32 bits)
    uint32_t idesc_fp;         // its MMA instruction descriptor (set by the launcher)
    int swiglu;                // 1: gated-linear-unit W8A8 -- B planes 0 (gate) and 1 (up), N
                               // outputs, each rne_bf16(SiLU(g) * u) with exponents ea + ew
                               // (gate) and ea + ewu (up)
    const int32_t* ewu;        // [N] up-projection weight exponents (swiglu)
};

int64_t tc_padded_k(int K);
size_t tc_split_bytes(int ndiag, int M, int N, int split);
// A planes [a_planes][M][lda], B planes [b_planes][N][ldb] (fp16, 16-byte aligned rows);
// the first kext columns of each row are the K extent (zeros are read beyond it)
// exact_split: run a.split parts as given (otherwise it is lowered until every part of
// every tile runs in one round of CTA pairs); split_run, if given, receives the parts run.
cudaError_t tc_gemm_launch(const TcArgs& a, const void* A16, int64_t lda, int a_planes, const void* B16, int64_t ldb,
                           int b_planes, int64_t kext, void* ws_split, cudaStream_t s, bool exact_split = false,
                           int* split_run = nullptr);
// one-thread kernel whose bounded wait on a never-arriving mbarrier expires (DEV_TIMEOUT)
cudaError_t selftest_wait_launch(uint64_t limit_ns, cudaStream_t s);
// exact int8 -> fp16 copies of two matrices in one launch (row strides Kp0, Kp1 multiples
// of 16, zero beyond K)
cudaError_t widen_pair_launch(const int8_t* X0, int64_t ldx0, int rows0, int K0, void* Y0, int64_t Kp0,
                              const int8_t* X1, int64_t ldx1, int rows1, int K1, void* Y1, int64_t Kp1,
                              cudaStream_t s);
// exact int8 -> fp16 copy of X [rows x K] into Y [rows x Kp], zero beyond K
cudaError_t widen_i8_f16_launch(const int8_t* X, int64_t ldx, int rows, int K, void* Y, int64_t Kp,
                                cudaStream_t s);

// rne_bf16(SiLU(G 2^(ea+ewg)) * U 2^(ea+ewu)) element by element (swiglu.cu)
cudaError_t swiglu_epilogue_launch(const int32_t* G, int64_t ldg, const int32_t* U, int64_t ldu, const int32_t* ea,
                                   const int32_t* ewg, const int32_t* ewu, uint16_t* C, int64_t ldc, int M, int N,
                                   cudaStream_t s);
cudaError_t swiglu_take_status(uint32_t* bits);

// 1 when the current device is a compute-capability 10.3 GPU (checked once per device).
int device_is_supported();

// Read-and-clear accessors of the per-unit device status words.
cudaError_t quantize_take_status(uint32_t* bits);
cudaError_t slice_take_status(uint32_t* bits);
cudaError_t tc_take_status(uint32_t* bits);

// Ozaki recombination: T [max_diag - 1][M][ldT] int32, plane d holding diagonal
// g = max_diag - d (largest weight index first) -> C fp32.
cudaError_t ozaki_combine_launch(const int32_t* T, int64_t ldT, int max_diag, const int32_t* e, const int32_t* f,
                                 float* C, int64_t ldc, int M, int N, cudaStream_t s);
// the same with the result rounded to fp64 (the fp64-target scheme)
cudaError_t ozaki_combine_f64out_launch(const int32_t* T, int64_t ldT, int max_diag, const int32_t* e,
                                        const int32_t* f, double* C, int64_t ldc, int M, int N, cudaStream_t s);

}  // namespace detgemm
