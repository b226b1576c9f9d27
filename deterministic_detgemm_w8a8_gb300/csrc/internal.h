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

enum EpilogueMode : int { EPI_BF16_POW2 = 0, EPI_STORE_I32 = 1 };

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
    void* C;              // bf16 bits or int32
    int64_t ldc;
    int32_t* ws_acc;      // [M x N] int32, zero on entry (split > 1)
    uint32_t* ws_cnt;     // one arrival counter per output tile, zero on entry (split > 1)
};

// Integer GEMM on the mma.sync int8 path (exact int32 accumulation).
size_t igemm_workspace_bytes(int M, int N, int split);
cudaError_t igemm_launch(const IGemmArgs& a, void* ws, cudaStream_t s);

// Pow2 quantizer and Ozaki slicer.
cudaError_t quantize_pow2_launch(const void* X, int x_dtype, int64_t ldx, int rows, int cols, int mode,
                                 int8_t* Q, int64_t ldq, int32_t* e, cudaStream_t s);
// Digit planes: ROWS -> S[t][row][j] with row stride lds >= cols; COLS -> S[t][col][r] with
// column stride lds >= rows. Padding bytes up to lds are written as zero.
cudaError_t slice_rows_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, int8_t* S,
                              int64_t lds, int32_t* e, cudaStream_t s);
cudaError_t slice_cols_launch(const float* X, int64_t ldx, int rows, int cols, int nslices, int8_t* S,
                              int64_t lds, int32_t* e, cudaStream_t s);

// Read-and-clear accessors of the per-unit device status words.
cudaError_t quantize_take_status(uint32_t* bits);
cudaError_t slice_take_status(uint32_t* bits);

// Ozaki recombination: T [ndiag][M][ldT] int32 (diagonal g at plane g - 2) -> C fp32.
cudaError_t ozaki_combine_launch(const int32_t* T, int64_t ldT, int max_diag, const int32_t* e, const int32_t* f,
                                 float* C, int64_t ldc, int M, int N, cudaStream_t s);

}  // namespace detgemm
