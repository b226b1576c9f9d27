// C ABI of libdetgemm (declared in include/detgemm.h): argument validation, workspace
// layout and kernel dispatch. Every argument/alignment/precondition check runs on the
// host before any CUDA call, so a rejected call has no effect and launches nothing.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/detgemm.h"
#include "common.cuh"
#include "internal.h"

namespace detgemm {

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
int g_dev_cc[kMaxDevices];  // 0 = unknown, else 10 * major + minor

detgemm_status check_device_impl() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DETGEMM_ERR_UNSUPPORTED_DEVICE;
    if (dev < 0 || dev >= kMaxDevices) return DETGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_dev_cc[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return DETGEMM_ERR_UNSUPPORTED_DEVICE;
        g_dev_cc[dev] = 10 * major + minor;
    }
    return g_dev_cc[dev] == 103 ? DETGEMM_OK : DETGEMM_ERR_UNSUPPORTED_DEVICE;
}

detgemm_status check_device() { return check_device_impl(); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool aligned2(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

detgemm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DETGEMM_OK : DETGEMM_ERR_CUDA; }

// Shared validation of the integer GEMM entry points.
detgemm_status validate_igemm(const void* A, int64_t lda, const void* W, int64_t ldw, const void* C, int64_t ldc,
                              int c_elem, int M, int N, int K, int split_k, const void* ws, size_t ws_bytes) {
    if (M < 0 || N < 0 || K < 1) return DETGEMM_ERR_INVALID_ARG;
    if (K > DETGEMM_MAX_K) return DETGEMM_ERR_PRECONDITION;
    int nkb = (K + 63) / 64;
    if (split_k < 1 || split_k > nkb) return DETGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DETGEMM_OK;
    if (!A || !W || !C) return DETGEMM_ERR_INVALID_ARG;
    if (lda < K || ldw < K || ldc < N) return DETGEMM_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(W) || !aligned16(C)) return DETGEMM_ERR_ALIGNMENT;
    if ((lda % 16) != 0 || (ldw % 16) != 0 || ((ldc * c_elem) % 16) != 0) return DETGEMM_ERR_ALIGNMENT;
    size_t need = detgemm_w8a8_workspace_size(M, N, K, split_k);
    if (need > 0 && (ws == nullptr || ws_bytes < need)) return DETGEMM_ERR_WORKSPACE;
    if (need > 0 && !aligned16(ws)) return DETGEMM_ERR_ALIGNMENT;
    return DETGEMM_OK;
}

// Ozaki workspace layout (each piece 256-byte aligned):
//   DA  fp16 [nslices][M][Kp]   DB fp16 [nslices][N][Kp]   (exact digit values; Kp = K
//                                                            rounded up to 64, zero padded)
//   e   int32 [M]               f  int32 [N]
//   T   int32 [max_diag - 1][M][ldT]  (plane d = diagonal max_diag - d; ldT = N rounded up to 4)
//   split-K sums and counters of the tensor-core engine (split_k > 1)
struct OzakiLayout {
    size_t da, db, e, f, T, split, total;
    int64_t Kp, ldT;
};

OzakiLayout ozaki_layout(int M, int N, int K, int nslices, int max_diag, int split_k) {
    OzakiLayout L;
    L.Kp = tc_padded_k(K);
    L.ldT = ((int64_t)N + 3) / 4 * 4;
    size_t off = 0;
    L.da = off; off += align256((size_t)nslices * M * L.Kp * 2);
    L.db = off; off += align256((size_t)nslices * N * L.Kp * 2);
    L.e = off; off += align256((size_t)M * 4);
    L.f = off; off += align256((size_t)N * 4);
    L.T = off; off += align256((size_t)(max_diag - 1) * M * L.ldT * 4);
    L.split = off; off += align256(tc_split_bytes(max_diag - 1, M, N, split_k));
    L.total = off;
    return L;
}

}  // namespace

int device_is_supported() { return check_device_impl() == DETGEMM_OK; }

}  // namespace detgemm

using namespace detgemm;

extern "C" {

const char* detgemm_status_string(detgemm_status s) {
    switch (s) {
        case DETGEMM_OK: return "DETGEMM_OK";
        case DETGEMM_ERR_INVALID_ARG: return "DETGEMM_ERR_INVALID_ARG";
        case DETGEMM_ERR_ALIGNMENT: return "DETGEMM_ERR_ALIGNMENT";
        case DETGEMM_ERR_PRECONDITION: return "DETGEMM_ERR_PRECONDITION";
        case DETGEMM_ERR_WORKSPACE: return "DETGEMM_ERR_WORKSPACE";
        case DETGEMM_ERR_UNSUPPORTED_DEVICE: return "DETGEMM_ERR_UNSUPPORTED_DEVICE";
        case DETGEMM_ERR_CUDA: return "DETGEMM_ERR_CUDA";
        case DETGEMM_ERR_TIMEOUT: return "DETGEMM_ERR_TIMEOUT";
        case DETGEMM_ERR_NONFINITE: return "DETGEMM_ERR_NONFINITE";
        case DETGEMM_ERR_RANGE: return "DETGEMM_ERR_RANGE";
    }
    return "DETGEMM_ERR_UNKNOWN";
}

int detgemm_version(void) { return 100; }

// Decode-shaped problems (decode_path: M <= 64) stream W
// through the register-fed warp-MMA kernels; everything larger runs on the tcgen05 engine
// over exact fp16 copies of the operands.
static bool w8a8_uses_tc(int M, int K) { return !decode_path(M, K); }

// tcgen05 path scratch: A16 [M][Kp] fp16 | W16 [N][Kp] fp16 | split-K sums and counters
struct TcW8a8Layout {
    int64_t Kp;
    size_t a16, w16, split, total;
};

static TcW8a8Layout tc_w8a8_layout(int M, int N, int K, int split_k) {
    TcW8a8Layout L;
    L.Kp = tc_padded_k(K);
    size_t off = 0;
    L.a16 = off; off += align256((size_t)M * L.Kp * 2);
    L.w16 = off; off += align256((size_t)N * L.Kp * 2);
    L.split = off; off += align256(tc_split_bytes(1, M, N, split_k));
    L.total = off;
    return L;
}

size_t detgemm_w8a8_workspace_size(int M, int N, int K, int split_k) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    if (w8a8_uses_tc(M, K)) return tc_w8a8_layout(M, N, K, split_k).total;
    return igemm_workspace_bytes(M, N, K, split_k);
}

static detgemm_status run_tc(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw, const int32_t* ea,
                             const int32_t* ew, const uint16_t* bias, void* C, int64_t ldc, int mode, int M, int N, int K, int split_k,
                             void* ws, cudaStream_t stream, bool exact_split, int* parts_run) {
    const TcW8a8Layout L = tc_w8a8_layout(M, N, K, split_k);
    char* base = reinterpret_cast<char*>(ws);
    cudaError_t e = widen_pair_launch(A, lda, M, K, base + L.a16, L.Kp, W, ldw, N, K, base + L.w16, L.Kp, stream);
    if (e != cudaSuccess) return DETGEMM_ERR_CUDA;
    TcArgs a = {};
    a.M = M;
    a.N = N;
    a.ndiag = 1;
    a.diag_first[0] = 0;
    a.diag_nseg[0] = 1;
    a.segA[0] = 0;
    a.segB[0] = 0;
    a.split = split_k;
    a.mode = mode;
    a.ea = ea;
    a.ew = ew;
    a.bias = bias;
    a.C = C;
    a.ldc = ldc;
    a.c_plane = 0;
    return from_cuda(tc_gemm_launch(a, base + L.a16, L.Kp, 1, base + L.w16, L.Kp, 1, L.Kp, base + L.split, stream,
                                    exact_split, parts_run));
}

// exact_split: run exactly the split_k contiguous K parts asked for (or, on the decode path,
// skinny_exact_parts of them) instead of the launchers' own choice; parts_run (optional)
// receives the number of parts run.
static detgemm_status run_igemm(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw, const int32_t* ea,
                                const int32_t* ew, const uint16_t* bias, void* C, int64_t ldc, int mode, int M, int N, int K, int split_k,
                                void* ws, cudaStream_t stream, bool exact_split = false, int* parts_run = nullptr) {
    if (w8a8_uses_tc(M, K))
        return run_tc(A, lda, W, ldw, ea, ew, bias, C, ldc, mode, M, N, K, split_k, ws, stream, exact_split, parts_run);
    if (exact_split) {
        if (parts_run) *parts_run = skinny_exact_parts(K, split_k);
        return from_cuda(skinny_launch(A, lda, W, ldw, ea, ew, bias, C, ldc, mode, M, N, K, split_k, ws, stream, true));
    }
    if (parts_run) *parts_run = 0;  // the decode kernels' own cut
    IGemmArgs a = {};
    a.seg[0] = Seg{A, W};
    a.nseg = 1;
    a.lda = lda;
    a.ldw = ldw;
    a.M = M;
    a.N = N;
    a.K = K;
    a.split = split_k;
    a.mode = mode;
    a.ea = ea;
    a.ew = ew;
    a.bias = bias;
    a.C = C;
    a.ldc = ldc;
    return from_cuda(igemm_launch(a, ws, stream));
}

static detgemm_status w8a8_impl(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw, const int32_t* ea,
                                const int32_t* ew, const uint16_t* bias, bool with_bias, uint16_t* C, int64_t ldc,
                                int M, int N, int K, int split_k, void* ws, size_t ws_bytes,
                                detgemm_stream_t stream, bool exact_split = false, int* parts_run = nullptr) {
    detgemm_status st = validate_igemm(A, lda, W, ldw, C, ldc, 2, M, N, K, split_k, ws, ws_bytes);
    if (st != DETGEMM_OK) return st;
    if (M == 0 || N == 0) return DETGEMM_OK;
    if (!ea || !ew || (with_bias && !bias)) return DETGEMM_ERR_INVALID_ARG;
    if (!aligned4(ea) || !aligned4(ew) || (with_bias && !aligned2(bias))) return DETGEMM_ERR_ALIGNMENT;
    if ((st = check_device()) != DETGEMM_OK) return st;
    return run_igemm(A, lda, W, ldw, ea, ew, with_bias ? bias : nullptr, C, ldc,
                     with_bias ? EPI_BF16_POW2_BIAS : EPI_BF16_POW2, M, N, K, split_k, ws,
                     reinterpret_cast<cudaStream_t>(stream), exact_split, parts_run);
}

detgemm_status detgemm_w8a8(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw, const int32_t* ea,
                            const int32_t* ew, uint16_t* C, int64_t ldc, int M, int N, int K, int split_k, void* ws,
                            size_t ws_bytes, detgemm_stream_t stream) {
    return w8a8_impl(A, lda, W, ldw, ea, ew, nullptr, false, C, ldc, M, N, K, split_k, ws, ws_bytes, stream);
}

detgemm_status detgemm_w8a8_split_exact(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw,
                                        const int32_t* ea, const int32_t* ew, uint16_t* C, int64_t ldc, int M, int N,
                                        int K, int split_k, void* ws, size_t ws_bytes, int* parts_run,
                                        detgemm_stream_t stream) {
    if (parts_run) *parts_run = 0;
    return w8a8_impl(A, lda, W, ldw, ea, ew, nullptr, false, C, ldc, M, N, K, split_k, ws, ws_bytes, stream, true,
                     parts_run);
}

detgemm_status detgemm_w8a8_bias(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw, const int32_t* ea,
                                 const int32_t* ew, const uint16_t* bias, uint16_t* C, int64_t ldc, int M, int N,
                                 int K, int split_k, void* ws, size_t ws_bytes, detgemm_stream_t stream) {
    return w8a8_impl(A, lda, W, ldw, ea, ew, bias, true, C, ldc, M, N, K, split_k, ws, ws_bytes, stream);
}

detgemm_status detgemm_gemm_s8_i32(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw, int32_t* C,
                                   int64_t ldc, int M, int N, int K, int split_k, void* ws, size_t ws_bytes,
                                   detgemm_stream_t stream) {
    detgemm_status st = validate_igemm(A, lda, W, ldw, C, ldc, 4, M, N, K, split_k, ws, ws_bytes);
    if (st != DETGEMM_OK) return st;
    if (M == 0 || N == 0) return DETGEMM_OK;
    if ((st = check_device()) != DETGEMM_OK) return st;
    return run_igemm(A, lda, W, ldw, nullptr, nullptr, nullptr, C, ldc, EPI_STORE_I32, M, N, K, split_k, ws,
                     reinterpret_cast<cudaStream_t>(stream));
}

// Fused linear layer scratch. Tensor-core path: A16 [M][Kp] fp16 | W16 [N][Kp] fp16 (only
// when no widened weight is given) | ea [M] | split-K sums and counters. Decode-shaped
// path: Q int8 [M][K16] | ea [M] | the decode-shaped GEMM's scratch.
struct LinearLayout {
    int64_t Kp, K16;
    size_t a, w16, ea, gemm, total;
};

static LinearLayout linear_layout(int M, int N, int K, int split_k, bool have_w16) {
    LinearLayout L;
    L.Kp = tc_padded_k(K);
    L.K16 = ((int64_t)K + 15) / 16 * 16;
    size_t off = 0;
    if (w8a8_uses_tc(M, K)) {
        L.a = off; off += align256((size_t)M * L.Kp * 2);
        L.w16 = off; off += have_w16 ? 0 : align256((size_t)N * L.Kp * 2);
        L.ea = off; off += align256((size_t)M * 4);
        L.gemm = off; off += align256(tc_split_bytes(1, M, N, split_k));
    } else {
        L.a = off; off += align256((size_t)M * L.K16);
        L.w16 = off;
        L.ea = off; off += align256((size_t)M * 4);
        L.gemm = off; off += align256(igemm_workspace_bytes(M, N, K, split_k));
    }
    L.total = off;
    return L;
}

size_t detgemm_linear_w8a8_workspace_size(int M, int N, int K, int split_k, int have_w16) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return linear_layout(M, N, K, split_k, have_w16 != 0).total;
}

static detgemm_status linear_impl(const void* X, int x_dtype, int64_t ldx, int mode, const int8_t* W, int64_t ldw,
                                  const uint16_t* W16, int64_t ldw16, const int32_t* ew, const uint16_t* bias,
                                  bool with_bias, uint16_t* C, int64_t ldc, int32_t* ea_out, int M, int N, int K,
                                  int split_k, void* ws, size_t ws_bytes, detgemm_stream_t stream) {
    if (M < 0 || N < 0 || K < 1) return DETGEMM_ERR_INVALID_ARG;
    if (x_dtype != DETGEMM_DTYPE_BF16 && x_dtype != DETGEMM_DTYPE_F32) return DETGEMM_ERR_INVALID_ARG;
    if (mode != DETGEMM_POW2_NEAREST && mode != DETGEMM_POW2_CEIL) return DETGEMM_ERR_INVALID_ARG;
    if (K > DETGEMM_MAX_K) return DETGEMM_ERR_PRECONDITION;
    if (split_k < 1 || split_k > (K + 63) / 64) return DETGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DETGEMM_OK;
    if (!X || !W || !ew || !C || ldx < K || ldw < K || ldc < N) return DETGEMM_ERR_INVALID_ARG;
    if (W16 && ldw16 < K) return DETGEMM_ERR_INVALID_ARG;
    if (with_bias && !bias) return DETGEMM_ERR_INVALID_ARG;
    if (with_bias && !aligned2(bias)) return DETGEMM_ERR_ALIGNMENT;
    const int epi = with_bias ? EPI_BF16_POW2_BIAS : EPI_BF16_POW2;
    if (!with_bias) bias = nullptr;
    const int xs = x_dtype == DETGEMM_DTYPE_BF16 ? 2 : 4;
    if (!aligned16(X) || !aligned16(W) || !aligned16(C) || !aligned4(ew) || (ea_out && !aligned4(ea_out)))
        return DETGEMM_ERR_ALIGNMENT;
    if ((ldx * xs) % 16 || ldw % 16 || (ldc * 2) % 16) return DETGEMM_ERR_ALIGNMENT;
    if (W16 && (!aligned16(W16) || ldw16 % 8)) return DETGEMM_ERR_ALIGNMENT;
    const bool tc = w8a8_uses_tc(M, K);
    const bool use_w16 = tc && W16 != nullptr;
    const LinearLayout L = linear_layout(M, N, K, split_k, use_w16);
    if (ws == nullptr || ws_bytes < L.total) return DETGEMM_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return DETGEMM_ERR_ALIGNMENT;
    detgemm_status st = check_device();
    if (st != DETGEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char* base = reinterpret_cast<char*>(ws);
    int32_t* ea = ea_out ? ea_out : reinterpret_cast<int32_t*>(base + L.ea);
    cudaError_t err;
    if (!tc) {
        // decode-shaped: int8 rows, then the W-streaming kernel on them
        int8_t* Q = reinterpret_cast<int8_t*>(base + L.a);
        err = quantize_pow2_launch(X, x_dtype, ldx, M, K, mode, Q, L.K16, ea, s);
        if (err != cudaSuccess) return DETGEMM_ERR_CUDA;
        return run_igemm(Q, L.K16, W, ldw, ea, ew, bias, C, ldc, epi, M, N, K, split_k, base + L.gemm, s);
    }
    // tensor-core path: the quantizer writes the activation operand directly in its fp16
    // carrier form (no int8 copy, no widening pass over it)
    err = quantize_pow2_f16_launch(X, x_dtype, ldx, M, K, mode, base + L.a, L.Kp, ea, s);
    if (err != cudaSuccess) return DETGEMM_ERR_CUDA;
    const void* wop = W16;
    int64_t ldwop = ldw16;
    if (!use_w16) {
        err = widen_i8_f16_launch(W, ldw, N, K, base + L.w16, L.Kp, s);
        if (err != cudaSuccess) return DETGEMM_ERR_CUDA;
        wop = base + L.w16;
        ldwop = L.Kp;
    }
    TcArgs a = {};
    a.M = M;
    a.N = N;
    a.ndiag = 1;
    a.diag_first[0] = 0;
    a.diag_nseg[0] = 1;
    a.split = split_k;
    a.mode = epi;
    a.ea = ea;
    a.ew = ew;
    a.bias = bias;
    a.C = C;
    a.ldc = ldc;
    return from_cuda(tc_gemm_launch(a, base + L.a, L.Kp, 1, wop, ldwop, 1, K, base + L.gemm, s));
}

detgemm_status detgemm_linear_w8a8(const void* X, int x_dtype, int64_t ldx, int mode, const int8_t* W, int64_t ldw,
                                   const uint16_t* W16, int64_t ldw16, const int32_t* ew, uint16_t* C, int64_t ldc,
                                   int32_t* ea_out, int M, int N, int K, int split_k, void* ws, size_t ws_bytes,
                                   detgemm_stream_t stream) {
    return linear_impl(X, x_dtype, ldx, mode, W, ldw, W16, ldw16, ew, nullptr, false, C, ldc, ea_out, M, N, K, split_k,
                       ws, ws_bytes, stream);
}

detgemm_status detgemm_linear_w8a8_bias(const void* X, int x_dtype, int64_t ldx, int mode, const int8_t* W,
                                        int64_t ldw, const uint16_t* W16, int64_t ldw16, const int32_t* ew,
                                        const uint16_t* bias, uint16_t* C, int64_t ldc, int32_t* ea_out, int M, int N,
                                        int K, int split_k, void* ws, size_t ws_bytes, detgemm_stream_t stream) {
    return linear_impl(X, x_dtype, ldx, mode, W, ldw, W16, ldw16, ew, bias, true, C, ldc, ea_out, M, N, K, split_k, ws,
                       ws_bytes, stream);
}

detgemm_status detgemm_quantize_pow2(const void* X, int x_dtype, int64_t ldx, int rows, int cols, int mode,
                                     int8_t* Q, int64_t ldq, int32_t* e, detgemm_stream_t stream) {
    if (rows < 0 || cols < 0) return DETGEMM_ERR_INVALID_ARG;
    if (x_dtype != DETGEMM_DTYPE_BF16 && x_dtype != DETGEMM_DTYPE_F32) return DETGEMM_ERR_INVALID_ARG;
    if (mode != DETGEMM_POW2_NEAREST && mode != DETGEMM_POW2_CEIL) return DETGEMM_ERR_INVALID_ARG;
    if (rows == 0) return DETGEMM_OK;
    if (!X || !Q || !e) return DETGEMM_ERR_INVALID_ARG;
    if (ldx < cols || ldq < cols) return DETGEMM_ERR_INVALID_ARG;
    const int xs = x_dtype == DETGEMM_DTYPE_BF16 ? 2 : 4;
    if (!aligned16(X) || !aligned16(Q) || !aligned4(e)) return DETGEMM_ERR_ALIGNMENT;
    if ((ldx * xs) % 16 != 0 || ldq % 16 != 0) return DETGEMM_ERR_ALIGNMENT;
    detgemm_status st = check_device();
    if (st != DETGEMM_OK) return st;
    return from_cuda(quantize_pow2_launch(X, x_dtype, ldx, rows, cols, mode, Q, ldq, e,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

detgemm_status detgemm_slice_f32(const float* X, int64_t ldx, int rows, int cols, int axis, int nslices, int8_t* S,
                                 int32_t* e, detgemm_stream_t stream) {
    if (rows < 0 || cols < 0) return DETGEMM_ERR_INVALID_ARG;
    if (axis != DETGEMM_AXIS_ROWS && axis != DETGEMM_AXIS_COLS) return DETGEMM_ERR_INVALID_ARG;
    if (nslices < 1 || nslices > 9) return DETGEMM_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) {
        if ((axis == DETGEMM_AXIS_ROWS ? rows : cols) == 0) return DETGEMM_OK;
    }
    if (!X || !S || !e) return DETGEMM_ERR_INVALID_ARG;
    if (ldx < cols) return DETGEMM_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(S) || !aligned4(e)) return DETGEMM_ERR_ALIGNMENT;
    if ((ldx * 4) % 16 != 0) return DETGEMM_ERR_ALIGNMENT;
    detgemm_status st = check_device();
    if (st != DETGEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (axis == DETGEMM_AXIS_ROWS) return from_cuda(slice_rows_launch(X, ldx, rows, cols, nslices, S, cols, e, s));
    return from_cuda(slice_cols_launch(X, ldx, rows, cols, nslices, S, rows, e, s));
}

detgemm_status detgemm_slice_f64(const double* X, int64_t ldx, int rows, int cols, int axis, int nslices, int8_t* S,
                                 int32_t* e, detgemm_stream_t stream) {
    if (rows < 0 || cols < 0) return DETGEMM_ERR_INVALID_ARG;
    if (nslices < 1 || nslices > 12) return DETGEMM_ERR_INVALID_ARG;
    if (axis != DETGEMM_AXIS_ROWS && axis != DETGEMM_AXIS_COLS) return DETGEMM_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return DETGEMM_OK;
    if (!X || !S || !e || ldx < cols) return DETGEMM_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(S) || !aligned4(e) || (ldx * 8) % 16) return DETGEMM_ERR_ALIGNMENT;
    detgemm_status st = check_device();
    if (st != DETGEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return from_cuda(slice_f64_launch(X, ldx, rows, cols, axis, nslices, S, axis == DETGEMM_AXIS_ROWS ? cols : rows,
                                      e, s));
}

size_t detgemm_ozaki_workspace_size(int M, int N, int K, int nslices, int max_diag, int split_k) {
    if (M <= 0 || N <= 0 || K <= 0 || nslices < 1 || max_diag < 2) return 0;
    return ozaki_layout(M, N, K, nslices, max_diag, split_k).total;
}

// Shared Ozaki driver: slice A per row and B per column into fp16 digit planes, all
// diagonals' exact slice products in one tensor-core launch (largest first; group d is
// diagonal g = max_diag - d and pairs A slice sA with B slice g - sA), then the combine.
static detgemm_status ozaki_run(const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                                bool f64, int M, int N, int K, int nslices, int max_diag, int split_k, void* ws,
                                size_t ws_bytes, detgemm_stream_t stream, bool exact_split = false,
                                int* parts_run = nullptr) {
    if (M < 0 || N < 0 || K < 1) return DETGEMM_ERR_INVALID_ARG;
    const int max_slices = f64 ? 12 : 9;
    if (nslices < 1 || nslices > max_slices || max_diag < 2 || max_diag > 2 * nslices || max_diag > kTcMaxDiag)
        return DETGEMM_ERR_INVALID_ARG;
    int nkb = (K + 63) / 64;
    if (split_k < 1 || split_k > nkb) return DETGEMM_ERR_INVALID_ARG;
    // every diagonal sum must stay in int32: at most min(g - 1, nslices) pairs of K products of |d| <= 127
    int pairs = max_diag - 1 < nslices ? max_diag - 1 : nslices;
    if ((long long)pairs * K * 127 * 127 >= 2147483648LL) return DETGEMM_ERR_PRECONDITION;
    int total_pairs = 0;
    for (int g = 2; g <= max_diag; ++g)
        for (int sA = 1; sA <= nslices; ++sA) total_pairs += (g - sA >= 1 && g - sA <= nslices) ? 1 : 0;
    if (total_pairs > kTcMaxSeg) return DETGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DETGEMM_OK;
    if (!A || !B || !C) return DETGEMM_ERR_INVALID_ARG;
    if (lda < K || ldb < N || ldc < N) return DETGEMM_ERR_INVALID_ARG;
    const int es = f64 ? 8 : 4;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return DETGEMM_ERR_ALIGNMENT;
    if ((lda * es) % 16 || (ldb * es) % 16 || (ldc * es) % 16) return DETGEMM_ERR_ALIGNMENT;
    OzakiLayout L = ozaki_layout(M, N, K, nslices, max_diag, split_k);
    if (ws == nullptr || ws_bytes < L.total) return DETGEMM_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return DETGEMM_ERR_ALIGNMENT;
    detgemm_status st = check_device();
    if (st != DETGEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char* base = reinterpret_cast<char*>(ws);
    int32_t* e = reinterpret_cast<int32_t*>(base + L.e);
    int32_t* f = reinterpret_cast<int32_t*>(base + L.f);
    int32_t* T = reinterpret_cast<int32_t*>(base + L.T);
    cudaError_t err;
    if (f64) {
        err = slice_f64_f16_launch(static_cast<const double*>(A), lda, M, K, 0, nslices, base + L.da, L.Kp, e, s);
        if (err == cudaSuccess)
            err = slice_f64_f16_launch(static_cast<const double*>(B), ldb, K, N, 1, nslices, base + L.db, L.Kp, f, s);
    } else {
        err = slice_rows_f16_launch(static_cast<const float*>(A), lda, M, K, nslices, base + L.da, L.Kp, e, s);
        if (err == cudaSuccess)
            err = slice_cols_f16_launch(static_cast<const float*>(B), ldb, K, N, nslices, base + L.db, L.Kp, f, s);
    }
    if (err != cudaSuccess) return DETGEMM_ERR_CUDA;
    TcArgs a = {};
    a.M = M;
    a.N = N;
    a.ndiag = max_diag - 1;
    int nseg = 0;
    for (int d = 0; d < a.ndiag; ++d) {
        const int g = max_diag - d;
        a.diag_first[d] = nseg;
        for (int sA = 1; sA <= nslices; ++sA) {
            const int tB = g - sA;
            if (tB < 1 || tB > nslices) continue;
            a.segA[nseg] = (int16_t)(sA - 1);
            a.segB[nseg] = (int16_t)(tB - 1);
            ++nseg;
        }
        a.diag_nseg[d] = nseg - a.diag_first[d];
    }
    a.split = split_k;  // <= ceil(K / 64) <= the K blocks of every diagonal
    a.mode = EPI_STORE_I32;
    a.C = T;
    a.ldc = L.ldT;
    a.c_plane = (int64_t)M * L.ldT;
    err = tc_gemm_launch(a, base + L.da, L.Kp, nslices, base + L.db, L.Kp, nslices, L.Kp, base + L.split, s,
                         exact_split, parts_run);
    if (err == cudaSuccess)
        err = f64 ? ozaki_combine_f64out_launch(T, L.ldT, max_diag, e, f, static_cast<double*>(C), ldc, M, N, s)
                  : ozaki_combine_launch(T, L.ldT, max_diag, e, f, static_cast<float*>(C), ldc, M, N, s);
    return from_cuda(err);
}

detgemm_status detgemm_ozaki_f32(const float* A, int64_t lda, const float* B, int64_t ldb, float* C, int64_t ldc,
                                 int M, int N, int K, int nslices, int max_diag, int split_k, void* ws,
                                 size_t ws_bytes, detgemm_stream_t stream) {
    return ozaki_run(A, lda, B, ldb, C, ldc, false, M, N, K, nslices, max_diag, split_k, ws, ws_bytes, stream);
}

detgemm_status detgemm_ozaki_f32_split_exact(const float* A, int64_t lda, const float* B, int64_t ldb, float* C,
                                             int64_t ldc, int M, int N, int K, int nslices, int max_diag, int split_k,
                                             void* ws, size_t ws_bytes, int* parts_run, detgemm_stream_t stream) {
    if (parts_run) *parts_run = 0;
    return ozaki_run(A, lda, B, ldb, C, ldc, false, M, N, K, nslices, max_diag, split_k, ws, ws_bytes, stream, true,
                     parts_run);
}

detgemm_status detgemm_ozaki_f64(const double* A, int64_t lda, const double* B, int64_t ldb, double* C, int64_t ldc,
                                 int M, int N, int K, int nslices, int max_diag, int split_k, void* ws,
                                 size_t ws_bytes, detgemm_stream_t stream) {
    return ozaki_run(A, lda, B, ldb, C, ldc, true, M, N, K, nslices, max_diag, split_k, ws, ws_bytes, stream);
}

size_t detgemm_ozaki_f64_workspace_size(int M, int N, int K, int nslices, int max_diag, int split_k) {
    return detgemm_ozaki_workspace_size(M, N, K, nslices, max_diag, split_k);
}

detgemm_status detgemm_ozaki_combine(const int32_t* T, int64_t ldT, int max_diag, const int32_t* e,
                                     const int32_t* f, void* C, int c_dtype, int64_t ldc, int M, int N,
                                     detgemm_stream_t stream) {
    if (M < 0 || N < 0 || max_diag < 2 || max_diag > 18) return DETGEMM_ERR_INVALID_ARG;
    if (c_dtype != DETGEMM_DTYPE_F32 && c_dtype != DETGEMM_DTYPE_F64) return DETGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DETGEMM_OK;
    if (!T || !e || !f || !C || ldT < N || ldc < N) return DETGEMM_ERR_INVALID_ARG;
    const int cs = c_dtype == DETGEMM_DTYPE_F64 ? 8 : 4;
    if (!aligned16(T) || !aligned16(C) || !aligned4(e) || !aligned4(f)) return DETGEMM_ERR_ALIGNMENT;
    if ((ldT * 4) % 16 || (ldc * cs) % 16) return DETGEMM_ERR_ALIGNMENT;
    detgemm_status st = check_device();
    if (st != DETGEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (c_dtype == DETGEMM_DTYPE_F64)
        return from_cuda(ozaki_combine_f64out_launch(T, ldT, max_diag, e, f, static_cast<double*>(C), ldc, M, N, s));
    return from_cuda(ozaki_combine_launch(T, ldT, max_diag, e, f, static_cast<float*>(C), ldc, M, N, s));
}

detgemm_status detgemm_widen_i8_f16(const int8_t* X, int64_t ldx, int rows, int cols, uint16_t* Y, int64_t ldy,
                                    detgemm_stream_t stream) {
    if (rows < 0 || cols < 0) return DETGEMM_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return DETGEMM_OK;
    if (!X || !Y || ldx < cols || ldy < cols) return DETGEMM_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Y) || ldx % 16 != 0 || ldy % 8 != 0) return DETGEMM_ERR_ALIGNMENT;
    detgemm_status st = check_device();
    if (st != DETGEMM_OK) return st;
    // the widening kernel writes 8-element groups up to ldy rounded down to 8 (all of ldy),
    // zero beyond cols
    return from_cuda(widen_i8_f16_launch(X, ldx, rows, cols, Y, ldy, reinterpret_cast<cudaStream_t>(stream)));
}

size_t detgemm_w8a8_f16ops_workspace_size(int M, int N, int K, int split_k) {
    (void)K;
    if (M <= 0 || N <= 0) return 0;
    return tc_split_bytes(1, M, N, split_k);
}

detgemm_status detgemm_w8a8_f16ops(const uint16_t* A16, int64_t lda, const uint16_t* W16, int64_t ldw,
                                   const int32_t* ea, const int32_t* ew, uint16_t* C, int64_t ldc, int M, int N,
                                   int K, int split_k, void* ws, size_t ws_bytes, detgemm_stream_t stream) {
    if (M < 0 || N < 0 || K < 1) return DETGEMM_ERR_INVALID_ARG;
    if (K > DETGEMM_MAX_K) return DETGEMM_ERR_PRECONDITION;
    if (split_k < 1 || split_k > (K + 63) / 64) return DETGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DETGEMM_OK;
    if (!A16 || !W16 || !C || !ea || !ew) return DETGEMM_ERR_INVALID_ARG;
    if (lda < K || ldw < K || ldc < N) return DETGEMM_ERR_INVALID_ARG;
    if (!aligned16(A16) || !aligned16(W16) || !aligned16(C) || !aligned4(ea) || !aligned4(ew))
        return DETGEMM_ERR_ALIGNMENT;
    if (lda % 8 != 0 || ldw % 8 != 0 || ldc % 8 != 0) return DETGEMM_ERR_ALIGNMENT;
    const size_t need = detgemm_w8a8_f16ops_workspace_size(M, N, K, split_k);
    if (need > 0 && (ws == nullptr || ws_bytes < need)) return DETGEMM_ERR_WORKSPACE;
    if (need > 0 && (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return DETGEMM_ERR_ALIGNMENT;
    detgemm_status st = check_device();
    if (st != DETGEMM_OK) return st;
    TcArgs a = {};
    a.M = M;
    a.N = N;
    a.ndiag = 1;
    a.diag_first[0] = 0;
    a.diag_nseg[0] = 1;
    a.split = split_k;
    a.mode = EPI_BF16_POW2;
    a.ea = ea;
    a.ew = ew;
    a.C = C;
    a.ldc = ldc;
    return from_cuda(tc_gemm_launch(a, A16, lda, 1, W16, ldw, 1, K, ws, reinterpret_cast<cudaStream_t>(stream)));
}

detgemm_status detgemm_gemm_fixed_f16(const uint16_t* A, int64_t lda, const uint16_t* W, int64_t ldw, float* C,
                                      int64_t ldc, int M, int N, int K, int dtype, detgemm_stream_t stream) {
    if (M < 0 || N < 0 || K < 1) return DETGEMM_ERR_INVALID_ARG;
    if (dtype != DETGEMM_DTYPE_F16 && dtype != DETGEMM_DTYPE_BF16) return DETGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DETGEMM_OK;
    if (!A || !W || !C || lda < K || ldw < K || ldc < N) return DETGEMM_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(W) || !aligned16(C)) return DETGEMM_ERR_ALIGNMENT;
    if (lda % 8 || ldw % 8 || ldc % 4) return DETGEMM_ERR_ALIGNMENT;
    detgemm_status st = check_device();
    if (st != DETGEMM_OK) return st;
    TcArgs a = {};
    a.M = M;
    a.N = N;
    a.ndiag = 1;
    a.diag_first[0] = 0;
    a.diag_nseg[0] = 1;
    a.split = 1;
    a.mode = EPI_STORE_I32;
    a.C = C;
    a.ldc = ldc;
    a.fp_mode = dtype == DETGEMM_DTYPE_BF16 ? 2 : 1;
    return from_cuda(tc_gemm_launch(a, A, lda, 1, W, ldw, 1, K, nullptr, reinterpret_cast<cudaStream_t>(stream)));
}

// Gated W8A8 scratch: A16 [M][Kp] fp16 | W16 [2][N][Kp] fp16 (gate plane, up plane)
static size_t swiglu_ws(int M, int N, int K, int64_t* Kp, size_t* w16_off) {
    *Kp = tc_padded_k(K);
    *w16_off = align256((size_t)M * *Kp * 2);
    return *w16_off + align256((size_t)2 * N * *Kp * 2);
}

size_t detgemm_w8a8_swiglu_workspace_size(int M, int N, int K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    int64_t Kp;
    size_t off;
    return swiglu_ws(M, N, K, &Kp, &off);
}

detgemm_status detgemm_w8a8_swiglu(const int8_t* A, int64_t lda, const int8_t* Wg, const int8_t* Wu, int64_t ldw,
                                   const int32_t* ea, const int32_t* ewg, const int32_t* ewu, uint16_t* C, int64_t ldc,
                                   int M, int N, int K, void* ws, size_t ws_bytes, detgemm_stream_t stream) {
    if (M < 0 || N < 0 || K < 1) return DETGEMM_ERR_INVALID_ARG;
    if (K > DETGEMM_MAX_K) return DETGEMM_ERR_PRECONDITION;
    if (M == 0 || N == 0) return DETGEMM_OK;
    if (!A || !Wg || !Wu || !ea || !ewg || !ewu || !C || lda < K || ldw < K || ldc < N) return DETGEMM_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(C) || !aligned4(ea) || !aligned4(ewg) ||
        !aligned4(ewu))
        return DETGEMM_ERR_ALIGNMENT;
    if (lda % 16 || ldw % 16 || (ldc * 2) % 16) return DETGEMM_ERR_ALIGNMENT;
    int64_t Kp;
    size_t w16;
    const size_t need = swiglu_ws(M, N, K, &Kp, &w16);
    if (!ws || ws_bytes < need) return DETGEMM_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return DETGEMM_ERR_ALIGNMENT;
    detgemm_status st = check_device();
    if (st != DETGEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char* base = reinterpret_cast<char*>(ws);
    char* Wp = base + w16;
    cudaError_t e = widen_pair_launch(A, lda, M, K, base, Kp, Wg, ldw, N, K, Wp, Kp, s);
    if (e == cudaSuccess) e = widen_i8_f16_launch(Wu, ldw, N, K, Wp + (size_t)N * Kp * 2, Kp, s);
    if (e != cudaSuccess) return DETGEMM_ERR_CUDA;
    TcArgs a = {};
    a.M = M;
    a.N = N;
    a.ndiag = 1;
    a.diag_first[0] = 0;
    a.diag_nseg[0] = 1;
    a.split = 1;
    a.mode = EPI_BF16_POW2;
    a.ea = ea;
    a.ew = ewg;
    a.ewu = ewu;
    a.C = C;
    a.ldc = ldc;
    a.swiglu = 1;
    return from_cuda(tc_gemm_launch(a, base, Kp, 1, Wp, Kp, 2, Kp, nullptr, s));
}

detgemm_status detgemm_swiglu_bf16(const int32_t* G, int64_t ldg, const int32_t* U, int64_t ldu, const int32_t* ea,
                                   const int32_t* ewg, const int32_t* ewu, uint16_t* C, int64_t ldc, int M, int N,
                                   detgemm_stream_t stream) {
    if (M < 0 || N < 0) return DETGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DETGEMM_OK;
    if (!G || !U || !ea || !ewg || !ewu || !C || ldg < N || ldu < N || ldc < N) return DETGEMM_ERR_INVALID_ARG;
    if (!aligned4(G) || !aligned4(U) || !aligned4(ea) || !aligned4(ewg) || !aligned4(ewu) || !aligned2(C))
        return DETGEMM_ERR_ALIGNMENT;
    detgemm_status st = check_device();
    if (st != DETGEMM_OK) return st;
    return from_cuda(swiglu_epilogue_launch(G, ldg, U, ldu, ea, ewg, ewu, C, ldc, M, N,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

detgemm_status detgemm_selftest_timeout(int limit_ms, detgemm_stream_t stream) {
    if (limit_ms < 1 || limit_ms > 2000) return DETGEMM_ERR_INVALID_ARG;
    detgemm_status st = check_device();
    if (st != DETGEMM_OK) return st;
    return from_cuda(selftest_wait_launch((uint64_t)limit_ms * 1000000ull, reinterpret_cast<cudaStream_t>(stream)));
}

detgemm_status detgemm_get_device_status(detgemm_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return DETGEMM_ERR_CUDA;
    uint32_t v = 0, bits = 0;
    if (quantize_take_status(&bits) != cudaSuccess) return DETGEMM_ERR_CUDA;
    v |= bits;
    if (slice_take_status(&bits) != cudaSuccess) return DETGEMM_ERR_CUDA;
    v |= bits;
    if (tc_take_status(&bits) != cudaSuccess) return DETGEMM_ERR_CUDA;
    v |= bits;
    if (skinny_take_status(&bits) != cudaSuccess) return DETGEMM_ERR_CUDA;
    v |= bits;
    if (swiglu_take_status(&bits) != cudaSuccess) return DETGEMM_ERR_CUDA;
    v |= bits;
    if (v & DEV_TIMEOUT) return DETGEMM_ERR_TIMEOUT;
    if (v & DEV_NONFINITE) return DETGEMM_ERR_NONFINITE;
    if (v & DEV_RANGE) return DETGEMM_ERR_RANGE;
    return DETGEMM_OK;
}

}  // extern "C"
