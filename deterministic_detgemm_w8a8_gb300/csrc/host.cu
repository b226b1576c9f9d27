// detgemm_w8a8_host: the W8A8 GEMM on operands that live in host memory, with the
// host-to-device copies, the computation and the device-to-host copy of the result
// overlapped.
//
// The rows of A are cut into chunks; chunk c's rows are copied in on one stream while
// chunk c - 1 is computed on the caller's stream and chunk c - 2's result is copied out on
// a third stream. The first chunk is half the size of the others, so that the copy-out
// stream starts sooner, and the last one takes what is left. Every chunk runs the same exact W8A8 path as detgemm_w8a8 on its rows
// ("Deterministic LLM Inference Across GPU Kernels ...", §II: the int32 accumulator and
// so the bf16 result of a row do not depend on which rows are computed with it), so the
// result bits are those of detgemm_w8a8 on the whole matrix.
//
// Device memory is the caller's buffer (no allocation here): the weight (int8 and its
// exact fp16 copy), the weight exponents, and two chunk slots (int8 rows, their fp16
// copy, their exponents and their bf16 results). The two copy streams and the events
// that order the pipeline are created once per device and reused; a mutex serialises the
// enqueueing of concurrent calls.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/detgemm.h"
#include "internal.h"

namespace detgemm {
namespace {

constexpr int kMaxDev = 64;
constexpr int kSlots = 2;

struct Pipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, wready = nullptr;
    cudaEvent_t inev[kSlots] = {}, comp[kSlots] = {}, outd[kSlots] = {};
};

std::mutex g_host_mutex;
Pipe g_pipe[kMaxDev];

cudaError_t pipe_for_device(Pipe** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    Pipe& p = g_pipe[dev];
    if (p.in == nullptr) {
        const unsigned ef = cudaEventDisableTiming;
        if ((e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&p.start, ef)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&p.wready, ef)) != cudaSuccess) return e;
        for (int i = 0; i < kSlots; ++i) {
            if ((e = cudaEventCreateWithFlags(&p.inev[i], ef)) != cudaSuccess) return e;
            if ((e = cudaEventCreateWithFlags(&p.comp[i], ef)) != cudaSuccess) return e;
            if ((e = cudaEventCreateWithFlags(&p.outd[i], ef)) != cudaSuccess) return e;
        }
    }
    *out = &p;
    return cudaSuccess;
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

// Buffer layout. Rows are stored with 16-byte aligned strides: int8 rows of K16 bytes,
// fp16 rows of Kp elements (the tensor-core engine's padded K), bf16 results of N8.
struct HostLayout {
    bool tc;        // tensor-core path, or the decode-shaped path (decode_path(M, K))
    int R;          // rows per chunk
    int64_t K16, Kp, N8;
    size_t w, ew, w16, ws;
    size_t a[kSlots], ea[kSlots], a16[kSlots], c[kSlots];
    size_t total;
};

HostLayout host_layout(int M, int N, int K) {
    HostLayout L = {};
    L.tc = !decode_path(M, K);
    L.K16 = ((int64_t)K + 15) / 16 * 16;
    L.Kp = tc_padded_k(K);
    L.N8 = ((int64_t)N + 7) / 8 * 8;
    // chunks of about a quarter of M (the first one half that; see below), each a multiple
    // of the engine's 256-row tile
    L.R = L.tc ? (int)((((int64_t)M + 3) / 4 + 255) / 256 * 256) : M;
    size_t off = 0;
    L.w = off; off += up256((size_t)N * L.K16);
    L.ew = off; off += up256((size_t)N * 4);
    L.w16 = off; off += L.tc ? up256((size_t)N * L.Kp * 2) : 0;
    const int slots = L.tc ? kSlots : 1;
    for (int s = 0; s < slots; ++s) {
        L.a[s] = off; off += up256((size_t)L.R * L.K16);
        L.ea[s] = off; off += up256((size_t)L.R * 4);
        L.a16[s] = off; off += L.tc ? up256((size_t)L.R * L.Kp * 2) : 0;
        L.c[s] = off; off += up256((size_t)L.R * L.N8 * 2);
    }
    L.ws = off;
    off += up256(L.tc ? detgemm_w8a8_f16ops_workspace_size(L.R, N, K, 1) : detgemm_w8a8_workspace_size(M, N, K, 1));
    L.total = off;
    return L;
}

}  // namespace
}  // namespace detgemm

using namespace detgemm;

extern "C" {

size_t detgemm_w8a8_host_buffer_size(int M, int N, int K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return host_layout(M, N, K).total;
}

detgemm_status detgemm_w8a8_host(const int8_t* A, int64_t lda, const int8_t* W, int64_t ldw, const int32_t* ea,
                                 const int32_t* ew, uint16_t* C, int64_t ldc, int M, int N, int K, void* buf,
                                 size_t buf_bytes, detgemm_stream_t stream) {
    if (M < 0 || N < 0 || K < 1) return DETGEMM_ERR_INVALID_ARG;
    if (K > DETGEMM_MAX_K) return DETGEMM_ERR_PRECONDITION;
    if (M == 0 || N == 0) return DETGEMM_OK;
    if (!A || !W || !ea || !ew || !C || lda < K || ldw < K || ldc < N) return DETGEMM_ERR_INVALID_ARG;
    const HostLayout L = host_layout(M, N, K);
    if (buf == nullptr || buf_bytes < L.total) return DETGEMM_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(buf) & 255u) != 0) return DETGEMM_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char* b = reinterpret_cast<char*>(buf);
    int8_t* Wd = reinterpret_cast<int8_t*>(b + L.w);
    int32_t* ewd = reinterpret_cast<int32_t*>(b + L.ew);

    if (!device_is_supported()) return DETGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_host_mutex);
    Pipe* p = nullptr;
    if (pipe_for_device(&p) != cudaSuccess) return DETGEMM_ERR_CUDA;
#define CHK(x)                                            \
    do {                                                  \
        if ((x) != cudaSuccess) return DETGEMM_ERR_CUDA;  \
    } while (0)
    // the buffer is free once the caller's stream has finished what it holds
    CHK(cudaEventRecord(p->start, s));
    CHK(cudaStreamWaitEvent(p->in, p->start, 0));
    CHK(cudaStreamWaitEvent(p->out, p->start, 0));
    CHK(cudaMemcpy2DAsync(Wd, L.K16, W, ldw, K, N, cudaMemcpyHostToDevice, p->in));
    CHK(cudaMemcpyAsync(ewd, ew, (size_t)N * 4, cudaMemcpyHostToDevice, p->in));
    CHK(cudaEventRecord(p->wready, p->in));
    CHK(cudaStreamWaitEvent(s, p->wready, 0));

    if (!L.tc) {
        // decode-shaped: one chunk through detgemm_w8a8 (its W-streaming kernels)
        int8_t* Ad = reinterpret_cast<int8_t*>(b + L.a[0]);
        int32_t* ead = reinterpret_cast<int32_t*>(b + L.ea[0]);
        uint16_t* Cd = reinterpret_cast<uint16_t*>(b + L.c[0]);
        CHK(cudaMemcpy2DAsync(Ad, L.K16, A, lda, K, M, cudaMemcpyHostToDevice, p->in));
        CHK(cudaMemcpyAsync(ead, ea, (size_t)M * 4, cudaMemcpyHostToDevice, p->in));
        CHK(cudaEventRecord(p->inev[0], p->in));
        CHK(cudaStreamWaitEvent(s, p->inev[0], 0));
        const size_t wsb = detgemm_w8a8_workspace_size(M, N, K, 1);
        detgemm_status st = detgemm_w8a8(Ad, L.K16, Wd, L.K16, ead, ewd, Cd, L.N8, M, N, K, 1, b + L.ws, wsb, stream);
        if (st != DETGEMM_OK) return st;
        CHK(cudaEventRecord(p->comp[0], s));
        CHK(cudaStreamWaitEvent(p->out, p->comp[0], 0));
        CHK(cudaMemcpy2DAsync(C, (size_t)ldc * 2, Cd, (size_t)L.N8 * 2, (size_t)N * 2, M, cudaMemcpyDeviceToHost,
                              p->out));
        CHK(cudaEventRecord(p->outd[0], p->out));
        CHK(cudaStreamWaitEvent(s, p->outd[0], 0));
        return DETGEMM_OK;
    }

    // tensor-core path: the weight is widened once, then the chunks are pipelined
    uint16_t* W16 = reinterpret_cast<uint16_t*>(b + L.w16);
    CHK(widen_i8_f16_launch(Wd, L.K16, N, K, W16, L.Kp, s));
    const size_t wsb = detgemm_w8a8_f16ops_workspace_size(L.R, N, K, 1);
    const int first = L.R / 2 / 256 * 256 > 256 ? L.R / 2 / 256 * 256 : 256;
    int nchunks = 0;
    for (int c = 0, r0 = 0; r0 < M; ++c) {
        const int want = c == 0 && L.R < M ? first : L.R;
        const int rows = M - r0 < want ? M - r0 : want;
        nchunks = c + 1;
        const int sl = c % kSlots;
        int8_t* Ad = reinterpret_cast<int8_t*>(b + L.a[sl]);
        int32_t* ead = reinterpret_cast<int32_t*>(b + L.ea[sl]);
        uint16_t* A16 = reinterpret_cast<uint16_t*>(b + L.a16[sl]);
        uint16_t* Cd = reinterpret_cast<uint16_t*>(b + L.c[sl]);
        // copy in once the computation two chunks back no longer reads this slot
        if (c >= kSlots) CHK(cudaStreamWaitEvent(p->in, p->comp[sl], 0));
        CHK(cudaMemcpy2DAsync(Ad, L.K16, A + (int64_t)r0 * lda, lda, K, rows, cudaMemcpyHostToDevice, p->in));
        CHK(cudaMemcpyAsync(ead, ea + r0, (size_t)rows * 4, cudaMemcpyHostToDevice, p->in));
        CHK(cudaEventRecord(p->inev[sl], p->in));
        // compute once the rows are in and the copy-out two chunks back has read this slot
        CHK(cudaStreamWaitEvent(s, p->inev[sl], 0));
        if (c >= kSlots) CHK(cudaStreamWaitEvent(s, p->outd[sl], 0));
        CHK(widen_i8_f16_launch(Ad, L.K16, rows, K, A16, L.Kp, s));
        detgemm_status st = detgemm_w8a8_f16ops(A16, L.Kp, W16, L.Kp, ead, ewd, Cd, L.N8, rows, N, K, 1,
                                                b + L.ws, wsb, stream);
        if (st != DETGEMM_OK) return st;
        CHK(cudaEventRecord(p->comp[sl], s));
        // copy the chunk's result out
        CHK(cudaStreamWaitEvent(p->out, p->comp[sl], 0));
        CHK(cudaMemcpy2DAsync(C + (int64_t)r0 * ldc, (size_t)ldc * 2, Cd, (size_t)L.N8 * 2, (size_t)N * 2, rows,
                              cudaMemcpyDeviceToHost, p->out));
        CHK(cudaEventRecord(p->outd[sl], p->out));
        r0 += rows;
    }
    // the caller's stream completes only when every result has reached host memory
    for (int sl = 0; sl < kSlots && sl < nchunks; ++sl) CHK(cudaStreamWaitEvent(s, p->outd[sl], 0));
#undef CHK
    return DETGEMM_OK;
}

}  // extern "C"
