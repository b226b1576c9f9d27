"""Batch-invariant exact GEMM for NVIDIA GB300 — Python binding of libdetgemm.

A thin ctypes layer over the C ABI declared in ``include/detgemm.h``: it checks
tensor dtypes/devices, allocates outputs and scratch with PyTorch, and passes raw
device pointers and the current CUDA stream. Every step of the computation runs in
the library's CUDA kernels; there is no CPU path. If ``libdetgemm.so`` has not been
built, importing works but every call raises ``DetGemmError``.

Functions mirror the C entry points:

* :func:`w8a8`           C = rne_bf16((A W^T) * 2^(ea_i + ew_j))      (bf16 out)
* :func:`w8a8_host`      the same on host (pinned) tensors, copies overlapped with compute
* :func:`w8a8_split_exact`  w8a8 with exactly the K cut asked for (invariance checks)
* :func:`gemm_s8_i32`    C = A W^T, exact int32
* :func:`quantize_pow2`  per-row power-of-two scale and int8 values
* :func:`linear_w8a8`    quantize_pow2 of bf16/fp32 activations + w8a8, fused
* :func:`slice_f32`      Ozaki digit planes with shared exponents
* :func:`ozaki_f32`      Ozaki-scheme fp32 GEMM C = A B
* :func:`ozaki_combine`  its fixed-order fp64 recombination step alone
* :func:`ozaki_f64`      the fp64-target Ozaki GEMM (DGEMM emulation), :func:`slice_f64`
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdetgemm.so")

OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_PRECONDITION, ERR_WORKSPACE = 0, 1, 2, 3, 4
ERR_UNSUPPORTED_DEVICE, ERR_CUDA, ERR_TIMEOUT, ERR_NONFINITE, ERR_RANGE = 5, 6, 7, 8, 9
DTYPE_BF16, DTYPE_F32, DTYPE_F64, DTYPE_F16 = 0, 1, 2, 3
POW2_NEAREST, POW2_CEIL = 0, 1
AXIS_ROWS, AXIS_COLS = 0, 1
MAX_K = 131071
NOALLOC_SCRATCH_BYTES = 8 << 20  # scratch array size of detgemm_w8a8_noalloc

# every symbol include/detgemm.h declares, with its ctypes signature
_P, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "detgemm_status_string": ([_I32], ctypes.c_char_p),
    "detgemm_version": ([], _I32),
    "detgemm_w8a8": ([_P, _I64, _P, _I64, _P, _P, _P, _I64, _I32, _I32, _I32, _I32, _P, _SZ, _P], _I32),
    "detgemm_w8a8_workspace_size": ([_I32, _I32, _I32, _I32], _SZ),
    "detgemm_w8a8_bias": ([_P, _I64, _P, _I64, _P, _P, _P, _P, _I64, _I32, _I32, _I32, _I32, _P, _SZ, _P], _I32),
    "detgemm_gemm_s8_i32": ([_P, _I64, _P, _I64, _P, _I64, _I32, _I32, _I32, _I32, _P, _SZ, _P], _I32),
    "detgemm_quantize_pow2": ([_P, _I32, _I64, _I32, _I32, _I32, _P, _I64, _P, _P], _I32),
    "detgemm_slice_f32": ([_P, _I64, _I32, _I32, _I32, _I32, _P, _P, _P], _I32),
    "detgemm_ozaki_f32": ([_P, _I64, _P, _I64, _P, _I64, _I32, _I32, _I32, _I32, _I32, _I32, _P, _SZ, _P], _I32),
    "detgemm_ozaki_workspace_size": ([_I32, _I32, _I32, _I32, _I32, _I32], _SZ),
    "detgemm_ozaki_combine": ([_P, _I64, _I32, _P, _P, _P, _I32, _I64, _I32, _I32, _P], _I32),
    "detgemm_slice_f64": ([_P, _I64, _I32, _I32, _I32, _I32, _P, _P, _P], _I32),
    "detgemm_ozaki_f64": ([_P, _I64, _P, _I64, _P, _I64, _I32, _I32, _I32, _I32, _I32, _I32, _P, _SZ, _P], _I32),
    "detgemm_ozaki_f64_workspace_size": ([_I32, _I32, _I32, _I32, _I32, _I32], _SZ),
    "detgemm_w8a8_host": ([_P, _I64, _P, _I64, _P, _P, _P, _I64, _I32, _I32, _I32, _P, _SZ, _P], _I32),
    "detgemm_w8a8_host_buffer_size": ([_I32, _I32, _I32], _SZ),
    "detgemm_linear_w8a8": ([_P, _I32, _I64, _I32, _P, _I64, _P, _I64, _P, _P, _I64, _P, _I32, _I32, _I32, _I32,
                             _P, _SZ, _P], _I32),
    "detgemm_linear_w8a8_workspace_size": ([_I32, _I32, _I32, _I32, _I32], _SZ),
    "detgemm_linear_w8a8_bias": ([_P, _I32, _I64, _I32, _P, _I64, _P, _I64, _P, _P, _P, _I64, _P, _I32, _I32, _I32,
                                  _I32, _P, _SZ, _P], _I32),
    "detgemm_get_device_status": ([_P], _I32),
    "detgemm_w8a8_noalloc": ([_P, _I64, _P, _I64, _P, _P, _P, _I64, _I32, _I32, _I32, _I32, _P], _I32),
    "detgemm_w8a8_noalloc_scratch_size": ([_I32, _I32, _I32, _I32], _SZ),
    "detgemm_widen_i8_f16": ([_P, _I64, _I32, _I32, _P, _I64, _P], _I32),
    "detgemm_w8a8_f16ops": ([_P, _I64, _P, _I64, _P, _P, _P, _I64, _I32, _I32, _I32, _I32, _P, _SZ, _P], _I32),
    "detgemm_w8a8_f16ops_workspace_size": ([_I32, _I32, _I32, _I32], _SZ),
    "detgemm_selftest_timeout": ([_I32, _P], _I32),
    "detgemm_w8a8_split_exact": ([_P, _I64, _P, _I64, _P, _P, _P, _I64, _I32, _I32, _I32, _I32, _P, _SZ, _P, _P],
                                 _I32),
    "detgemm_w8a8_swiglu": ([_P, _I64, _P, _P, _I64, _P, _P, _P, _P, _I64, _I32, _I32, _I32, _P, _SZ, _P], _I32),
    "detgemm_w8a8_swiglu_workspace_size": ([_I32, _I32, _I32], _SZ),
    "detgemm_swiglu_bf16": ([_P, _I64, _P, _I64, _P, _P, _P, _P, _I64, _I32, _I32, _P], _I32),
    "detgemm_gemm_fixed_f16": ([_P, _I64, _P, _I64, _P, _I64, _I32, _I32, _I32, _I32, _P], _I32),
    "detgemm_epilogue_inject": ([_P, _I64, _I32, _P, _P, _I32, _I32, ctypes.c_uint32, _P, _I64, _I32, _I32, _P], _I32),
    "detgemm_ozaki_f32_split_exact": ([_P, _I64, _P, _I64, _P, _I64, _I32, _I32, _I32, _I32, _I32, _I32, _P, _SZ,
                                       _P, _P], _I32),
}

_lock = threading.Lock()
_lib = None


class DetGemmError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        name = status_string(status) if _lib is not None else str(status)
        super().__init__(f"{where}: {name}" if where else name)


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libdetgemm.so (raises DetGemmError-compatible RuntimeError if absent)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libdetgemm.so not found at {path}; build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(path)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().detgemm_status_string(status).decode()


def _check(status: int, where: str):
    if status != OK:
        raise DetGemmError(status, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _req(t: torch.Tensor, dtype, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() == 2 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit stride along its last dimension")
    if t.dim() == 1 and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _ld(t: torch.Tensor) -> int:
    """Row stride in elements; a single row may use any stride, so report an aligned one."""
    if t.shape[0] > 1:
        return t.stride(0)
    per = 16 // t.element_size()
    return max(per, (t.shape[1] + per - 1) // per * per)


def empty2d(rows: int, cols: int, dtype, device) -> torch.Tensor:
    """[rows, cols] tensor whose row stride is a multiple of 16 bytes (the library's rule)."""
    esize = torch.empty((), dtype=dtype).element_size()
    per = 16 // esize
    ld = max(per, (cols + per - 1) // per * per)
    return torch.empty((rows, ld), dtype=dtype, device=device)[:, :cols]


def _workspace(nbytes: int, device, ws):
    if nbytes == 0:
        return None, 0
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise ValueError(f"workspace too small: need {nbytes} bytes")
        return ws, ws.numel() * ws.element_size()
    return torch.empty(nbytes, dtype=torch.uint8, device=device), nbytes


def w8a8_workspace_size(M: int, N: int, K: int, split_k: int = 1) -> int:
    return int(load().detgemm_w8a8_workspace_size(M, N, K, split_k))


def ozaki_workspace_size(M, N, K, nslices=7, max_diag=8, split_k=1) -> int:
    return int(load().detgemm_ozaki_workspace_size(M, N, K, nslices, max_diag, split_k))


def _bias_vec(bias, N, device):
    if bias is None:
        return None
    if not isinstance(bias, torch.Tensor) or bias.dtype != torch.bfloat16 or bias.shape != (N,):
        raise ValueError("bias must be a bfloat16 tensor of shape [N]")
    if bias.device != device or not bias.is_contiguous():
        raise ValueError("bias must be contiguous on the operands' device")
    return bias


def w8a8(A, W, ea, ew, split_k: int = 1, out=None, ws=None, stream=None, bias=None) -> torch.Tensor:
    """C = rne_bf16((A W^T) * 2^(ea_i + ew_j) [+ bias_j]); A int8 [M,K], W int8 [N,K], ea/ew
    int32, bias (optional) bfloat16 [N] added before the one rounding.
    Returns a torch.bfloat16 tensor [M, N] (or writes ``out``)."""
    lib = load()
    _req(A, torch.int8, "A"); _req(W, torch.int8, "W")
    _req(ea, torch.int32, "ea"); _req(ew, torch.int32, "ew")
    M, K = A.shape
    N = W.shape[0]
    if W.shape[1] != K or ea.shape != (M,) or ew.shape != (N,):
        raise ValueError("shape mismatch")
    if out is None:
        out = empty2d(M, N, torch.bfloat16, A.device)
    _req(out, torch.bfloat16, "out")
    bias = _bias_vec(bias, N, A.device)
    wsb, wsn = _workspace(w8a8_workspace_size(M, N, K, split_k), A.device, ws)
    if bias is not None:
        st = lib.detgemm_w8a8_bias(A.data_ptr(), _ld(A), W.data_ptr(), _ld(W), ea.data_ptr(), ew.data_ptr(),
                                   bias.data_ptr(), out.data_ptr(), _ld(out), M, N, K, split_k,
                                   wsb.data_ptr() if wsb is not None else None, wsn, _stream(stream))
        _check(st, "detgemm_w8a8_bias")
        return out
    st = lib.detgemm_w8a8(A.data_ptr(), _ld(A), W.data_ptr(), _ld(W), ea.data_ptr(), ew.data_ptr(),
                          out.data_ptr(), _ld(out), M, N, K, split_k,
                          wsb.data_ptr() if wsb is not None else None, wsn, _stream(stream))
    _check(st, "detgemm_w8a8")
    return out


def w8a8_split_exact(A, W, ea, ew, split_k: int, out=None, ws=None, stream=None):
    """w8a8 with the K cut made exactly as asked (detgemm_w8a8_split_exact): returns
    (C, parts_run), parts_run being the number of contiguous K parts the call ran."""
    lib = load()
    _req(A, torch.int8, "A"); _req(W, torch.int8, "W")
    _req(ea, torch.int32, "ea"); _req(ew, torch.int32, "ew")
    M, K = A.shape
    N = W.shape[0]
    if W.shape[1] != K or ea.shape != (M,) or ew.shape != (N,):
        raise ValueError("shape mismatch")
    if out is None:
        out = empty2d(M, N, torch.bfloat16, A.device)
    _req(out, torch.bfloat16, "out")
    wsb, wsn = _workspace(w8a8_workspace_size(M, N, K, split_k), A.device, ws)
    parts = ctypes.c_int(0)
    st = lib.detgemm_w8a8_split_exact(A.data_ptr(), _ld(A), W.data_ptr(), _ld(W), ea.data_ptr(), ew.data_ptr(),
                                      out.data_ptr(), _ld(out), M, N, K, split_k,
                                      wsb.data_ptr() if wsb is not None else None, wsn, ctypes.byref(parts),
                                      _stream(stream))
    _check(st, "detgemm_w8a8_split_exact")
    return out, parts.value


def _req_host(t: torch.Tensor, dtype, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if (t.dim() == 2 and t.stride(1) != 1) or (t.dim() == 1 and not t.is_contiguous()):
        raise ValueError(f"{name} must have unit stride along its last dimension")


def w8a8_host_buffer_size(M: int, N: int, K: int) -> int:
    return int(load().detgemm_w8a8_host_buffer_size(M, N, K))


def w8a8_host(A, W, ea, ew, out=None, buf=None, stream=None, sync: bool = True) -> torch.Tensor:
    """w8a8 on HOST tensors (pin them for overlap): A int8 [M,K], W int8 [N,K], ea/ew int32;
    returns a host bfloat16 tensor [M, N] (or writes ``out``). The host-to-device copies,
    the computation and the copy back are pipelined over chunks of rows on the current
    CUDA device; ``buf`` is the device scratch (allocated here if None). With sync=False
    the result is valid only after the stream has been synchronized."""
    lib = load()
    _req_host(A, torch.int8, "A"); _req_host(W, torch.int8, "W")
    _req_host(ea, torch.int32, "ea"); _req_host(ew, torch.int32, "ew")
    M, K = A.shape
    N = W.shape[0]
    if W.shape[1] != K or ea.shape != (M,) or ew.shape != (N,):
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, pin_memory=A.is_pinned())
    _req_host(out, torch.bfloat16, "out")
    dev = torch.device("cuda", torch.cuda.current_device())
    need = w8a8_host_buffer_size(M, N, K)
    if buf is None:
        buf = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if buf.numel() * buf.element_size() < need:
        raise ValueError(f"buffer too small: need {need} bytes")
    s = stream if stream is not None else torch.cuda.current_stream()
    st = lib.detgemm_w8a8_host(A.data_ptr(), A.stride(0) if M > 1 else K, W.data_ptr(), W.stride(0) if N > 1 else K,
                               ea.data_ptr(), ew.data_ptr(), out.data_ptr(), out.stride(0) if M > 1 else N,
                               M, N, K, buf.data_ptr(), buf.numel() * buf.element_size(), s.cuda_stream)
    _check(st, "detgemm_w8a8_host")
    if sync:
        s.synchronize()
    return out


def gemm_s8_i32(A, W, split_k: int = 1, out=None, ws=None, stream=None) -> torch.Tensor:
    """Exact int32 accumulator C = A W^T."""
    lib = load()
    _req(A, torch.int8, "A"); _req(W, torch.int8, "W")
    M, K = A.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("shape mismatch")
    if out is None:
        out = empty2d(M, N, torch.int32, A.device)
    _req(out, torch.int32, "out")
    wsb, wsn = _workspace(w8a8_workspace_size(M, N, K, split_k), A.device, ws)
    st = lib.detgemm_gemm_s8_i32(A.data_ptr(), _ld(A), W.data_ptr(), _ld(W), out.data_ptr(), _ld(out),
                                 M, N, K, split_k, wsb.data_ptr() if wsb is not None else None, wsn,
                                 _stream(stream))
    _check(st, "detgemm_gemm_s8_i32")
    return out


def quantize_pow2(X, mode: int = POW2_NEAREST, stream=None):
    """Per-row pow2 quantization of a bf16 or fp32 [rows, cols] tensor -> (Q int8, e int32)."""
    lib = load()
    if X.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif X.dtype == torch.float32:
        dt = DTYPE_F32
    else:
        raise TypeError("X must be bfloat16 or float32")
    _req(X, X.dtype, "X")
    rows, cols = X.shape
    Q = empty2d(rows, cols, torch.int8, X.device)
    e = torch.empty((rows,), dtype=torch.int32, device=X.device)
    st = lib.detgemm_quantize_pow2(X.data_ptr(), dt, _ld(X), rows, cols, mode, Q.data_ptr(), _ld(Q),
                                   e.data_ptr(), _stream(stream))
    _check(st, "detgemm_quantize_pow2")
    return Q, e


def linear_w8a8(X, W, ew, mode: int = POW2_NEAREST, W16=None, split_k: int = 1, out=None, ea_out=None, ws=None,
                stream=None, bias=None) -> torch.Tensor:
    """W8A8 linear layer on bf16/fp32 activations X [M, K]: per-row pow2 quantization of X
    fused with the exact GEMM against int8 W [N, K] (ew int32 [N]); bf16 [M, N] out.
    W16 (optional) is W widened once by widen_i8_f16; ea_out (optional) int32 [M] receives
    the activation exponents; bias (optional) bfloat16 [N] is added before the one rounding."""
    lib = load()
    if X.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif X.dtype == torch.float32:
        dt = DTYPE_F32
    else:
        raise TypeError("X must be bfloat16 or float32")
    _req(X, X.dtype, "X"); _req(W, torch.int8, "W"); _req(ew, torch.int32, "ew")
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K or ew.shape != (N,):
        raise ValueError("shape mismatch")
    if W16 is not None:
        _req(W16, torch.float16, "W16")
        if W16.shape != (N, K):
            raise ValueError("W16 shape mismatch")
    if ea_out is not None:
        _req(ea_out, torch.int32, "ea_out")
        if ea_out.shape != (M,):
            raise ValueError("ea_out shape mismatch")
    if out is None:
        out = empty2d(M, N, torch.bfloat16, X.device)
    _req(out, torch.bfloat16, "out")
    bias = _bias_vec(bias, N, X.device)
    need = int(lib.detgemm_linear_w8a8_workspace_size(M, N, K, split_k, 1 if W16 is not None else 0))
    wsb, wsn = _workspace(need, X.device, ws)
    w16p, w16ld = (W16.data_ptr(), _ld(W16)) if W16 is not None else (None, 0)
    eap = ea_out.data_ptr() if ea_out is not None else None
    wsp = wsb.data_ptr() if wsb is not None else None
    if bias is not None:
        st = lib.detgemm_linear_w8a8_bias(X.data_ptr(), dt, _ld(X), mode, W.data_ptr(), _ld(W), w16p, w16ld,
                                          ew.data_ptr(), bias.data_ptr(), out.data_ptr(), _ld(out), eap, M, N, K,
                                          split_k, wsp, wsn, _stream(stream))
        _check(st, "detgemm_linear_w8a8_bias")
        return out
    st = lib.detgemm_linear_w8a8(X.data_ptr(), dt, _ld(X), mode, W.data_ptr(), _ld(W), w16p, w16ld,
                                 ew.data_ptr(), out.data_ptr(), _ld(out), eap, M, N, K, split_k, wsp, wsn,
                                 _stream(stream))
    _check(st, "detgemm_linear_w8a8")
    return out


def slice_f32(X, axis: int = AXIS_ROWS, nslices: int = 7, stream=None):
    """Ozaki digits of fp32 X: (S int8 [nslices, rows, cols] or [nslices, cols, rows], e int32)."""
    lib = load()
    _req(X, torch.float32, "X")
    rows, cols = X.shape
    shape = (nslices, rows, cols) if axis == AXIS_ROWS else (nslices, cols, rows)
    S = torch.empty(shape, dtype=torch.int8, device=X.device)
    e = torch.empty((rows if axis == AXIS_ROWS else cols,), dtype=torch.int32, device=X.device)
    st = lib.detgemm_slice_f32(X.data_ptr(), _ld(X), rows, cols, axis, nslices, S.data_ptr(), e.data_ptr(),
                               _stream(stream))
    _check(st, "detgemm_slice_f32")
    return S, e


def ozaki_f32(A, B, nslices: int = 7, max_diag: int = 8, split_k: int = 1, out=None, ws=None,
              stream=None) -> torch.Tensor:
    """Ozaki-scheme fp32 GEMM C = A B (A [M,K], B [K,N] fp32 row-major)."""
    lib = load()
    _req(A, torch.float32, "A"); _req(B, torch.float32, "B")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("shape mismatch")
    if out is None:
        out = empty2d(M, N, torch.float32, A.device)
    _req(out, torch.float32, "out")
    need = ozaki_workspace_size(M, N, K, nslices, max_diag, split_k)
    wsb, wsn = _workspace(need, A.device, ws)
    st = lib.detgemm_ozaki_f32(A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), out.data_ptr(), _ld(out),
                               M, N, K, nslices, max_diag, split_k,
                               wsb.data_ptr() if wsb is not None else None, wsn, _stream(stream))
    _check(st, "detgemm_ozaki_f32")
    return out


def ozaki_f32_split_exact(A, B, split_k: int, nslices: int = 7, max_diag: int = 8, out=None, ws=None,
                          stream=None):
    """ozaki_f32 with every diagonal's K range cut into exactly split_k parts
    (detgemm_ozaki_f32_split_exact): returns (C, parts_run)."""
    lib = load()
    _req(A, torch.float32, "A"); _req(B, torch.float32, "B")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("shape mismatch")
    if out is None:
        out = empty2d(M, N, torch.float32, A.device)
    _req(out, torch.float32, "out")
    wsb, wsn = _workspace(ozaki_workspace_size(M, N, K, nslices, max_diag, split_k), A.device, ws)
    parts = ctypes.c_int(0)
    st = lib.detgemm_ozaki_f32_split_exact(A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), out.data_ptr(), _ld(out),
                                           M, N, K, nslices, max_diag, split_k,
                                           wsb.data_ptr() if wsb is not None else None, wsn, ctypes.byref(parts),
                                           _stream(stream))
    _check(st, "detgemm_ozaki_f32_split_exact")
    return out, parts.value


def ozaki_combine(T, e, f, out=None, dtype=torch.float32, stream=None) -> torch.Tensor:
    """Fixed-order recombination of exact diagonal sums: T int32 [max_diag - 1, M, N]
    (plane p holds the diagonal g = max_diag - p), e int32 [M], f int32 [N] -> fp32 or
    fp64 [M, N] (``dtype``)."""
    lib = load()
    _req(T, torch.int32, "T"); _req(e, torch.int32, "e"); _req(f, torch.int32, "f")
    if T.dim() != 3 or T.stride(2) != 1 or T.stride(0) != T.shape[1] * T.stride(1):
        raise ValueError("T must be [planes, M, N] with contiguous rows and planes")
    nd, M, N = T.shape
    if e.shape != (M,) or f.shape != (N,):
        raise ValueError("shape mismatch")
    if dtype not in (torch.float32, torch.float64):
        raise TypeError("dtype must be float32 or float64")
    if out is None:
        out = empty2d(M, N, dtype, T.device)
    _req(out, dtype, "out")
    cdt = DTYPE_F64 if dtype == torch.float64 else DTYPE_F32
    st = lib.detgemm_ozaki_combine(T.data_ptr(), T.stride(1), nd + 1, e.data_ptr(), f.data_ptr(), out.data_ptr(),
                                   cdt, _ld(out), M, N, _stream(stream))
    _check(st, "detgemm_ozaki_combine")
    return out


def slice_f64(X, axis: int = AXIS_ROWS, nslices: int = 8, stream=None):
    """Ozaki digits of fp64 X: (S int8 [nslices, rows, cols] or [nslices, cols, rows], e int32)."""
    lib = load()
    _req(X, torch.float64, "X")
    rows, cols = X.shape
    shape = (nslices, rows, cols) if axis == AXIS_ROWS else (nslices, cols, rows)
    S = torch.empty(shape, dtype=torch.int8, device=X.device)
    e = torch.empty((rows if axis == AXIS_ROWS else cols,), dtype=torch.int32, device=X.device)
    st = lib.detgemm_slice_f64(X.data_ptr(), _ld(X), rows, cols, axis, nslices, S.data_ptr(), e.data_ptr(),
                               _stream(stream))
    _check(st, "detgemm_slice_f64")
    return S, e


def ozaki_f64_workspace_size(M, N, K, nslices=8, max_diag=9, split_k=1) -> int:
    return int(load().detgemm_ozaki_f64_workspace_size(M, N, K, nslices, max_diag, split_k))


def ozaki_f64(A, B, nslices: int = 8, max_diag: int = 9, split_k: int = 1, out=None, ws=None,
              stream=None) -> torch.Tensor:
    """fp64-target Ozaki-scheme GEMM C = A B (A [M,K], B [K,N] fp64 row-major)."""
    lib = load()
    _req(A, torch.float64, "A"); _req(B, torch.float64, "B")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("shape mismatch")
    if out is None:
        out = empty2d(M, N, torch.float64, A.device)
    _req(out, torch.float64, "out")
    need = ozaki_f64_workspace_size(M, N, K, nslices, max_diag, split_k)
    wsb, wsn = _workspace(need, A.device, ws)
    st = lib.detgemm_ozaki_f64(A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), out.data_ptr(), _ld(out),
                               M, N, K, nslices, max_diag, split_k,
                               wsb.data_ptr() if wsb is not None else None, wsn, _stream(stream))
    _check(st, "detgemm_ozaki_f64")
    return out


def w8a8_swiglu(A, Wg, Wu, ea, ewg, ewu, out=None, ws=None, stream=None) -> torch.Tensor:
    """Fused gated-linear-unit W8A8: C = rne_bf16(SiLU(A Wg^T 2^(ea+ewg)) * A Wu^T 2^(ea+ewu));
    A int8 [M,K], Wg / Wu int8 [N,K] (same row stride), exponents int32; bf16 [M, N] out."""
    lib = load()
    _req(A, torch.int8, "A"); _req(Wg, torch.int8, "Wg"); _req(Wu, torch.int8, "Wu")
    _req(ea, torch.int32, "ea"); _req(ewg, torch.int32, "ewg"); _req(ewu, torch.int32, "ewu")
    M, K = A.shape
    N = Wg.shape[0]
    if Wg.shape != (N, K) or Wu.shape != (N, K) or ea.shape != (M,) or ewg.shape != (N,) or ewu.shape != (N,):
        raise ValueError("shape mismatch")
    if _ld(Wg) != _ld(Wu):
        raise ValueError("Wg and Wu must share a row stride")
    if out is None:
        out = empty2d(M, N, torch.bfloat16, A.device)
    _req(out, torch.bfloat16, "out")
    wsb, wsn = _workspace(int(lib.detgemm_w8a8_swiglu_workspace_size(M, N, K)), A.device, ws)
    st = lib.detgemm_w8a8_swiglu(A.data_ptr(), _ld(A), Wg.data_ptr(), Wu.data_ptr(), _ld(Wg), ea.data_ptr(),
                                 ewg.data_ptr(), ewu.data_ptr(), out.data_ptr(), _ld(out), M, N, K,
                                 wsb.data_ptr() if wsb is not None else None, wsn, _stream(stream))
    _check(st, "detgemm_w8a8_swiglu")
    return out


def swiglu_bf16(G, U, ea, ewg, ewu, out=None, stream=None) -> torch.Tensor:
    """C = rne_bf16(SiLU(G 2^(ea+ewg)) * U 2^(ea+ewu)) on exact int32 accumulators G, U [M, N]
    (ea int32 [M], ewg / ewu int32 [N]); bf16 [M, N] out, rounded once."""
    lib = load()
    _req(G, torch.int32, "G"); _req(U, torch.int32, "U")
    _req(ea, torch.int32, "ea"); _req(ewg, torch.int32, "ewg"); _req(ewu, torch.int32, "ewu")
    M, N = G.shape
    if U.shape != (M, N) or ea.shape != (M,) or ewg.shape != (N,) or ewu.shape != (N,):
        raise ValueError("shape mismatch")
    if out is None:
        out = empty2d(M, N, torch.bfloat16, G.device)
    _req(out, torch.bfloat16, "out")
    st = lib.detgemm_swiglu_bf16(G.data_ptr(), _ld(G), U.data_ptr(), _ld(U), ea.data_ptr(), ewg.data_ptr(),
                                 ewu.data_ptr(), out.data_ptr(), _ld(out), M, N, _stream(stream))
    _check(st, "detgemm_swiglu_bf16")
    return out


def gemm_fixed_f16(A, W, out=None, stream=None) -> torch.Tensor:
    """Fixed-order fp16/bf16 GEMM C = A W^T (A [M,K], W [N,K], both float16 or both bfloat16):
    K walked in 16-wide tensor-core block FMAs from +0, never split; fp32 [M, N] out."""
    lib = load()
    if A.dtype not in (torch.float16, torch.bfloat16) or W.dtype != A.dtype:
        raise TypeError("A and W must both be float16 or both bfloat16")
    _req(A, A.dtype, "A"); _req(W, W.dtype, "W")
    M, K = A.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("shape mismatch")
    if out is None:
        out = empty2d(M, N, torch.float32, A.device)
    _req(out, torch.float32, "out")
    dt = DTYPE_BF16 if A.dtype == torch.bfloat16 else DTYPE_F16
    st = lib.detgemm_gemm_fixed_f16(A.data_ptr(), _ld(A), W.data_ptr(), _ld(W), out.data_ptr(), _ld(out), M, N, K, dt,
                                    _stream(stream))
    _check(st, "detgemm_gemm_fixed_f16")
    return out


def widen_i8_f16(X, stream=None) -> torch.Tensor:
    """Exact int8 -> fp16 copy [rows, cols] (row stride padded to 16 bytes, padding zeroed)."""
    lib = load()
    _req(X, torch.int8, "X")
    rows, cols = X.shape
    Y = empty2d(rows, cols, torch.float16, X.device)
    st = lib.detgemm_widen_i8_f16(X.data_ptr(), _ld(X), rows, cols, Y.data_ptr(), _ld(Y), _stream(stream))
    _check(st, "detgemm_widen_i8_f16")
    return Y


def w8a8_f16ops(A16, W16, ea, ew, split_k: int = 1, out=None, ws=None, stream=None) -> torch.Tensor:
    """W8A8 on operands widened by widen_i8_f16 (fp16 tensors holding int8 values)."""
    lib = load()
    _req(A16, torch.float16, "A16"); _req(W16, torch.float16, "W16")
    _req(ea, torch.int32, "ea"); _req(ew, torch.int32, "ew")
    M, K = A16.shape
    N = W16.shape[0]
    if W16.shape[1] != K or ea.shape != (M,) or ew.shape != (N,):
        raise ValueError("shape mismatch")
    if out is None:
        out = empty2d(M, N, torch.bfloat16, A16.device)
    _req(out, torch.bfloat16, "out")
    need = int(lib.detgemm_w8a8_f16ops_workspace_size(M, N, K, split_k))
    wsb, wsn = _workspace(need, A16.device, ws)
    st = lib.detgemm_w8a8_f16ops(A16.data_ptr(), _ld(A16), W16.data_ptr(), _ld(W16), ea.data_ptr(), ew.data_ptr(),
                                 out.data_ptr(), _ld(out), M, N, K, split_k,
                                 wsb.data_ptr() if wsb is not None else None, wsn, _stream(stream))
    _check(st, "detgemm_w8a8_f16ops")
    return out


FAULT_NONE, FAULT_F1_SCALE_PRECISION, FAULT_F2_DOUBLE_ROUNDING, FAULT_F3_ORDER, FAULT_F4_TRUNCATION = 0, 1, 2, 3, 4
SEVERITY_ONE, SEVERITY_ONE_PERCENT, SEVERITY_ALL = 0, 1, 2
SCALES_POW2, SCALES_F32 = 0, 1


def epilogue_inject(acc, sa, sw, fault: int = FAULT_NONE, severity: int = SEVERITY_ALL, seed: int = 0, out=None,
                    stream=None) -> torch.Tensor:
    """The W8A8 epilogue, or one injected fault (see include/detgemm_conformance.h), on exact
    int32 accumulators acc [M, N]; sa [M] / sw [N] are int32 exponents (power-of-two scales)
    or float32 scales. Returns bf16 [M, N]."""
    lib = load()
    _req(acc, torch.int32, "acc")
    M, N = acc.shape
    if sa.dtype == torch.int32 and sw.dtype == torch.int32:
        scales = SCALES_POW2
    elif sa.dtype == torch.float32 and sw.dtype == torch.float32:
        scales = SCALES_F32
    else:
        raise TypeError("sa and sw must both be int32 exponents or both float32 scales")
    _req(sa, sa.dtype, "sa"); _req(sw, sw.dtype, "sw")
    if sa.shape != (M,) or sw.shape != (N,):
        raise ValueError("shape mismatch")
    if out is None:
        out = empty2d(M, N, torch.bfloat16, acc.device)
    _req(out, torch.bfloat16, "out")
    st = lib.detgemm_epilogue_inject(acc.data_ptr(), _ld(acc), scales, sa.data_ptr(), sw.data_ptr(), fault, severity,
                                     seed & 0xFFFFFFFF, out.data_ptr(), _ld(out), M, N, _stream(stream))
    _check(st, "detgemm_epilogue_inject")
    return out


def selftest_timeout(limit_ms: int = 100, stream=None) -> None:
    """Launch the bounded-wait self-check (expires after limit_ms; see device_status)."""
    _check(load().detgemm_selftest_timeout(limit_ms, _stream(stream)), "detgemm_selftest_timeout")


def device_status(stream=None) -> int:
    """Synchronize the stream; return and clear the device status (OK, ERR_NONFINITE, ERR_TIMEOUT)."""
    return int(load().detgemm_get_device_status(_stream(stream)))
