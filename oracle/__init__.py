"""CPU oracle for the batch-invariant exact GEMM — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and its
Python binding) never imports, links or runs anything here, and this package
imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C, int64 triple loops, exact
power-of-two scaling, software round-to-nearest-even); this module only
compiles it with gcc and marshals numpy arrays into it.

Pins: every function here is checked in ``tests/test_oracle_*.py`` against
exact-rational brute force, hand-worked values, closed forms and invariants.
The slicing/combine *variant* of the Ozaki scheme (truncated 7-bit digits,
combine order g = max_diag..2) is the design's reading of a step the source
page leaves open; its bits are pinned to that written definition by a
Fraction-based brute force and tied to the page only through the error bound.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_PRECONDITION, ERR_NONFINITE = 0, 3, 8
BF16, F32, F16 = 0, 1, 3
NEAREST, CEIL = 0, 1
ROWS, COLS = 0, 1


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (gcc -O2, no FP contraction, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        # binary128 arithmetic: long double on AArch64, __float128 with libquadmath elsewhere
        quad = [] if platform.machine() in ("aarch64", "arm64") else ["-lquadmath"]
        subprocess.check_call(
            ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
             "-fopenmp", _SRC, "-o", tmp, "-lm"] + quad)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.oracle_rne_bf16.argtypes = [ctypes.c_double]
            lib.oracle_rne_bf16.restype = ctypes.c_uint16
            lib.oracle_w8a8.argtypes = [p, i64, p, i64, p, p, p, i64, i32, i32, i32, p, i32]
            lib.oracle_bias_round.argtypes = [i64, i64, ctypes.c_uint16]
            lib.oracle_bias_round.restype = ctypes.c_uint16
            lib.oracle_w8a8_bias.argtypes = [p, i64, p, i64, p, p, p, p, i64, i32, i32, i32, p, i32]
            lib.oracle_gemm_s8_i32.argtypes = [p, i64, p, i64, p, i64, i32, i32, i32, p, i32]
            lib.oracle_quantize_pow2.argtypes = [p, i32, i64, i32, i32, i32, p, i64, p]
            lib.oracle_slice_f32.argtypes = [p, i64, i32, i32, i32, i32, p, p]
            lib.oracle_ozaki_f32.argtypes = [p, i64, p, i64, p, i64, i32, i32, i32, i32, i32, p, i32]
            lib.oracle_ozaki_diagonals.argtypes = [p, p, i32, i32, i32, i32, i32, p]
            lib.oracle_ozaki_combine.argtypes = [p, i64, i32, p, p, p, i64, i32, i32]
            lib.oracle_ozaki_combine_f64.argtypes = [p, i64, i32, p, p, p, i64, i32, i32]
            lib.oracle_slice_f64.argtypes = [p, i64, i32, i32, i32, i32, p, p]
            lib.oracle_ozaki_f64.argtypes = [p, i64, p, i64, p, i64, i32, i32, i32, i32, i32, p, i32]
            lib.oracle_gemm_blockfma.argtypes = [p, i64, p, i64, i32, i32, i32, p, i64, i32, i32, i32]
            lib.oracle_silu_mul_bf16.argtypes = [i32, i32, i32, i32, p]
            lib.oracle_w8a8_swiglu.argtypes = [p, i64, p, p, i64, p, p, p, p, i64, i32, i32, i32, p, i32]
            for f in (lib.oracle_w8a8, lib.oracle_w8a8_bias, lib.oracle_gemm_s8_i32, lib.oracle_quantize_pow2,
                      lib.oracle_slice_f32, lib.oracle_ozaki_f32, lib.oracle_ozaki_diagonals,
                      lib.oracle_ozaki_combine, lib.oracle_ozaki_combine_f64, lib.oracle_slice_f64,
                      lib.oracle_ozaki_f64, lib.oracle_gemm_blockfma, lib.oracle_silu_mul_bf16,
                      lib.oracle_w8a8_swiglu):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _c(a, dtype):
    a = np.asarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return np.ascontiguousarray(a)


def _rows(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    return r, int(r.size)


def rne_bf16(v: float) -> int:
    """bf16 bits of the round-to-nearest-even of a double."""
    return int(_load().oracle_rne_bf16(float(v)))


def w8a8(A, W, ea, ew, rows=None, check=True):
    """C = rne_bf16((A W^T) * 2^(ea_i + ew_j)) as uint16 bf16 bits [rows x N]."""
    A, W = _c(A, np.int8), _c(W, np.int8)
    ea, ew = _c(ea, np.int32), _c(ew, np.int32)
    M, K = A.shape
    N = W.shape[0]
    assert W.shape[1] == K and ea.shape == (M,) and ew.shape == (N,)
    r, nr = _rows(rows)
    C = np.empty((nr if r is not None else M, N), dtype=np.uint16)
    st = _load().oracle_w8a8(A.ctypes.data, K, W.ctypes.data, K, ea.ctypes.data, ew.ctypes.data,
                             C.ctypes.data, N, M, N, K, r.ctypes.data if r is not None else None, nr)
    if check and st != OK:
        raise OracleError(f"oracle_w8a8 status {st}")
    return C


def bias_round(acc: int, E: int, b: int) -> int:
    """bf16 bits of rne_bf16(acc * 2^E + b) for an int64 acc and the bf16 bit pattern b."""
    return int(_load().oracle_bias_round(int(acc), int(E), int(b)))


def w8a8_bias(A, W, ea, ew, bias, rows=None, check=True):
    """C = rne_bf16((A W^T) * 2^(ea_i + ew_j) + b_j) as uint16 bf16 bits [rows x N]; bias is
    uint16 bf16 bits [N]."""
    A, W = _c(A, np.int8), _c(W, np.int8)
    ea, ew, bias = _c(ea, np.int32), _c(ew, np.int32), _c(bias, np.uint16)
    M, K = A.shape
    N = W.shape[0]
    assert W.shape[1] == K and ea.shape == (M,) and ew.shape == (N,) and bias.shape == (N,)
    r, nr = _rows(rows)
    C = np.empty((nr if r is not None else M, N), dtype=np.uint16)
    st = _load().oracle_w8a8_bias(A.ctypes.data, K, W.ctypes.data, K, ea.ctypes.data, ew.ctypes.data,
                                  bias.ctypes.data, C.ctypes.data, N, M, N, K,
                                  r.ctypes.data if r is not None else None, nr)
    if check and st != OK:
        raise OracleError(f"oracle_w8a8_bias status {st}")
    return C


def gemm_s8_i32(A, W, rows=None, check=True):
    """Exact accumulator C = A W^T as int32 [rows x N]."""
    A, W = _c(A, np.int8), _c(W, np.int8)
    M, K = A.shape
    N = W.shape[0]
    r, nr = _rows(rows)
    C = np.empty((nr if r is not None else M, N), dtype=np.int32)
    st = _load().oracle_gemm_s8_i32(A.ctypes.data, K, W.ctypes.data, K, C.ctypes.data, N, M, N, K,
                                    r.ctypes.data if r is not None else None, nr)
    if check and st != OK:
        raise OracleError(f"oracle_gemm_s8_i32 status {st}")
    return C


def quantize_pow2(X, mode=NEAREST, check=True):
    """Per-row pow2 quantization. X: float32 array or uint16 bf16 bits. Returns (Q, e)."""
    X = np.ascontiguousarray(X)
    if X.dtype == np.uint16:
        dt = BF16
    elif X.dtype == np.float32:
        dt = F32
    else:
        raise TypeError(X.dtype)
    rows, cols = X.shape
    Q = np.empty((rows, cols), dtype=np.int8)
    e = np.empty((rows,), dtype=np.int32)
    st = _load().oracle_quantize_pow2(X.ctypes.data, dt, cols, rows, cols, mode, Q.ctypes.data,
                                      cols, e.ctypes.data)
    if check and st != OK:
        raise OracleError(f"oracle_quantize_pow2 status {st}")
    return Q, e


def slice_f32(X, axis=ROWS, nslices=7, check=True):
    """Ozaki digits. Returns (S, e): S int8 [nslices x rows x cols] for axis ROWS,
    [nslices x cols x rows] for axis COLS; e int32 per row / per column."""
    X = _c(X, np.float32)
    rows, cols = X.shape
    S = np.empty((nslices, rows, cols) if axis == ROWS else (nslices, cols, rows), dtype=np.int8)
    e = np.empty((rows if axis == ROWS else cols,), dtype=np.int32)
    st = _load().oracle_slice_f32(X.ctypes.data, cols, rows, cols, axis, nslices, S.ctypes.data,
                                  e.ctypes.data)
    if check and st != OK:
        raise OracleError(f"oracle_slice_f32 status {st}")
    return S, e


def slice_f64(X, axis=ROWS, nslices=8, check=True):
    """Ozaki digits of an fp64 matrix (same layout as slice_f32)."""
    X = _c(X, np.float64)
    rows, cols = X.shape
    S = np.empty((nslices, rows, cols) if axis == ROWS else (nslices, cols, rows), dtype=np.int8)
    e = np.empty((rows if axis == ROWS else cols,), dtype=np.int32)
    st = _load().oracle_slice_f64(X.ctypes.data, cols, rows, cols, axis, nslices, S.ctypes.data,
                                  e.ctypes.data)
    if check and st != OK:
        raise OracleError(f"oracle_slice_f64 status {st}")
    return S, e


def ozaki_f32(A, B, nslices=7, max_diag=8, rows=None, check=True):
    """Ozaki-scheme fp32 GEMM C = A B (fp32 [rows x N])."""
    A, B = _c(A, np.float32), _c(B, np.float32)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    r, nr = _rows(rows)
    C = np.empty((nr if r is not None else M, N), dtype=np.float32)
    st = _load().oracle_ozaki_f32(A.ctypes.data, K, B.ctypes.data, N, C.ctypes.data, N, M, N, K,
                                  nslices, max_diag, r.ctypes.data if r is not None else None, nr)
    if check and st != OK:
        raise OracleError(f"oracle_ozaki_f32 status {st}")
    return C


def ozaki_f64(A, B, nslices=8, max_diag=9, rows=None, check=True):
    """fp64-target Ozaki-scheme GEMM C = A B (fp64 [rows x N])."""
    A, B = _c(A, np.float64), _c(B, np.float64)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    r, nr = _rows(rows)
    C = np.empty((nr if r is not None else M, N), dtype=np.float64)
    st = _load().oracle_ozaki_f64(A.ctypes.data, K, B.ctypes.data, N, C.ctypes.data, N, M, N, K,
                                  nslices, max_diag, r.ctypes.data if r is not None else None, nr)
    if check and st != OK:
        raise OracleError(f"oracle_ozaki_f64 status {st}")
    return C


def ozaki_diagonals(DA, DB, max_diag=8):
    """Exact per-diagonal sums T[i, j, g] (int64) from digit planes DA [s x M x K], DB [s x N x K]."""
    DA, DB = _c(DA, np.int8), _c(DB, np.int8)
    ns, M, K = DA.shape
    ns2, N, K2 = DB.shape
    assert ns == ns2 and K == K2
    T = np.empty((M, N, max_diag + 1), dtype=np.int64)
    _load().oracle_ozaki_diagonals(DA.ctypes.data, DB.ctypes.data, M, N, K, ns, max_diag, T.ctypes.data)
    return T


def ozaki_combine(T, e, f):
    """Fixed-order fp64 recombination of diagonal sums. T int32 [max_diag - 1, M, N],
    plane p holding the diagonal g = max_diag - p; e int32 [M], f int32 [N]. fp32 [M, N]."""
    T = _c(T, np.int32)
    e, f = _c(e, np.int32), _c(f, np.int32)
    nd, M, N = T.shape
    assert e.shape == (M,) and f.shape == (N,) and 1 <= nd <= 17
    C = np.empty((M, N), dtype=np.float32)
    _load().oracle_ozaki_combine(T.ctypes.data, N, nd + 1, e.ctypes.data, f.ctypes.data, C.ctypes.data, N, M, N)
    return C


def ozaki_combine_f64(T, e, f):
    """The fp64-target recombination: as ozaki_combine, result rounded to fp64 [M, N]."""
    T = _c(T, np.int32)
    e, f = _c(e, np.int32), _c(f, np.int32)
    nd, M, N = T.shape
    assert e.shape == (M,) and f.shape == (N,) and 1 <= nd <= 17
    C = np.empty((M, N), dtype=np.float64)
    _load().oracle_ozaki_combine_f64(T.ctypes.data, N, nd + 1, e.ctypes.data, f.ctypes.data, C.ctypes.data, N, M, N)
    return C


def gemm_blockfma(A, W, dtype=BF16, nfma=16, neab=2):
    """Fixed-order fp16/bf16 GEMM under the tensor-core block-FMA model: A [M, K] and W [N, K]
    as uint16 bit patterns (dtype BF16 or F16); returns fp32 bit patterns [M, N] (uint32)."""
    A = _c(A, np.uint16)
    W = _c(W, np.uint16)
    M, K = A.shape
    N = W.shape[0]
    assert W.shape[1] == K
    C = np.zeros((M, N), np.uint32)
    st = _load().oracle_gemm_blockfma(A.ctypes.data, K, W.ctypes.data, K, dtype, nfma, neab, C.ctypes.data, N,
                                      M, N, K)
    if st != OK:
        raise OracleError(f"oracle_gemm_blockfma: status {st}")
    return C


def silu_mul_bf16(gacc: int, uacc: int, Eg: int, Eu: int) -> int:
    """bf16 bits of rne(SiLU(g) * u) for g = gacc * 2^Eg, u = uacc * 2^Eu (exact reals)."""
    out = ctypes.c_uint16(0)
    st = _load().oracle_silu_mul_bf16(int(gacc), int(uacc), int(Eg), int(Eu), ctypes.byref(out))
    if st != OK:
        raise OracleError(f"oracle_silu_mul_bf16: status {st}")
    return int(out.value)


def w8a8_swiglu(A, Wg, Wu, ea, ewg, ewu, rows=None):
    """C = rne_bf16(SiLU(A Wg^T * 2^(ea+ewg)) * (A Wu^T * 2^(ea+ewu))), exact sums, one rounding."""
    A = _c(A, np.int8)
    Wg = _c(Wg, np.int8)
    Wu = _c(Wu, np.int8)
    ea, ewg, ewu = (_c(x, np.int32) for x in (ea, ewg, ewu))
    M, K = A.shape
    N = Wg.shape[0]
    assert Wg.shape == Wu.shape == (N, K)
    r, nr = _rows(rows)
    C = np.zeros((nr if rows is not None else M, N), np.uint16)
    st = _load().oracle_w8a8_swiglu(A.ctypes.data, K, Wg.ctypes.data, Wu.ctypes.data, K, ea.ctypes.data,
                                    ewg.ctypes.data, ewu.ctypes.data, C.ctypes.data, N, M, N, K,
                                    r.ctypes.data if r is not None else None, nr)
    if st != OK:
        raise OracleError(f"oracle_w8a8_swiglu: status {st}")
    return C
