"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

This package draws operand values only (see ``gen.c`` for the counter-based
generator); it holds none of the method's arithmetic. Tests and the bench draw
inputs here and hand the very same arrays to both sides.

Workload recipes (the shapes and value distributions of the five workloads the
method is exercised on; seeds fixed per workload, one stream id per tensor):

* ``tiny``     A int8 64x512, W int8 256x512 uniform in [-127, 127];
               ea[64], ew[256] uniform in [-12, -4]; seed 0.
* ``sweep``    W int8 6144x2048 ~ rne(N(0, 40)) clipped to +-127; A int8 2048x2048
               ~ rne(N(0, 20)) clipped; exponents in [-14, -6]; seed 1. Smaller M
               takes the first M rows of A and of ea.
* ``ffn``      gate/up: A 8192x4096, W 12288x4096; down: A 8192x12288,
               W 4096x12288; int8 ~ rne(N(0, 30)) clipped; exponents in [-14, -6]; seed 2.
* ``skinny``   A int8 16x65536, W int8 4096x65536 uniform in [-127, 127];
               exponents in [-16, -8]; seed 3.
* ``ozaki``    A, B fp32 4096x4096, entries N(0, 1) * 2^U, U uniform integer in
               [-8, 8]; seed 4.

Weights are drawn directly in the nn.Linear storage order W = B^T, i.e. [N x K]
row-major (K contiguous), element (j, k) at index j*K + k.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libsynthetic.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gen.c`` into ``libsynthetic.so`` next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
             _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, i32, dbl, ptr = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_double, ctypes.c_void_p)
            lib.gen_uniform_i8.argtypes = [u64, u64, i64, i32, i32, ptr]
            lib.gen_uniform_i32.argtypes = [u64, u64, i64, i32, i32, ptr]
            lib.gen_normal_i8.argtypes = [u64, u64, i64, dbl, i32, ptr]
            lib.gen_normal_pow2_f32.argtypes = [u64, u64, i64, i32, i32, ptr]
            lib.gen_normal_f32.argtypes = [u64, u64, i64, dbl, ptr]
            lib.gen_normal_pow2_f64.argtypes = [u64, u64, i64, i32, i32, ptr]
            for f in (lib.gen_uniform_i8, lib.gen_uniform_i32, lib.gen_normal_i8,
                      lib.gen_normal_pow2_f32, lib.gen_normal_f32, lib.gen_normal_pow2_f64):
                f.restype = None
            _lib = lib
    return _lib


def _out(shape, dtype, out):
    if out is None:
        out = np.empty(shape, dtype=dtype)
    assert out.dtype == dtype and out.flags.c_contiguous and out.shape == tuple(shape)
    return out


def uniform_i8(seed, stream, shape, lo=-127, hi=127, out=None):
    out = _out(shape, np.int8, out)
    _load().gen_uniform_i8(seed, stream, out.size, lo, hi, out.ctypes.data)
    return out


def uniform_i32(seed, stream, shape, lo, hi, out=None):
    out = _out(shape, np.int32, out)
    _load().gen_uniform_i32(seed, stream, out.size, lo, hi, out.ctypes.data)
    return out


def normal_i8(seed, stream, shape, sigma, clip=127, out=None):
    out = _out(shape, np.int8, out)
    _load().gen_normal_i8(seed, stream, out.size, float(sigma), clip, out.ctypes.data)
    return out


def normal_pow2_f32(seed, stream, shape, ulo=-8, uhi=8, out=None):
    out = _out(shape, np.float32, out)
    _load().gen_normal_pow2_f32(seed, stream, out.size, ulo, uhi, out.ctypes.data)
    return out


def normal_pow2_f64(seed, stream, shape, ulo=0, uhi=0, out=None):
    out = _out(shape, np.float64, out)
    _load().gen_normal_pow2_f64(seed, stream, out.size, ulo, uhi, out.ctypes.data)
    return out


def normal_f32(seed, stream, shape, sigma=1.0, out=None):
    out = _out(shape, np.float32, out)
    _load().gen_normal_f32(seed, stream, out.size, float(sigma), out.ctypes.data)
    return out


# ----------------------------------------------------------------------------------------
# Workload recipes
# ----------------------------------------------------------------------------------------

def w8a8_uniform(seed, M, N, K, elo, ehi, lo=-127, hi=127):
    """Uniform int8 operands and uniform integer exponents (tiny / skinny recipes)."""
    A = uniform_i8(seed, 0, (M, K), lo, hi)
    W = uniform_i8(seed, 1, (N, K), lo, hi)
    ea = uniform_i32(seed, 2, (M,), elo, ehi)
    ew = uniform_i32(seed, 3, (N,), elo, ehi)
    return A, W, ea, ew


def w8a8_normal(seed, M, N, K, sigma_a, sigma_w, elo, ehi, streams=(0, 1, 2, 3)):
    """Rounded-normal int8 operands clipped to +-127 (sweep / ffn recipes)."""
    A = normal_i8(seed, streams[0], (M, K), sigma_a)
    W = normal_i8(seed, streams[1], (N, K), sigma_w)
    ea = uniform_i32(seed, streams[2], (M,), elo, ehi)
    ew = uniform_i32(seed, streams[3], (N,), elo, ehi)
    return A, W, ea, ew


def tiny():
    """64x256x512 uniform int8, exponents in [-12, -4], seed 0."""
    return w8a8_uniform(0, 64, 256, 512, -12, -4)


def sweep(M=2048):
    """K=2048, N=6144 linear; rows 0..M-1 of one 2048-row draw, seed 1."""
    A, W, ea, ew = w8a8_normal(1, 2048, 6144, 2048, 20.0, 40.0, -14, -6)
    return np.ascontiguousarray(A[:M]), W, np.ascontiguousarray(ea[:M]), ew


def ffn_gate_up(M=8192):
    """Gate/up GEMM of the 8B-class FFN: K=4096, N=12288, seed 2 streams 0-3."""
    return w8a8_normal(2, M, 12288, 4096, 30.0, 30.0, -14, -6, streams=(0, 1, 2, 3))


def ffn_down(M=8192):
    """Down GEMM of the 8B-class FFN: K=12288, N=4096, seed 2 streams 4-7."""
    return w8a8_normal(2, M, 4096, 12288, 30.0, 30.0, -14, -6, streams=(4, 5, 6, 7))


def skinny():
    """Decode-shaped M=16, N=4096, K=65536 uniform int8, exponents in [-16, -8], seed 3."""
    return w8a8_uniform(3, 16, 4096, 65536, -16, -8)


def ozaki(n=4096, seed=4):
    """fp32 A, B (n x n, row-major) with entries N(0,1) * 2^U, U in [-8, 8]."""
    A = normal_pow2_f32(seed, 0, (n, n), -8, 8)
    B = normal_pow2_f32(seed, 1, (n, n), -8, 8)
    return A, B


def ozaki_f64(n=4096, seed=5, ulo=0, uhi=0):
    """fp64 A, B (n x n, row-major) with entries N(0,1) * 2^U, U uniform in [ulo, uhi]."""
    A = normal_pow2_f64(seed, 0, (n, n), ulo, uhi)
    B = normal_pow2_f64(seed, 1, (n, n), ulo, uhi)
    return A, B
