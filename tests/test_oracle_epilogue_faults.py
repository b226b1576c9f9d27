"""Epilogue faults and what a one-spacing tolerance can see (CPU; faults planted on the
oracle side, never in the product).

"Deterministic LLM Inference Across GPU Kernels: Power-of-Two INT8 Quantization Scales ...":
§II "Pipeline and alibi" — with the int32 accumulator exact, two kernels can differ only in
the epilogue (applying s_a s_w and rounding to bfloat16); §III–IV — the epilogue faults it
injects (scale precision, double rounding, multiplication order, output truncation) move an
output by at most one bfloat16 spacing, and by exactly one whenever they move it, so a
one-spacing tolerance cannot see them; under power-of-two scales the intermediate-precision
and order faults change nothing, while a wrong rounding mode is seen only by an equality
check; an operand fault (an int8 activation shifted) moves outputs by many spacings.

The pages name the faults but print no code for them. The faulty epilogues below are this
file's readings of the names, applied to exact accumulators:
  F1 scale precision:      the combined scale s_a s_w rounded to fp32, applied in fp32
  F2 double rounding:      the exact value rounded to fp32 first, then to bfloat16
  F3 multiplication order: (fp32(acc) * s_a) * s_w in fp32
  F4 output truncation:    the exact value rounded toward zero instead of to nearest even
The correct epilogue is the oracle's one rounding of acc * s_a * s_w (pow2 scales: the
oracle's rne_bf16 of the exact double acc * 2^(ea+ew); other scales: exact rationals).
"""
from fractions import Fraction

import numpy as np
import pytest

from exact import bf16_bits_to_fraction, pow2, rne_bf16_exact


def _rne_bf16_f32(x: np.ndarray) -> np.ndarray:
    """bf16 bits of the round-to-nearest-even of finite fp32 values."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _rz_bf16_f32(x: np.ndarray) -> np.ndarray:
    """bf16 bits of fp32 values rounded toward zero (the low 16 bits dropped)."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _spacings(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """distance in bf16 spacings between two arrays of finite bf16 bit patterns"""
    def key(x):
        x = x.astype(np.int64)
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    return np.abs(key(a) - key(b))


def test_helpers_agree_with_the_oracle(oracle_mod):
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(3000) * np.exp2(rng.integers(-30, 30, 3000))).astype(np.float32)
    want = np.array([oracle_mod.rne_bf16(float(v)) for v in x], dtype=np.uint16)
    assert (_rne_bf16_f32(x) == want).all()
    rz = _rz_bf16_f32(x)
    got = np.array([bf16_bits_to_fraction(int(b)) for b in rz], dtype=object)
    assert all(abs(g) <= abs(Fraction(float(v))) for g, v in zip(got, x))  # toward zero
    assert (_spacings(rz, want) <= 1).all()


def _pow2_case(seed, n, acc_bits):
    rng = np.random.default_rng(seed)
    acc = rng.integers(-(2 ** acc_bits) + 1, 2 ** acc_bits, n).astype(np.int64)
    ea = rng.integers(-14, -5, n)
    ew = rng.integers(-14, -5, n)
    return acc, ea, ew


def _faults_pow2(acc, ea, ew):
    sa = np.exp2(ea).astype(np.float32)
    sw = np.exp2(ew).astype(np.float32)
    f32acc = acc.astype(np.float32)
    exact64 = acc.astype(np.float64) * np.exp2((ea + ew).astype(np.float64))  # exact in fp64
    return {
        "F1": _rne_bf16_f32(f32acc * (sa * sw)),
        "F2": _rne_bf16_f32(exact64.astype(np.float32)),
        "F3": _rne_bf16_f32((f32acc * sa) * sw),
    }


def test_pow2_scales_leave_precision_and_order_faults_invisible(oracle_mod):
    # |acc| < 2^24: fp32 holds acc, the scales and every product exactly, so F1-F3 give
    # the correct bits everywhere; truncation (F4) differs, by exactly one spacing
    acc, ea, ew = _pow2_case(2, 4000, 24)
    exact = np.array([oracle_mod.rne_bf16(float(a) * 2.0 ** int(e)) for a, e in zip(acc, ea + ew)],
                     dtype=np.uint16)
    for name, got in _faults_pow2(acc, ea, ew).items():
        assert (got == exact).all(), name
    f4 = _rz_bf16_f32(acc.astype(np.float32) * np.exp2(ea + ew).astype(np.float32))
    d = _spacings(f4, exact)
    assert d.max() == 1 and (d == 1).sum() > 1000  # observable, always one spacing


def test_pow2_scales_large_accumulators_double_rounding(oracle_mod):
    # |acc| >= 2^24: rounding acc to fp32 first can flip a bf16 tie. Hand-worked case:
    # acc = 2^24 + 2^16 + 1 lies just above the tie between 2^24 and 2^24 + 2^17 (RNE: up,
    # 0x4B81); fp32 drops the +1 (a tie at 2^24 + 2^16, to even), and the bf16 tie then
    # rounds to even, down to 2^24 (0x4B80): one spacing.
    acc = np.array([2 ** 24 + 2 ** 16 + 1], dtype=np.int64)
    zero = np.zeros(1, dtype=np.int64)
    assert oracle_mod.rne_bf16(float(acc[0])) == 0x4B81
    assert _faults_pow2(acc, zero, zero)["F2"][0] == 0x4B80
    # in general: never more than one spacing
    acc, ea, ew = _pow2_case(3, 4000, 31)
    exact = np.array([oracle_mod.rne_bf16(float(a) * 2.0 ** int(e)) for a, e in zip(acc, ea + ew)],
                     dtype=np.uint16)
    for name, got in _faults_pow2(acc, ea, ew).items():
        assert _spacings(got, exact).max() <= 1, name


def test_real_scales_every_epilogue_fault_within_one_spacing():
    # checkpoint-like (non power-of-two) scales: the exact reference is rational
    rng = np.random.default_rng(4)
    n = 1500
    acc = rng.integers(-(2 ** 26), 2 ** 26, n).astype(np.int64)
    sa = (rng.uniform(1.0, 2.0, n) * np.exp2(rng.integers(-14, -6, n))).astype(np.float32)
    sw = (rng.uniform(1.0, 2.0, n) * np.exp2(rng.integers(-14, -6, n))).astype(np.float32)
    vals = [Fraction(int(a)) * Fraction(float(x)) * Fraction(float(y)) for a, x, y in zip(acc, sa, sw)]
    exact = np.array([rne_bf16_exact(v) for v in vals], dtype=np.uint16)
    f32acc = acc.astype(np.float32)
    faults = {
        "F1": _rne_bf16_f32(f32acc * (sa * sw)),
        "F2": _rne_bf16_f32(np.array([float(v) for v in vals]).astype(np.float32)),
        "F3": _rne_bf16_f32((f32acc * sa) * sw),
    }
    # F4: toward zero from the exact value (one spacing below |RNE| when RNE rounded up)
    f4 = exact.copy()
    for i, v in enumerate(vals):
        r = bf16_bits_to_fraction(int(exact[i]))
        if abs(r) > abs(v):
            f4[i] = exact[i] - 1
    faults["F4"] = f4
    for name, got in faults.items():
        d = _spacings(got, exact)
        assert d.max() <= 1, name  # a one-spacing tolerance passes every one of them
    assert (faults["F4"] != exact).sum() > n // 4  # truncation is observable, equality sees it


def test_operand_fault_moves_outputs_by_many_spacings(oracle_mod):
    # one int8 activation shifted by one step changes the exact accumulator itself
    rng = np.random.default_rng(5)
    M, N, K = 8, 512, 256
    A = rng.integers(-127, 128, size=(M, K), dtype=np.int8)
    W = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    ea = np.full(M, -10, np.int32)
    ew = np.full(N, -10, np.int32)
    good = oracle_mod.w8a8(A, W, ea, ew)
    A2 = A.copy()
    A2[3, 17] = A2[3, 17] + 1 if A2[3, 17] < 127 else A2[3, 17] - 1
    bad = oracle_mod.w8a8(A2, W, ea, ew)
    d = _spacings(bad, good)
    assert (d[np.arange(M) != 3] == 0).all()  # other rows untouched
    assert d.max() >= 8  # far beyond a one-spacing tolerance (near-cancelling sums move most)


@pytest.mark.gpu
def test_gpu_epilogue_is_the_correct_one_not_a_faulty_one(oracle_mod):
    # the product's epilogue agrees with the one correct rounding and differs from the
    # truncating one exactly where the reference says truncation differs
    import torch
    from gpu_util import bf16_bits, cuda, dg, to_dev
    dev = cuda()
    lib = dg()
    rng = np.random.default_rng(6)
    for M, N, K in ((16, 256, 512), (300, 264, 1024)):
        A = rng.integers(-127, 128, size=(M, K), dtype=np.int8)
        W = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
        ea = rng.integers(-14, -6, size=M).astype(np.int32)
        ew = rng.integers(-14, -6, size=N).astype(np.int32)
        acc = oracle_mod.gemm_s8_i32(A, W).astype(np.int64)
        E = (ea[:, None] + ew[None, :]).astype(np.float64)
        f4 = _rz_bf16_f32((acc.astype(np.float64) * np.exp2(E)).astype(np.float32))  # |acc| < 2^24 here
        want = oracle_mod.w8a8(A, W, ea, ew)
        got = bf16_bits(lib.w8a8(to_dev(A, dev), to_dev(W, dev), to_dev(ea, dev), to_dev(ew, dev)))
        assert (got == want).all()
        assert ((got != f4) == (want != f4)).all() and (got != f4).any()
