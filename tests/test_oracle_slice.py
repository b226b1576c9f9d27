"""Pins for the oracle's Ozaki slicing (frexp-shared exponent, 7-bit digits).

Source: "GPU Mechanism", §3 "Method", Interventions (a) ExactGEMM: operands cut
into 7-bit integer slices scaled by powers of two from frexp. Readings: one
exponent per row of A / per column of B (max|x| < 2^e), digits truncated toward
zero, signed, d_t in [-127, 127].
"""
from fractions import Fraction

import numpy as np
import pytest

from exact import pow2


def _recon(S, e, idx_fn, n):
    return sum(Fraction(int(S[t][idx_fn])) * pow2(int(e) - 7 * (t + 1)) for t in range(n))


def test_exponent_and_digit_ranges(oracle_mod):
    rng = np.random.default_rng(0)
    X = (rng.standard_normal((40, 70)) * np.exp2(rng.integers(-9, 9, size=(40, 70)))).astype(np.float32)
    S, e = oracle_mod.slice_f32(X, 0, 7)
    assert S.shape == (7, 40, 70)
    assert (np.abs(S.astype(np.int32)) <= 127).all()
    for i in range(40):
        a = np.abs(X[i]).max()
        assert a < 2.0 ** e[i] <= 2 * a


def test_reconstruction_exact_or_truncated(oracle_mod):
    rng = np.random.default_rng(1)
    X = (rng.standard_normal((30, 50)) * np.exp2(rng.integers(-40, 9, size=(30, 50)))).astype(np.float32)
    S, e = oracle_mod.slice_f32(X, 0, 7)
    for i in range(30):
        for j in range(50):
            x = Fraction(float(X[i, j]))
            r = sum(Fraction(int(S[t, i, j])) * pow2(int(e[i]) - 7 * (t + 1)) for t in range(7))
            # truncation toward zero: |r| <= |x|, same sign, error < one unit of the last digit
            assert abs(r) <= abs(x) and (r == 0 or (r > 0) == (x > 0))
            assert abs(x - r) < pow2(int(e[i]) - 49)
            # exact whenever x has no bits below 2^(e-49)
            if (x / pow2(int(e[i]) - 49)).denominator == 1:
                assert r == x
            # every nonzero digit carries the sign of x
            d = S[:, i, j].astype(np.int32)
            assert ((d == 0) | (np.sign(d) == np.sign(float(x)))).all()


def test_hand_worked_digits(oracle_mod):
    # row max 0.5 -> e = 0 (0.5 < 2^0); r = 0.5 = 64/128 -> d1 = 64
    # -0.75 * 2^10 in a row whose max is 0.99 * 2^10 -> e = 10, r = -0.75 -> d1 = -96
    # 1/3 (fp32) with max 1/3 -> e = -1, r = 2/3 -> digits of floor(2/3 * 2^49) in base 128
    X = np.array([[0.5, 0.25, 0.0]], np.float32)
    S, e = oracle_mod.slice_f32(X, 0, 7)
    assert e[0] == 0 and S[0, 0, 0] == 64 and S[0, 0, 1] == 32 and (S[1:, 0, :2] == 0).all()
    X = np.array([[-0.75 * 1024, 0.99 * 1024]], np.float32)
    S, e = oracle_mod.slice_f32(X, 0, 7)
    assert e[0] == 10 and S[0, 0, 0] == -96 and (S[1:, 0, 0] == 0).all()
    third = np.float32(1.0 / 3.0)
    S, e = oracle_mod.slice_f32(np.array([[third]], np.float32), 0, 7)
    assert e[0] == -1
    R = (Fraction(float(third)) * 2 * 2 ** 49).__floor__()
    want = [(R >> (7 * (6 - t))) & 127 for t in range(7)]
    assert [int(v) for v in S[:, 0, 0]] == want


def test_columns_equal_rows_of_transpose(oracle_mod):
    rng = np.random.default_rng(2)
    X = (rng.standard_normal((33, 17)) * np.exp2(rng.integers(-5, 5, size=(33, 17)))).astype(np.float32)
    Sc, ec = oracle_mod.slice_f32(X, 1, 7)
    Sr, er = oracle_mod.slice_f32(np.ascontiguousarray(X.T), 0, 7)
    assert Sc.shape == (7, 17, 33)
    assert (Sc == Sr).all() and (ec == er).all()


def test_zero_line_and_subnormals(oracle_mod):
    tiny = np.float32(2.0 ** -149)
    X = np.array([[0.0, 0.0], [tiny, -3 * tiny]], np.float32)
    S, e = oracle_mod.slice_f32(X, 0, 7)
    assert e[0] == 0 and (S[:, 0] == 0).all()
    # max 3 * 2^-149 -> e = -147; r = 1/4 and -3/4 -> d1 = 32, -96
    assert e[1] == -147 and S[0, 1, 0] == 32 and S[0, 1, 1] == -96


def test_nonfinite_reported(oracle_mod):
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.slice_f32(np.array([[1.0, np.nan]], np.float32), 0, 7)
