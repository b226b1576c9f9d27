"""Pins for the oracle's fp64-target Ozaki GEMM (DGEMM emulation on exact integer slice
products).

Source: "GPU Mechanism", §3 "Method", Interventions (a) ExactGEMM: operands cut into 7-bit
integer slices under power-of-two scales from frexp, exact integer slice products,
fixed-order fp64 recombination, one rounding. The page applies it to fp32 GEMMs; here the
same steps are applied to fp64 operands with enough slices for fp64's 53-bit significand
(8 slices = 56 bits by default, diagonals s + t <= 9) and the result rounded to fp64 — the
design's reading of the scheme's fp64 form. Its bits are pinned to that written definition
by exact-rational brute force; its accuracy by an error bound against the exact product,
derived in the test below; special cases with known answers (small integers, A I = A).
"""
from fractions import Fraction

import numpy as np
import pytest

from exact import pow2, rne_f64_exact


def _frexp_e(a: Fraction) -> int:
    e = 0
    while a >= pow2(e):
        e += 1
    while a < pow2(e - 1):
        e -= 1
    return e


def _digits(line, nslices):
    a = max(abs(Fraction(float(x))) for x in line)
    e = _frexp_e(a) if a > 0 else 0
    out = []
    for x in line:
        r = Fraction(float(x)) / pow2(e)
        ds = []
        for _ in range(nslices):
            v = r * 128
            d = int(v)  # trunc toward zero for Fraction
            ds.append(d)
            r = v - d
        out.append(ds)
    return e, out


def _brute(A, B, nslices=8, max_diag=9):
    M, K = A.shape
    N = B.shape[1]
    ea, DA = zip(*[_digits(A[i], nslices) for i in range(M)])
    fb, DB = zip(*[_digits(B[:, j], nslices) for j in range(N)])
    C = np.empty((M, N), np.float64)
    for i in range(M):
        for j in range(N):
            acc = 0.0
            for g in range(max_diag, 1, -1):
                T = sum(DA[i][k][s - 1] * DB[j][k][g - s - 1]
                        for s in range(1, nslices + 1) if 1 <= g - s <= nslices for k in range(K))
                acc = acc + float(Fraction(T) * pow2(-7 * g))  # exact conversion, IEEE fp64 add
            C[i, j] = rne_f64_exact(Fraction(acc) * pow2(ea[i] + fb[j]))
    return C, ea, fb


def test_bruteforce_tiny(oracle_mod):
    rng = np.random.default_rng(10)
    for (M, N, K, ns, md) in [(2, 3, 5, 8, 9), (3, 2, 11, 8, 9), (2, 2, 6, 5, 6), (2, 3, 4, 10, 11)]:
        A = rng.standard_normal((M, K)) * np.exp2(rng.integers(-20, 21, size=(M, K)))
        B = rng.standard_normal((K, N)) * np.exp2(rng.integers(-20, 21, size=(K, N)))
        C = oracle_mod.ozaki_f64(A, B, ns, md)
        want, _, _ = _brute(A, B, ns, md)
        assert (C.view(np.uint64) == want.view(np.uint64)).all()


def test_exact_for_small_integers(oracle_mod):
    rng = np.random.default_rng(11)
    A = rng.integers(-10 ** 6, 10 ** 6, size=(9, 40)).astype(np.float64)
    B = rng.integers(-10 ** 6, 10 ** 6, size=(40, 7)).astype(np.float64)
    C = oracle_mod.ozaki_f64(A, B)
    exact = A.astype(np.int64) @ B.astype(np.int64)  # |.| < 2^53
    assert (C == exact.astype(np.float64)).all()


def test_identity_reproduces_A(oracle_mod):
    # 8 slices hold 56 bits: every entry within 3 binades of its row max is captured
    # whole, and the fixed-order sums of its digits are exact
    rng = np.random.default_rng(12)
    n = 40
    A = rng.uniform(1, 8, size=(n, n)) * np.exp2(rng.integers(-300, 300, size=(n, 1))) * rng.choice([-1, 1], (n, n))
    C = oracle_mod.ozaki_f64(A, np.eye(n))
    assert (C.view(np.uint64) == A.view(np.uint64)).all()


def test_error_bound_vs_exact_product(oracle_mod):
    """Error bound of the defined algorithm (8 slices, s + t <= 9). Per product term, with
    a = 2^e (a' + alpha), |alpha| < 2^-56 (digits past the eighth) and the same for b,
    and the dropped pairs s + t >= 10 summing to < 7 * 127^2 * 2^-70 * 1.01 < 2^-53.1:
    |term error| < 2^(e+f) (2^-55 + 2^-53.1) < 2^(e+f) 2^-52.7. The eight fp64 additions
    of partial sums bounded by K 2^(e+f) add at most 8 K 2^(e+f) 2^-53, and the last
    rounding 2^-53 |C|. Bound: |C - exact| <= 2^-53 |C| + 10 K 2^(e_i + f_j - 53)."""
    rng = np.random.default_rng(13)
    M, K, N = 6, 48, 5
    A = rng.standard_normal((M, K)) * np.exp2(rng.integers(-12, 13, size=(M, K)))
    B = rng.standard_normal((K, N)) * np.exp2(rng.integers(-12, 13, size=(K, N)))
    C = oracle_mod.ozaki_f64(A, B)
    _, e = oracle_mod.slice_f64(A, 0, 8)
    _, f = oracle_mod.slice_f64(B, 1, 8)
    for i in range(M):
        for j in range(N):
            exact = sum(Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K))
            err = abs(Fraction(float(C[i, j])) - exact)
            bound = pow2(-53) * abs(Fraction(float(C[i, j]))) + 10 * K * pow2(int(e[i]) + int(f[j]) - 53)
            assert err <= bound, (i, j)
    # and the bound is not loose: dropping the two smallest diagonals (max_diag 7) breaks it
    C8 = oracle_mod.ozaki_f64(A, B, 8, 7)
    worst = max(abs(Fraction(float(C8[i, j])) - sum(Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
                                                     for k in range(K)))
                / (10 * K * pow2(int(e[i]) + int(f[j]) - 53)) for i in range(M) for j in range(N))
    assert worst > 1


def test_slice_f64_reconstructs(oracle_mod):
    rng = np.random.default_rng(14)
    X = rng.standard_normal((7, 33)) * np.exp2(rng.integers(-40, 40, size=(7, 33)))
    X[2] = 0.0
    X[3, :5] = 5e-324 * np.arange(5)  # subnormals in a row with normal values
    for nslices in (8, 11):
        S, e = oracle_mod.slice_f64(X, 0, nslices)
        assert S.min() >= -127 and S.max() <= 127
        assert e[2] == 0 and (S[:, 2] == 0).all()
        for i in range(7):
            for k in range(33):
                x = Fraction(float(X[i, k]))
                approx = pow2(int(e[i])) * sum(Fraction(int(S[t, i, k])) * pow2(-7 * (t + 1)) for t in range(nslices))
                assert abs(x - approx) < pow2(int(e[i]) - 7 * nslices)
                assert approx == 0 or (approx > 0) == (x > 0)


@pytest.mark.parametrize("max_diag", [2, 9, 13, 18])
def test_combine_f64_bruteforce(oracle_mod, max_diag):
    rng = np.random.default_rng(70 + max_diag)
    M, N = 4, 30
    T = rng.integers(-2 ** 31 + 1, 2 ** 31, size=(max_diag - 1, M, N)).astype(np.int32)
    e = rng.integers(-1100, 1000, size=M).astype(np.int32)
    f = rng.integers(-1000, 900, size=N).astype(np.int32)
    e[0], f[0], f[1] = -1060, -20, 70  # fp64 subnormal results, and large ones
    C = oracle_mod.ozaki_combine_f64(T, e, f)
    for i in range(M):
        for j in range(N):
            acc = 0.0
            for p in range(max_diag - 1):
                acc = acc + float(Fraction(int(T[p, i, j])) * pow2(-7 * (max_diag - p)))
            want = rne_f64_exact(Fraction(acc) * pow2(int(e[i]) + int(f[j])))
            assert C[i, j] == want or (np.isnan(C[i, j]) and np.isnan(want)), (i, j)
            assert np.signbit(C[i, j]) == np.signbit(want)
