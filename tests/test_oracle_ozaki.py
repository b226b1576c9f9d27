"""Pins for the oracle's Ozaki-scheme fp32 GEMM.

Source: "GPU Mechanism", §3 "Method", Interventions (a) ExactGEMM and §2 "Exact
GEMM by error-free transformation". The page fixes: frexp-scaled 7-bit integer
slices, exact integer slice products, fixed-order fp64 recombination, one
rounding. The slice count (7) and the kept pairs (s + t <= 8) are those of the
workload definition; the combine order g = 8..2 and truncated digits are the
design's reading of steps the page leaves open (its bits are pinned below to
that written definition by exact-rational brute force, and to the page by the
error bound and by special cases whose exact answer is known).
"""
from fractions import Fraction

import numpy as np
import pytest

from exact import pow2, rne_f32_exact


def _frexp_e(a: Fraction) -> int:
    """smallest e with a < 2^e (a > 0)."""
    e = 0
    while a >= pow2(e):
        e += 1
    while a < pow2(e - 1):
        e -= 1
    return e


def _brute_ozaki(A, B, nslices=7, max_diag=8):
    """Exact-rational restatement: Fraction digits, Python-int diagonal sums,
    IEEE fp64 (Python float) combine in the order g = max_diag..2, then fp32 RNE."""
    M, K = A.shape
    N = B.shape[1]

    def digits(line):
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

    ea, DA = zip(*[digits(A[i]) for i in range(M)])
    fb, DB = zip(*[digits(B[:, j]) for j in range(N)])
    C = np.empty((M, N), np.float32)
    for i in range(M):
        for j in range(N):
            T = {}
            for g in range(2, max_diag + 1):
                T[g] = sum(DA[i][k][s - 1] * DB[j][k][g - s - 1]
                           for s in range(1, nslices + 1) if 1 <= g - s <= nslices
                           for k in range(K))
            acc = 0.0
            for g in range(max_diag, 1, -1):
                acc = acc + float(Fraction(T[g]) * pow2(-7 * g))  # exact conversion
            C[i, j] = rne_f32_exact(Fraction(acc) * pow2(ea[i] + fb[j]))
    return C


def test_bruteforce_tiny(oracle_mod):
    rng = np.random.default_rng(0)
    for (M, N, K) in [(2, 3, 5), (3, 2, 17)]:
        A = (rng.standard_normal((M, K)) * np.exp2(rng.integers(-8, 9, size=(M, K)))).astype(np.float32)
        B = (rng.standard_normal((K, N)) * np.exp2(rng.integers(-8, 9, size=(K, N)))).astype(np.float32)
        C = oracle_mod.ozaki_f32(A, B)
        assert (C.view(np.uint32) == _brute_ozaki(A, B).view(np.uint32)).all()


def test_combine_order_hand_worked(oracle_mod):
    """Cancellation case worked by hand: the fp64 combine order decides the bits.

    A row (e = 0):   x_0..x_128 = 0.5 (digit d1 = 64),   x_129 = 2^-7 (d1 = 1)
    B column (f = 0): y_0 = 0.5 (d1 = 64), y_1..y_128 = -2^-8 (d2 = -64), y_129 = 2^-49 (d7 = 1)
    Diagonals: T_2 = 64*64 = 4096, T_3 = 128 * 64 * (-64) = -524288, T_8 = 1, others 0.
    Terms: T_2 2^-14 = 0.25, T_3 2^-21 = -0.25, T_8 2^-56 = 2^-56.
    g = 8..2 (the defined order): 2^-56 - 0.25 is the midpoint between -0.25 and
    -(0.25 - 2^-55) -> ties to even -> -0.25; then + 0.25 = +0.  C = +0.0.
    g = 2..8 would give 0.25 - 0.25 + 2^-56 = 2^-56 (the exact product).
    """
    K = 130
    x = np.full((1, K), 0.5, np.float32)
    x[0, 129] = 2.0 ** -7
    y = np.full((K, 1), -(2.0 ** -8), np.float32)
    y[0, 0] = 0.5
    y[129, 0] = 2.0 ** -49
    C = oracle_mod.ozaki_f32(x, y)
    assert C.view(np.uint32)[0, 0] == 0x00000000
    # the exact product is 2^-56: the defined combine loses it, within the error bound
    exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(x[0], y[:, 0]))
    assert exact == pow2(-56)
    absab = np.abs(x.astype(np.float64)) @ np.abs(y.astype(np.float64))
    assert abs(float(exact)) <= 4 * 2.0 ** -24 * absab[0, 0]


def test_exact_when_all_bits_captured(oracle_mod):
    # small integers: every digit is captured, every partial sum is exact, so the
    # result is the correctly rounded exact product
    rng = np.random.default_rng(1)
    A = rng.integers(-1000, 1001, size=(20, 64)).astype(np.float32)
    B = rng.integers(-1000, 1001, size=(64, 24)).astype(np.float32)
    C = oracle_mod.ozaki_f32(A, B)
    exact = A.astype(np.int64) @ B.astype(np.int64)  # |.| < 2^53: float() is exact below
    assert (C == exact.astype(np.float64).astype(np.float32)).all()


def test_identity_reproduces_A(oracle_mod):
    rng = np.random.default_rng(2)
    n = 48
    # rows spanning at most 17 binades: every bit of A lies within 49 bits of the row max
    A = (rng.uniform(1, 2, size=(n, n)) * np.exp2(rng.integers(-8, 9, size=(n, n)))
         * rng.choice([-1, 1], size=(n, n))).astype(np.float32)
    C = oracle_mod.ozaki_f32(A, np.eye(n, dtype=np.float32))
    assert (C.view(np.uint32) == A.view(np.uint32)).all()


def test_error_bound_vs_fp64(oracle_mod, synth):
    # |C - C_fp64| <= 4 * 2^-24 * (|A||B|)_ij (the workload's stated bound)
    A = synth.normal_pow2_f32(4, 0, (64, 512), -8, 8)
    B = synth.normal_pow2_f32(4, 1, (512, 96), -8, 8)
    C = oracle_mod.ozaki_f32(A, B).astype(np.float64)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    absab = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    assert (np.abs(C - ref) <= 4 * 2.0 ** -24 * absab).all()


def test_diagonal_sums_match_integer_matmul(oracle_mod):
    rng = np.random.default_rng(3)
    A = (rng.standard_normal((9, 40)) * 100).astype(np.float32)
    B = (rng.standard_normal((40, 11)) * 0.01).astype(np.float32)
    DA, _ = oracle_mod.slice_f32(A, 0, 7)
    DB, _ = oracle_mod.slice_f32(B, 1, 7)
    T = oracle_mod.ozaki_diagonals(DA, DB, 8)
    for g in range(2, 9):
        want = np.zeros((9, 11), np.int64)
        for s in range(1, 8):
            t = g - s
            if 1 <= t <= 7:
                want += DA[s - 1].astype(np.int64) @ DB[t - 1].astype(np.int64).T
        assert (T[:, :, g] == want).all()


def test_rows_subset_and_zero(oracle_mod):
    rng = np.random.default_rng(4)
    A = (rng.standard_normal((12, 30))).astype(np.float32)
    A[3] = 0.0
    B = (rng.standard_normal((30, 7))).astype(np.float32)
    full = oracle_mod.ozaki_f32(A, B)
    assert (full[3] == 0).all()
    sub = oracle_mod.ozaki_f32(A, B, rows=[11, 3, 0])
    assert (sub.view(np.uint32) == full[[11, 3, 0]].view(np.uint32)).all()


def test_nonfinite_reported(oracle_mod):
    A = np.array([[1.0, np.inf]], np.float32)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.ozaki_f32(A, np.ones((2, 2), np.float32))


def _random_diagonals(rng, nd, M, N):
    """Diagonal sums drawn to exercise every rounding of the fp64 combine: full-range
    int32 values (the late sums then drop up to ~20 bits, and ties occur), small values,
    and values with many trailing zero bits (exact ties at the 53-bit boundary)."""
    full = rng.integers(-2 ** 31 + 1, 2 ** 31, size=(nd, M, N), dtype=np.int64)
    small = rng.integers(-3000, 3001, size=(nd, M, N), dtype=np.int64)
    shifted = rng.integers(-2 ** 10, 2 ** 10, size=(nd, M, N), dtype=np.int64) << rng.integers(0, 20, size=(nd, M, N))
    pick = rng.integers(0, 3, size=(nd, M, N))
    T = np.where(pick == 0, full, np.where(pick == 1, small, shifted))
    return np.clip(T, -2 ** 31 + 1, 2 ** 31 - 1).astype(np.int32)


def _brute_combine(Tcol, max_diag, e, f):
    """IEEE binary64 (Python float, round to nearest even) on exact conversions of
    T_g 2^(-7g) in the order g = max_diag..2, then the exact-rational fp32 rounding."""
    acc = 0.0
    for p in range(max_diag - 1):
        g = max_diag - p
        acc = acc + float(Fraction(int(Tcol[p])) * pow2(-7 * g))
    return rne_f32_exact(Fraction(acc) * pow2(int(e) + int(f)))


@pytest.mark.parametrize("max_diag", [2, 5, 8, 13, 18])
def test_combine_step_bruteforce(oracle_mod, max_diag):
    rng = np.random.default_rng(50 + max_diag)
    M, N = 6, 40
    T = _random_diagonals(rng, max_diag - 1, M, N)
    e = rng.integers(-40, 41, size=M).astype(np.int32)
    f = rng.integers(-40, 41, size=N).astype(np.int32)
    C = oracle_mod.ozaki_combine(T, e, f)
    for i in range(M):
        for j in range(N):
            want = _brute_combine(T[:, i, j], max_diag, e[i], f[j])
            assert C[i, j].view(np.uint32) == np.float32(want).view(np.uint32), (i, j)


def test_combine_step_hand_worked_order(oracle_mod):
    # T_8 = 1, T_3 = -524288, T_2 = 4096 (the cancellation case above): g = 8..2 gives +0
    T = np.zeros((7, 1, 1), np.int32)
    T[0, 0, 0] = 1        # plane 0: g = 8
    T[5, 0, 0] = -524288  # plane 5: g = 3
    T[6, 0, 0] = 4096     # plane 6: g = 2
    C = oracle_mod.ozaki_combine(T, np.zeros(1, np.int32), np.zeros(1, np.int32))
    assert C.view(np.uint32)[0, 0] == 0


def test_combine_step_matches_full_gemm(oracle_mod):
    rng = np.random.default_rng(6)
    A = (rng.standard_normal((5, 33)) * np.exp2(rng.integers(-8, 9, size=(5, 33)))).astype(np.float32)
    B = (rng.standard_normal((33, 9)) * np.exp2(rng.integers(-8, 9, size=(33, 9)))).astype(np.float32)
    DA, e = oracle_mod.slice_f32(A, 0, 7)
    DB, f = oracle_mod.slice_f32(B, 1, 7)
    T = oracle_mod.ozaki_diagonals(DA, DB, 8)                       # [M, N, g]
    planes = np.stack([T[:, :, g] for g in range(8, 1, -1)]).astype(np.int32)
    C = oracle_mod.ozaki_combine(planes, e, f)
    assert (C.view(np.uint32) == oracle_mod.ozaki_f32(A, B).view(np.uint32)).all()
