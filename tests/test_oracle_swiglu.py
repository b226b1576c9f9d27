"""Pins of the gated-linear-unit epilogue oracle, out = rne_bf16(SiLU(g) * u) of the exact
scaled accumulators (the W8A8 epilogue of "Deterministic LLM Inference Across GPU Kernels
...", §II "Pipeline and alibi": one rounding, here of SiLU(gate) * up).

The oracle evaluates in binary128; the pins come from elsewhere: an independent mpmath
evaluation at 300-700 bits, converted exactly to a Fraction and rounded by the table-search
rne_bf16_exact; hand-worked values (tests/golden/swiglu_cases.txt), including a large gate
whose exact product g * u sits on a bf16 midpoint; sign symmetry in u; monotonicity in u; and
the composition with exact int64 dot products on small matrices."""
import os
from fractions import Fraction

import mpmath
import numpy as np
import pytest

from exact import rne_bf16_exact

HERE = os.path.dirname(os.path.abspath(__file__))


def _mp_ref(gacc, uacc, Eg, Eu):
    if gacc == 0 or uacc == 0:
        return 0
    g = Fraction(gacc) * Fraction(2) ** Eg
    mpmath.mp.prec = max(300, 64 + 2 * int(abs(g)))
    y = mpmath.mpf(gacc) * mpmath.mpf(2) ** Eg * mpmath.mpf(uacc) * mpmath.mpf(2) ** Eu / (1 + mpmath.exp(-mpmath.mpf(gacc) * mpmath.mpf(2) ** Eg))
    man, exp = abs(mpmath.mpf(y)).man_exp  # magnitude: man_exp does not carry the sign
    mag = Fraction(int(man)) * Fraction(2) ** int(exp)
    return rne_bf16_exact(-mag if y < 0 else mag)


def test_hand_worked(oracle_mod):
    n = 0
    for line in open(os.path.join(HERE, "golden", "swiglu_cases.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        g, u, eg, eu, want = line.split()
        assert oracle_mod.silu_mul_bf16(int(g), int(u), int(eg), int(eu)) == int(want, 16), line
        assert _mp_ref(int(g), int(u), int(eg), int(eu)) == int(want, 16), line
        n += 1
    assert n == 6


def test_against_high_precision_evaluation(oracle_mod):
    rng = np.random.default_rng(1)
    cases = []
    for _ in range(1500):  # typical FFN magnitudes
        cases.append((int(rng.integers(-2 ** 20, 2 ** 20)), int(rng.integers(-2 ** 20, 2 ** 20)),
                      int(rng.integers(-24, -14)), int(rng.integers(-24, -14))))
    for _ in range(1500):  # full accumulator range, wide exponents (|g| up to ~400)
        ga = int(rng.integers(-2 ** 31 + 1, 2 ** 31))
        eg = int(rng.integers(-60, -22))
        cases.append((ga, int(rng.integers(-2 ** 31 + 1, 2 ** 31)), eg, int(rng.integers(-60, 40))))
    for _ in range(300):  # large gates: the product decides, save on midpoints
        cases.append((int(rng.integers(64, 400)), int(rng.integers(-2 ** 12, 2 ** 12)), 0, int(rng.integers(-12, 0))))
    for _ in range(300):  # deep negative gates: tiny and subnormal outputs
        cases.append((int(rng.integers(-400, -40)), int(rng.integers(1, 2 ** 31)), 0, int(rng.integers(30, 41))))
    bad = [(c, oracle_mod.silu_mul_bf16(*c), _mp_ref(*c)) for c in cases
           if oracle_mod.silu_mul_bf16(*c) != _mp_ref(*c)]
    assert not bad, bad[:5]


def test_midpoint_products_with_large_gates(oracle_mod):
    # g * u exactly on a bf16 midpoint: the exact y = SiLU(g) u is just inside it
    for g in (70, 96, 128, 300):
        for u_num, Eu in ((259, 0), (1029, -3), (-515, 1)):
            want = _mp_ref(g, u_num, 0, Eu)
            assert oracle_mod.silu_mul_bf16(g, u_num, 0, Eu) == want, (g, u_num, Eu)


def test_sign_symmetry_and_monotonicity(oracle_mod):
    rng = np.random.default_rng(2)
    for _ in range(300):
        g, u = int(rng.integers(-2 ** 24, 2 ** 24)), int(rng.integers(1, 2 ** 24))
        eg, eu = int(rng.integers(-30, -16)), int(rng.integers(-30, -16))
        a = oracle_mod.silu_mul_bf16(g, u, eg, eu)
        b = oracle_mod.silu_mul_bf16(g, -u, eg, eu)
        assert b == a ^ 0x8000 or (a & 0x7FFF) == 0 == (b & 0x7FFF)
    # for g > 0 the output grows with u (as bf16 magnitudes of positive values)
    vals = [oracle_mod.silu_mul_bf16(12345, u, -10, -12) for u in range(1, 4000, 7)]
    assert all(x <= y for x, y in zip(vals, vals[1:]))


def test_gemm_composition(oracle_mod):
    rng = np.random.default_rng(3)
    A = rng.integers(-127, 128, (5, 40), dtype=np.int8)
    Wg = rng.integers(-127, 128, (6, 40), dtype=np.int8)
    Wu = rng.integers(-127, 128, (6, 40), dtype=np.int8)
    ea = rng.integers(-12, -6, 5).astype(np.int32)
    ewg = rng.integers(-12, -6, 6).astype(np.int32)
    ewu = rng.integers(-12, -6, 6).astype(np.int32)
    C = oracle_mod.w8a8_swiglu(A, Wg, Wu, ea, ewg, ewu)
    for i in range(5):
        for j in range(6):
            g = int(np.dot(A[i].astype(np.int64), Wg[j].astype(np.int64)))
            u = int(np.dot(A[i].astype(np.int64), Wu[j].astype(np.int64)))
            assert C[i, j] == _mp_ref(g, u, int(ea[i] + ewg[j]), int(ea[i] + ewu[j]))
    rows = [4, 1]
    assert (oracle_mod.w8a8_swiglu(A, Wg, Wu, ea, ewg, ewu, rows=rows) == C[rows]).all()


def test_hard_inputs_near_midpoints(oracle_mod):
    # inputs within 2^-20 / 2^-52 of a rounding boundary (tests/golden/make_swiglu_hard_inputs.py)
    n = 0
    for line in open(os.path.join(HERE, "golden", "swiglu_hard_inputs.txt")):
        if line.startswith("#"):
            continue
        g, u, eg, eu, _ = line.split()
        assert oracle_mod.silu_mul_bf16(int(g), int(u), int(eg), int(eu)) == _mp_ref(int(g), int(u), int(eg), int(eu))
        n += 1
    assert n >= 50
