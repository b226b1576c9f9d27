"""Pins of the oracle's biased W8A8 epilogue (CPU).

Definition: the epilogue is the one rounding of the exactly scaled int32 accumulator
("Deterministic LLM Inference Across GPU Kernels: Power-of-Two INT8 Quantization Scales
...", §II "Pipeline and alibi"); a bias b_j (bfloat16) joins that exact value before the
rounding:  C_ij = rne_bf16(acc_ij * 2^(ea_i + ew_j) + b_j).
Readings (not on the page): b = +-0 leaves the unbiased result (x + 0 = x, the sign of an
underflowing x included); a non-finite b passes through; an exact zero sum gives +0.

The oracle rounds through an fp64 two-sum with a halfway-point correction. Here it is
checked against the exact rational sum rounded by a search over every bf16 value
(tests/exact.py), which shares no arithmetic with it, on hand-worked golden rows, on
random and near-halfway inputs, and on whole matrices.
"""
import os
from fractions import Fraction

import numpy as np

from exact import bf16_bits_to_fraction, pow2, rne_bf16_exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "w8a8_bias_cases.txt")


def exact_bias(acc: int, E: int, b: int) -> int:
    """rne_bf16(acc * 2^E + b) from exact rationals, with the readings above."""
    if (b & 0x7F80) == 0x7F80:
        return b
    x = Fraction(acc) * pow2(E)
    if (b & 0x7FFF) == 0:
        return rne_bf16_exact(x)
    v = x + bf16_bits_to_fraction(b)
    if v == 0:
        return 0
    return rne_bf16_exact(v)


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = line.split()
        rows.append((int(f[0]), int(f[1]), int(f[2], 16), int(f[3], 16), " ".join(f[4:])))
    return rows


def test_golden_rows_are_the_exact_definition():
    rows = _golden_rows()
    assert len(rows) >= 30
    for acc, E, b, want, why in rows:
        assert exact_bias(acc, E, b) == want, (acc, E, hex(b), why)


def test_oracle_matches_golden_rows(oracle_mod):
    for acc, E, b, want, why in _golden_rows():
        assert oracle_mod.bias_round(acc, E, b) == want, (acc, E, hex(b), why)


def _finite_bf16(rng, lo_field, hi_field, n):
    field = rng.integers(lo_field, hi_field + 1, n)
    frac = rng.integers(0, 128, n)
    sign = rng.integers(0, 2, n) << 15
    return (sign | (field << 7) | frac).astype(np.int64)


def test_random_against_exact_rationals(oracle_mod):
    rng = np.random.default_rng(11)
    n = 4000
    accs = rng.integers(-(2 ** 31), 2 ** 31, n)
    small = rng.integers(-300, 301, n)
    accs = np.where(rng.random(n) < 0.3, small, accs)
    Es = rng.integers(-170, 100, n)
    bits = _finite_bf16(rng, 0, 254, n)
    for acc, E, b in zip(accs.tolist(), Es.tolist(), bits.tolist()):
        assert oracle_mod.bias_round(acc, E, b) == exact_bias(acc, E, b), (acc, E, hex(b))


def test_near_halfway_sums(oracle_mod):
    # x's last unit placed a few bits around b's rounding position: many exact ties and
    # values one unit off a tie, on both sides of binade boundaries
    rng = np.random.default_rng(12)
    ties = 0
    for _ in range(6000):
        b = int(_finite_bf16(rng, 1, 250, 1)[0])
        field = (b >> 7) & 0xFF
        eb = field - 134  # b = mb * 2^eb with an 8-bit mb
        acc = int(rng.integers(-(2 ** 12), 2 ** 12))
        E = eb - 1 - int(rng.integers(0, 4))  # E = eb - 1 and an odd acc: a halfway sum
        want = exact_bias(acc, E, b)
        got = oracle_mod.bias_round(acc, E, b)
        assert got == want, (acc, E, hex(b))
        v = Fraction(acc) * pow2(E) + bf16_bits_to_fraction(b)
        lo = rne_bf16_exact(v)
        if v != 0 and bf16_bits_to_fraction(lo) != v:
            ties += _halfway(abs(v))
    assert ties > 500


def _halfway(a: Fraction) -> bool:
    """a > 0 lies exactly halfway between two neighbouring bf16 numbers"""
    p = a.numerator.bit_length() - a.denominator.bit_length()
    if pow2(p) > a:
        p -= 1  # now 2^p <= a < 2^(p+1)
    q = a / pow2(max(p - 7, -133))  # a in units of the bf16 spacing at a
    return q.denominator == 2


def test_halfway_helper():
    assert _halfway(Fraction(257)) and _halfway(Fraction(1) + pow2(-8)) and _halfway(pow2(-134))
    assert not _halfway(Fraction(256)) and not _halfway(Fraction(1) + pow2(-9))
    assert _halfway(Fraction(1) - pow2(-9)) and not _halfway(Fraction(1) - pow2(-10))


def test_zero_bias_is_the_unbiased_epilogue(oracle_mod):
    rng = np.random.default_rng(13)
    M, N, K = 9, 40, 300
    A = rng.integers(-128, 128, (M, K), dtype=np.int8)
    W = rng.integers(-128, 128, (N, K), dtype=np.int8)
    ea = rng.integers(-150, 20, M).astype(np.int32)
    ew = rng.integers(-40, 10, N).astype(np.int32)
    for zero in (0x0000, 0x8000):
        bias = np.full(N, zero, dtype=np.uint16)
        assert (oracle_mod.w8a8_bias(A, W, ea, ew, bias) == oracle_mod.w8a8(A, W, ea, ew)).all()


def test_matrix_against_exact_rationals(oracle_mod):
    # the matrix entry point: accumulators from numpy's int64 matmul, each output rounded
    # from the exact rational sum
    rng = np.random.default_rng(14)
    M, N, K = 7, 33, 260
    A = rng.integers(-127, 128, (M, K), dtype=np.int8)
    W = rng.integers(-127, 128, (N, K), dtype=np.int8)
    ea = rng.integers(-14, -6, M).astype(np.int32)
    ew = rng.integers(-14, -6, N).astype(np.int32)
    acc = A.astype(np.int64) @ W.astype(np.int64).T
    # biases near the outputs' magnitude (a few columns special)
    typical = acc[0].astype(np.float64) * np.exp2(ea[0] + ew)
    bias = np.array([int(rne_bf16_exact(Fraction(float(-t) * 0.75))) for t in typical], dtype=np.uint16)
    bias[0], bias[1], bias[2] = 0x8000, 0x7F80, 0x0001
    got = oracle_mod.w8a8_bias(A, W, ea, ew, bias)
    for i in range(M):
        for j in range(N):
            want = exact_bias(int(acc[i, j]), int(ea[i]) + int(ew[j]), int(bias[j]))
            assert got[i, j] == want, (i, j)


def test_bias_commutes_with_row_selection(oracle_mod):
    # a row's result does not depend on the rows computed with it
    rng = np.random.default_rng(15)
    M, N, K = 12, 20, 64
    A = rng.integers(-127, 128, (M, K), dtype=np.int8)
    W = rng.integers(-127, 128, (N, K), dtype=np.int8)
    ea = rng.integers(-14, -6, M).astype(np.int32)
    ew = rng.integers(-14, -6, N).astype(np.int32)
    bias = _finite_bf16(rng, 110, 130, N).astype(np.uint16)
    full = oracle_mod.w8a8_bias(A, W, ea, ew, bias)
    rows = [11, 0, 5]
    assert (oracle_mod.w8a8_bias(A, W, ea, ew, bias, rows=rows) == full[rows]).all()
