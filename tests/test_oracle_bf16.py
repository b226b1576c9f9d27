"""Pins for the oracle's W8A8 epilogue rounding: rne_bf16(acc * 2^E).

Each check compares the oracle against something other than itself: the
hand-worked golden cases, and an exact-rational nearest-value search over the
table of every bf16 value (tests/exact.py).
"""
import os
import random
from fractions import Fraction

import numpy as np
import pytest

from exact import bf16_bits_to_fraction, pow2, rne_bf16_exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "w8a8_epilogue_cases.txt")


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        acc, e, bits = line.split()[:3]
        rows.append((int(acc), int(e), int(bits, 16)))
    return rows


@pytest.mark.parametrize("acc,e,bits", _golden_rows())
def test_golden_cases_exact_search(acc, e, bits):
    # the golden table itself agrees with the exact search (guards typos in the table)
    assert rne_bf16_exact(Fraction(acc) * pow2(e)) == bits


@pytest.mark.parametrize("acc,e,bits", _golden_rows())
def test_golden_cases_oracle(oracle_mod, acc, e, bits):
    v = float(np.ldexp(float(acc), e))
    assert oracle_mod.rne_bf16(v) == bits


def test_oracle_rne_matches_exact_search_random(oracle_mod):
    rng = random.Random(1234)
    for _ in range(4000):
        acc = rng.randint(-(2 ** 31) + 1, 2 ** 31 - 1)
        if rng.random() < 0.3:
            acc = rng.randint(-300, 300)
        e = rng.randint(-175, 135)
        exact = Fraction(acc) * pow2(e)
        v = float(np.ldexp(float(acc), e))  # exact in fp64 for this range
        assert Fraction(v) == exact
        assert oracle_mod.rne_bf16(v) == rne_bf16_exact(exact), (acc, e)


def test_oracle_rne_exact_ties_and_neighbours(oracle_mod):
    # midpoints between consecutive bf16 values (exact ties) and one fp64 ulp around them
    rng = random.Random(7)
    for _ in range(1500):
        b = rng.randint(0x0001, 0x7F7E)
        lo, hi = bf16_bits_to_fraction(b), bf16_bits_to_fraction(b + 1)
        mid = (lo + hi) / 2
        m = float(mid)
        assert Fraction(m) == mid
        for v in (m, np.nextafter(m, np.inf), np.nextafter(m, -np.inf)):
            for s in (1, -1):
                assert oracle_mod.rne_bf16(s * float(v)) == rne_bf16_exact(s * Fraction(float(v)))


def test_oracle_rne_every_bf16_value_roundtrips(oracle_mod):
    for b in range(0x0000, 0x7F80, 7):
        v = float(bf16_bits_to_fraction(b))
        assert oracle_mod.rne_bf16(v) == b
        assert oracle_mod.rne_bf16(-v) == (b | 0x8000)
