"""Pins for the oracle's power-of-two quantizer.

Source: "Deterministic LLM Inference Across GPU Kernels: Power-of-Two INT8
Quantization Scales ...", §V (weights requantized under a power-of-two scale)
and §V.C (nearest arm vs ceiling arm; the ceiling arm never shrinks a scale,
the nearest arm may clip outliers). Readings: absmax-symmetric scale s = a/127,
nearest in the log domain, q = clamp(rne(x / 2^e), -127, 127).
"""
from fractions import Fraction

import numpy as np
import pytest

from exact import pow2


def _bf16_bits(x):
    """fp32 values that are exactly bf16 -> their bf16 bit patterns."""
    b = np.asarray(x, np.float32).view(np.uint32)
    assert ((b & 0xFFFF) == 0).all()
    return (b >> 16).astype(np.uint16)


def _rne_int(fr: Fraction) -> int:
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


@pytest.mark.parametrize("mode", [0, 1])
def test_exponent_is_optimal(oracle_mod, mode):
    rng = np.random.default_rng(mode)
    X = (rng.standard_normal((300, 64)) * np.exp2(rng.integers(-30, 30, size=(300, 1)))).astype(np.float32)
    X[5] = 0.0
    Q, e = oracle_mod.quantize_pow2(X, mode)
    for i in range(300):
        a = max(abs(Fraction(float(x))) for x in X[i])
        if a == 0:
            assert e[i] == 0 and (Q[i] == 0).all()
            continue
        s = a / 127
        E = int(e[i])
        if mode == 1:  # ceiling: 2^E >= s > 2^(E-1)
            assert pow2(E) >= s > pow2(E - 1)
        else:  # nearest in log domain: 2^(2E-1) <= s^2 < 2^(2E+1)
            assert pow2(2 * E - 1) <= s * s < pow2(2 * E + 1)


@pytest.mark.parametrize("mode", [0, 1])
def test_values_bruteforce(oracle_mod, mode):
    rng = np.random.default_rng(10 + mode)
    X = (rng.standard_normal((50, 200)) * 3.0).astype(np.float32)
    X[:, 7] = X[:, 3] * 0.5  # force some ties after scaling for a few rows
    Q, e = oracle_mod.quantize_pow2(X, mode)
    for i in range(50):
        for j in range(200):
            q = _rne_int(Fraction(float(X[i, j])) / pow2(int(e[i])))
            assert int(Q[i, j]) == max(-127, min(127, q))


def test_ceiling_never_clips_and_error_bound(oracle_mod):
    rng = np.random.default_rng(3)
    X = (rng.standard_normal((64, 512)) * 7.0).astype(np.float32)
    Q, e = oracle_mod.quantize_pow2(X, 1)
    deq = Q.astype(np.float64) * np.exp2(e.astype(np.float64))[:, None]
    assert (np.abs(deq - X) <= np.exp2(e.astype(np.float64) - 1)[:, None]).all()


def test_already_quantized_rows_roundtrip(oracle_mod):
    # x = q0 * 2^e0 with max|q0| large enough that e0 is the chosen exponent
    rng = np.random.default_rng(4)
    for mode, qmax in ((0, 90), (1, 64)):
        for _ in range(40):
            e0 = int(rng.integers(-20, 20))
            q0 = rng.integers(-127, 128, size=33)
            q0[0] = int(rng.integers(qmax, 128)) * (1 if rng.random() < 0.5 else -1)
            X = (q0.astype(np.float64) * 2.0 ** e0).astype(np.float32)[None, :]
            Q, e = oracle_mod.quantize_pow2(X, mode)
            assert e[0] == e0 and (Q[0] == q0).all()


def test_nearest_arm_clips_outliers(oracle_mod):
    # a = 100 -> s = 100/127; log2 s = -0.345 -> nearest e = 0, so 100 stays, no clip;
    # a = 120 -> s = 0.945 -> e = 0 too; a = 127*1.5 -> s = 1.5, log2 = 0.585 -> e = 1
    X = np.array([[100.0, 1.0]], np.float32)
    Q, e = oracle_mod.quantize_pow2(X, 0)
    assert e[0] == 0 and Q[0, 0] == 100
    # a = 127 * 2^0.4 = 167.6: log2 s = 0.4 -> nearest e = 0 -> q clipped to 127;
    # the ceiling arm picks e = 1 and q = rne(83.8) = 84
    X = np.array([[167.625, -3.0]], np.float32)
    Q, e = oracle_mod.quantize_pow2(X, 0)
    assert e[0] == 0 and Q[0, 0] == 127 and Q[0, 1] == -3
    Q, e = oracle_mod.quantize_pow2(X, 1)
    assert e[0] == 1 and Q[0, 0] == 84 and Q[0, 1] == -2  # -1.5 -> -2 (ties to even)


def test_bf16_input_every_value_one_scale(oracle_mod):
    # a row holding its max 127 * 2^3 followed by many bf16 values below it
    bits = np.arange(0x0000, 0x4480, 3, dtype=np.uint32)  # every third bf16 pattern below 1024
    vals = (bits << 16).view(np.float32)
    vals = vals[np.abs(vals) <= 1016.0]
    row = np.concatenate([[np.float32(1016.0)], vals, -vals]).astype(np.float32)
    Q, e = oracle_mod.quantize_pow2(_bf16_bits(row)[None, :], 1)
    assert e[0] == 3
    for x, q in zip(row, Q[0]):
        assert int(q) == max(-127, min(127, _rne_int(Fraction(float(x)) / 8)))
    Qf, ef = oracle_mod.quantize_pow2(row[None, :], 1)  # fp32 path agrees
    assert (Qf == Q).all() and (ef == e).all()


def test_monotone_in_x(oracle_mod):
    rng = np.random.default_rng(9)
    x = np.sort(rng.standard_normal(4000).astype(np.float32) * 5)
    Q, _ = oracle_mod.quantize_pow2(x[None, :], 0)
    assert (np.diff(Q[0].astype(np.int32)) >= 0).all()


def test_nonfinite_reported(oracle_mod):
    X = np.array([[1.0, np.inf]], np.float32)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.quantize_pow2(X, 0)
