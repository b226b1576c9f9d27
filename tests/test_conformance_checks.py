"""The conformance checks (host logic, CPU): distances in bfloat16 spacings, operand digests,
the accumulator's exactness preconditions, the power-of-two identity and the one-spacing
tolerance ("Deterministic LLM Inference Across GPU Kernels ...", §III "Nine Faults", §IV)."""
import numpy as np

from deterministic_detgemm_w8a8_gb300 import conformance as c


def test_spacings_count_representable_values_between():
    # 1.0 and its neighbours; +0 and -0 coincide; crossing zero counts both sides
    assert c.bf16_spacings(np.array([0x3F80]), np.array([0x3F81]))[0] == 1
    assert c.bf16_spacings(np.array([0x3F80]), np.array([0x3F7F]))[0] == 1
    assert c.bf16_spacings(np.array([0x8000]), np.array([0x0000]))[0] == 0
    assert c.bf16_spacings(np.array([0x8001]), np.array([0x0001]))[0] == 2
    assert c.bf16_spacings(np.array([0x7F7F]), np.array([0x7F80]))[0] > 10 ** 9  # to infinity
    assert c.bf16_spacings(np.array([0x7F80]), np.array([0x7F80]))[0] == 0


def test_checks_fire_and_stay_silent_as_defined():
    A = np.ones((2, 8), np.int8)
    W = np.ones((3, 8), np.int8)
    d = c.operand_digest(A, W)
    assert c.check_shared_operands(d, d) == c.SILENT
    A2 = A.copy()
    A2[0, 0] = 2
    assert c.check_shared_operands(c.operand_digest(A2, W), d) == c.FIRE
    assert c.check_exactness_preconditions(A, W) == c.SILENT
    big = np.full((1, c.MAX_K + 1), 127, np.int8)
    assert c.check_exactness_preconditions(big, big) == c.FIRE
    ref = np.array([0x3F80, 0x4000], np.uint16)
    one_off = np.array([0x3F81, 0x4000], np.uint16)
    assert c.check_pow2_identity(ref, ref, True) == c.SILENT
    assert c.check_pow2_identity(one_off, ref, True) == c.FIRE
    assert c.check_pow2_identity(one_off, ref, False) == c.NA
    assert c.check_tolerance(one_off, ref) == c.SILENT  # one spacing is within the tolerance
    assert c.check_tolerance(np.array([0x3F82, 0x4000], np.uint16), ref) == c.FIRE
    assert c.check_token_level() == c.NA


def test_faulted_mask_severities():
    assert c.faulted_mask(37, 41, 0, 5).sum() == 1
    assert c.faulted_mask(37, 41, 2, 5).all()
    m = c.faulted_mask(300, 300, 1, 9)
    assert 0.007 < m.mean() < 0.013
    assert (m == c.faulted_mask(300, 300, 1, 9)).all() and (m != c.faulted_mask(300, 300, 1, 10)).any()
