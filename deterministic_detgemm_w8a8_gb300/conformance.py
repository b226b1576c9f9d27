"""Conformance checks for W8A8 deployments and the epilogue fault injector behind them.

"Deterministic LLM Inference Across GPU Kernels: Power-of-Two INT8 Quantization Scales
and the Limits of Tolerance-Based Conformance", §III "Nine Faults" and §IV "How much can a
tolerance see?": a measurement instrument injects faults into a W8A8 kernel and runs
conformance checks of five kinds on its output — shared operands, the accumulator's
exactness preconditions, power-of-two identity, a real-scale tolerance of one bfloat16
spacing, and token-level risk. The pages report that the checks catch operand and
precondition faults, while epilogue faults move an output by at most one spacing and stay
invisible to the tolerance; under power-of-two scales an equality check sees a wrong rounding
mode. The checks below are this module's readings of those names (the pages print neither
their code nor their thresholds beyond the one-spacing tolerance); the faults themselves run
on the GPU in detgemm_epilogue_inject (include/detgemm_conformance.h).

Every check returns "fire", "silent" or "n/a" (not applicable to the arms given).
"""
from __future__ import annotations

import hashlib

import numpy as np

FIRE, SILENT, NA = "fire", "silent", "n/a"
MAX_K = 131071  # K * 128^2 < 2^31: any int8 operands accumulate exactly in int32


def bf16_spacings(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bfloat16 spacings between two arrays of bf16 bit patterns (finite
    values; +0 and -0 are the same point). Infinite or NaN patterns count as an unbounded
    distance unless both sides hold the same pattern."""
    a = np.asarray(a, dtype=np.uint16).astype(np.int64)
    b = np.asarray(b, dtype=np.uint16).astype(np.int64)
    key = lambda x: np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    d = np.abs(key(a) - key(b))
    nonfinite = ((a & 0x7F80) == 0x7F80) | ((b & 0x7F80) == 0x7F80)
    return np.where(nonfinite, np.where(a == b, 0, np.iinfo(np.int64).max), d)


def operand_digest(*arrays) -> str:
    """SHA-256 over the bytes of the given operand arrays (shape and dtype included)."""
    h = hashlib.sha256()
    for x in arrays:
        x = np.ascontiguousarray(x)
        h.update(str((x.shape, x.dtype.str)).encode())
        h.update(x.tobytes())
    return h.hexdigest()


def check_shared_operands(digest_arm: str, digest_reference: str) -> str:
    """Both arms multiplied the same int8 operands under the same scales."""
    return SILENT if digest_arm == digest_reference else FIRE


def check_exactness_preconditions(A: np.ndarray, W: np.ndarray) -> str:
    """The int32 accumulator is exact: K within the library's bound and
    K * max|A| * max|W| < 2^31 for the operands actually given."""
    K = A.shape[1]
    if K != W.shape[1]:
        return FIRE
    amax = int(np.abs(A.astype(np.int64)).max(initial=0))
    wmax = int(np.abs(W.astype(np.int64)).max(initial=0))
    return SILENT if K <= MAX_K and K * amax * wmax < 2 ** 31 else FIRE


def check_pow2_identity(out: np.ndarray, reference: np.ndarray, scales_pow2: bool) -> str:
    """Under power-of-two scales the epilogue has one correct result: bit equality."""
    if not scales_pow2:
        return NA
    return SILENT if np.array_equal(np.asarray(out, np.uint16), np.asarray(reference, np.uint16)) else FIRE


def check_tolerance(out: np.ndarray, reference: np.ndarray, spacings: int = 1) -> str:
    """Every output within `spacings` bfloat16 spacings of the reference (one spacing is
    the smallest nonzero allowance)."""
    return SILENT if int(bf16_spacings(out, reference).max(initial=0)) <= spacings else FIRE


def check_token_level(logits=None) -> str:
    """Token-level risk needs logit margins, which a layer-level run does not produce."""
    return NA if logits is None else FIRE


def run_checks(out, reference, *, digest_arm: str, digest_reference: str, A, W, scales_pow2: bool) -> dict:
    """All five checks on one arm's output against the reference arm's output."""
    return {
        "shared_operands": check_shared_operands(digest_arm, digest_reference),
        "exactness_preconditions": check_exactness_preconditions(A, W),
        "pow2_identity": check_pow2_identity(out, reference, scales_pow2),
        "tolerance_1_spacing": check_tolerance(out, reference, 1),
        "token_level": check_token_level(None),
    }


def mix32(x: int) -> int:
    """The injector's 32-bit mixer (xorshift-multiply rounds), for locating faulted outputs."""
    x &= 0xFFFFFFFF
    x ^= x >> 16
    x = (x * 0x7FEB352D) & 0xFFFFFFFF
    x ^= x >> 15
    x = (x * 0x846CA68B) & 0xFFFFFFFF
    x ^= x >> 16
    return x


def faulted_mask(M: int, N: int, severity: int, seed: int) -> np.ndarray:
    """Which outputs detgemm_epilogue_inject faults at a severity (0 one element, 1 about one
    percent, 2 all) and seed."""
    if severity == 2:
        return np.ones((M, N), dtype=bool)
    if severity == 1:
        idx = np.arange(M * N, dtype=np.uint64)
        x = (idx ^ np.uint64(seed & 0xFFFFFFFF)) & np.uint64(0xFFFFFFFF)
        x ^= x >> np.uint64(16)
        x = (x * np.uint64(0x7FEB352D)) & np.uint64(0xFFFFFFFF)
        x ^= x >> np.uint64(15)
        x = (x * np.uint64(0x846CA68B)) & np.uint64(0xFFFFFFFF)
        x ^= x >> np.uint64(16)
        return (x % np.uint64(100) == 0).reshape(M, N)
    m = np.zeros((M, N), dtype=bool)
    m[mix32(seed) % M, mix32(seed ^ 0x9E3779B9) % N] = True
    return m
