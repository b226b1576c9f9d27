"""Pins for the oracle's W8A8 GEMM (int64 accumulator, exact pow2 scaling, one RNE).

Source: "Deterministic LLM Inference Across GPU Kernels: Power-of-Two INT8
Quantization Scales ...", §II "Pipeline and alibi" (Y = (A W^T) s_a s_w with an
INT32 accumulator; any tiling / split-K / tree gives the identical accumulator;
pow2 scales make the two multiplication orders agree) and §II.E (int64 reference
accumulator). All-ones probe: "Taming Bitwise Behavior in GPU Kernels with Tensor
Core", Appendix D.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from exact import pow2, rne_bf16_exact


def _rand(seed, M, N, K, elo=-12, ehi=-4):
    rng = np.random.default_rng(seed)
    A = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    W = rng.integers(-128, 128, size=(N, K), dtype=np.int8)
    ea = rng.integers(elo, ehi + 1, size=M, dtype=np.int32)
    ew = rng.integers(elo, ehi + 1, size=N, dtype=np.int32)
    return A, W, ea, ew


def test_w8a8_bruteforce_tiny(oracle_mod):
    # Python-int dot products and exact-rational rounding on tiny shapes
    for seed, (M, N, K) in enumerate([(1, 1, 1), (3, 5, 7), (4, 6, 33), (2, 3, 130)]):
        A, W, ea, ew = _rand(seed, M, N, K, -140, 20)
        C = oracle_mod.w8a8(A, W, ea, ew)
        for i in range(M):
            for j in range(N):
                acc = sum(int(A[i, k]) * int(W[j, k]) for k in range(K))
                want = rne_bf16_exact(Fraction(acc) * pow2(int(ea[i]) + int(ew[j])))
                assert int(C[i, j]) == want, (i, j, acc)


def test_accumulator_bruteforce(oracle_mod):
    A, W, _, _ = _rand(11, 5, 7, 300)
    C = oracle_mod.gemm_s8_i32(A, W)
    for i in range(5):
        for j in range(7):
            assert int(C[i, j]) == sum(int(A[i, k]) * int(W[j, k]) for k in range(300))


def test_all_ones_probe_gives_K(oracle_mod):
    # golden: all-ones operands make every accumulator equal K (8648, not 8640)
    path = os.path.join(os.path.dirname(__file__), "golden", "ones_accumulator.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    for M, N, K, want, dropped in [tuple(map(int, r)) for r in rows]:
        A = np.ones((M, K), dtype=np.int8)
        W = np.ones((N, K), dtype=np.int8)
        C = oracle_mod.gemm_s8_i32(A, W)
        assert (C == want).all() and want != dropped
        # the bf16 output rounds 8648 to 8640 (0x4607) with E = 0
        Cb = oracle_mod.w8a8(A, W, np.zeros(M, np.int32), np.zeros(N, np.int32))
        assert (Cb == 0x4607).all()


def test_tail_sentinel_picked_up_once(oracle_mod):
    # one nonzero at position k* (walked over the K tail): acc = A[i,k*] * W[j,k*]
    K = 200
    W = np.ones((3, K), np.int8)
    for ks in (0, 63, 64, 127, 191, 192, 199):
        A = np.zeros((2, K), np.int8)
        A[:, ks] = [5, -7]
        C = oracle_mod.gemm_s8_i32(A, W)
        assert (C[0] == 5).all() and (C[1] == -7).all()


def test_k_permutation_and_split_invariance(oracle_mod):
    # integer accumulation has no order: permuting k, or cutting K into contiguous
    # parts and adding the parts, leaves every accumulator unchanged
    A, W, ea, ew = _rand(3, 9, 11, 777)
    full = oracle_mod.gemm_s8_i32(A, W).astype(np.int64)
    perm = np.random.default_rng(0).permutation(777)
    assert (oracle_mod.gemm_s8_i32(A[:, perm], W[:, perm]) == full).all()
    for cuts in ([0, 100, 777], [0, 64, 128, 500, 777], [0, 1, 776, 777]):
        parts = sum(oracle_mod.gemm_s8_i32(np.ascontiguousarray(A[:, a:b]),
                                           np.ascontiguousarray(W[:, a:b])).astype(np.int64)
                    for a, b in zip(cuts[:-1], cuts[1:]))
        assert (parts == full).all()
    Cfull = oracle_mod.w8a8(A, W, ea, ew)
    assert (oracle_mod.w8a8(A[:, perm], W[:, perm], ea, ew) == Cfull).all()


def test_rows_are_independent_of_M(oracle_mod):
    A, W, ea, ew = _rand(5, 40, 16, 96)
    full = oracle_mod.w8a8(A, W, ea, ew)
    for M in (1, 7, 23):
        assert (oracle_mod.w8a8(A[:M].copy(), W, ea[:M].copy(), ew) == full[:M]).all()
    rows = [39, 0, 17]
    assert (oracle_mod.w8a8(A, W, ea, ew, rows=rows) == full[rows]).all()


def test_pow2_commutation(oracle_mod):
    # the result depends on ea_i + ew_j only: moving the scale between the two
    # factors (or applying it in either order) gives identical bits
    A, W, ea, ew = _rand(8, 12, 10, 64, -30, 10)
    C = oracle_mod.w8a8(A, W, ea, ew)
    E = ea[:, None].astype(np.int64) + ew[None, :]
    # fold every (i, j) exponent into the row exponent of a one-row problem
    for i in range(12):
        for j in range(0, 10, 3):
            c = oracle_mod.w8a8(A[i:i + 1], W[j:j + 1], np.array([E[i, j]], np.int32),
                                np.zeros(1, np.int32))
            d = oracle_mod.w8a8(A[i:i + 1], W[j:j + 1], np.zeros(1, np.int32),
                                np.array([E[i, j]], np.int32))
            assert c[0, 0] == C[i, j] == d[0, 0]


def test_worst_case_bound_and_precondition(oracle_mod):
    # K * 128^2 < 2^31 holds up to K = 131071: all -128 operands stay exact
    K = 131071
    A = np.full((1, K), -128, np.int8)
    W = np.full((1, K), -128, np.int8)
    assert int(oracle_mod.gemm_s8_i32(A, W)[0, 0]) == K * 16384
    # one more element leaves the int32 accumulator: the oracle refuses
    A = np.full((1, K + 1), -128, np.int8)
    W = np.full((1, K + 1), -128, np.int8)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.gemm_s8_i32(A, W)


def test_zero_and_negative_zero(oracle_mod):
    A = np.array([[0, 0], [1, 0]], np.int8)
    W = np.array([[1, 1], [-1, 0]], np.int8)
    C = oracle_mod.w8a8(A, W, np.array([0, -300], np.int32), np.array([0, 0], np.int32))
    assert C[0, 0] == 0x0000 and C[0, 1] == 0x0000  # acc = 0 gives +0
    assert C[1, 0] == 0x0000  # 2^-300 underflows to +0
    assert C[1, 1] == 0x8000  # -2^-300 underflows to -0
