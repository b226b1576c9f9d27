"""Pins of the fixed-order fp16/bf16 GEMM oracle (the tensor-core block-FMA model of the
"GPU Arithmetic Emulator" README, section "Tensor Core Matmul": blocks of 16 exact products
and the fp32 accumulator aligned to the largest exponent in a window of 23 + 2 fraction
bits, terms truncated toward zero, the sum truncated to fp32; K walked in order from +0).

Checked against what the page and the arithmetic fix, not against the oracle itself:
hand-worked blocks (tests/golden/blockfma_cases.txt), the closed form of a block whose
products share one exponent (the exact sum truncated to fp32, computed with Fractions),
exact small-integer dot products, and invariants (negation symmetry, which pins truncation
toward zero; power-of-two scaling; order-freedom inside a block; zero padding of K).
"""
import os
from fractions import Fraction

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


def _bits(x, dtype):
    t = torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _val(bits, dtype):
    t = torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(
        torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.float().numpy().astype(np.float64)


def _f32(bits):
    return np.asarray(bits, np.uint32).view(np.float32)


def _rz_f32_exact(v: Fraction) -> int:
    """fp32 bits of v truncated toward zero (normal range), by exact comparison."""
    if v == 0:
        return 0
    sign = 0x80000000 if v < 0 else 0
    a = abs(v)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    frac = int(a * 2 ** 23) - 2 ** 23  # floor of the 23 fraction bits
    return sign | ((e + 127) << 23) | frac


def test_hand_worked_blocks(oracle_mod):
    n = 0
    for line in open(os.path.join(HERE, "golden", "blockfma_cases.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        dtype, a, b, want = line.split()
        A = np.array([[int(x, 16) for x in a.split(",")]], np.uint16)
        W = np.array([[int(x, 16) for x in b.split(",")]], np.uint16)
        got = oracle_mod.gemm_blockfma(A, W, dtype=oracle_mod.BF16 if dtype == "bf16" else oracle_mod.F16)
        assert int(got[0, 0]) == int(want, 16), line
        n += 1
    assert n >= 6


def test_single_block_of_one_exponent_is_the_truncated_exact_sum(oracle_mod):
    # every product has exponent 0 (significands in [1, 2) times [1, 2)): no term loses a bit
    # in the window, so the block FMA is the exact sum truncated toward zero to fp32
    rng = np.random.default_rng(1)
    for dtype in ("bf16", "fp16"):
        p = 7 if dtype == "bf16" else 10
        for _ in range(200):
            K = int(rng.integers(1, 17))
            a = (1 + rng.integers(0, 2 ** p, K) / 2 ** p) * rng.choice([-1, 1], K)
            b = 1 + rng.integers(0, 2 ** p, K) / 2 ** p
            A, W = _bits(a[None], dtype), _bits(b[None], dtype)
            exact = sum(Fraction(float(x)) * Fraction(float(y)) for x, y in zip(_val(A, dtype)[0], _val(W, dtype)[0]))
            got = oracle_mod.gemm_blockfma(A, W, dtype=oracle_mod.BF16 if dtype == "bf16" else oracle_mod.F16)
            assert int(got[0, 0]) == _rz_f32_exact(exact), (dtype, a, b)


def test_small_integer_dot_products_are_exact(oracle_mod):
    rng = np.random.default_rng(2)
    A = rng.integers(-8, 9, (7, 300)).astype(np.float32)
    W = rng.integers(-8, 9, (5, 300)).astype(np.float32)
    got = _f32(oracle_mod.gemm_blockfma(_bits(A, "bf16"), _bits(W, "bf16")))
    assert (got.astype(np.float64) == A.astype(np.float64) @ W.T.astype(np.float64)).all()


def _random(rng, M, N, K, spread, dtype):
    a = rng.standard_normal((M, K)) * np.exp2(rng.integers(-spread, spread + 1, (M, K)))
    w = rng.standard_normal((N, K)) * np.exp2(rng.integers(-spread, spread + 1, (N, K)))
    return _bits(a, dtype), _bits(w, dtype)


def test_invariants(oracle_mod):
    rng = np.random.default_rng(3)
    for dtype, dt in (("bf16", oracle_mod.BF16), ("fp16", oracle_mod.F16)):
        A, W = _random(rng, 9, 11, 77, 6 if dtype == "fp16" else 20, dtype)
        C = oracle_mod.gemm_blockfma(A, W, dtype=dt)
        # negation symmetry: truncation toward zero treats both signs alike (a floor would not)
        assert (oracle_mod.gemm_blockfma(A ^ np.uint16(0x8000), W, dtype=dt) == C ^ np.uint32(0x80000000)).all()
        # zero padding of K changes nothing (a block of zero products keeps the accumulator)
        Ap = np.concatenate([A, np.zeros((9, 35), np.uint16)], axis=1)
        Wp = np.concatenate([W, np.zeros((11, 35), np.uint16)], axis=1)
        assert (oracle_mod.gemm_blockfma(Ap, Wp, dtype=dt) == C).all()
        # order inside a block is free: permute the 16 columns of every block alike
        perm = np.concatenate([b * 16 + rng.permutation(16) for b in range(77 // 16)] +
                              [np.arange(77 // 16 * 16, 77)])
        assert (oracle_mod.gemm_blockfma(A[:, perm], W[:, perm], dtype=dt) == C).all()
    # power-of-two scaling of A (bf16 exponent field + 3, no overflow): result exponent + 3
    A, W = _random(rng, 6, 7, 50, 10, "bf16")
    nz = (A & 0x7F80) != 0
    A3 = np.where(nz, A + np.uint16(3 << 7), A).astype(np.uint16)
    C = oracle_mod.gemm_blockfma(A, W)
    C3 = oracle_mod.gemm_blockfma(A3, W)
    cnz = (C & 0x7F800000) != 0
    assert (C3[cnz] == C[cnz] + np.uint32(3 << 23)).all()


def test_order_across_blocks_matters(oracle_mod):
    # the same products regrouped across blocks give different sums somewhere: the walk
    # order is part of the definition (the point of a written descriptor)
    rng = np.random.default_rng(4)
    A, W = _random(rng, 16, 16, 64, 12, "bf16")
    C = oracle_mod.gemm_blockfma(A, W)
    rot = np.roll(np.arange(64), 8)
    C2 = oracle_mod.gemm_blockfma(A[:, rot], W[:, rot])
    assert (C != C2).any()
