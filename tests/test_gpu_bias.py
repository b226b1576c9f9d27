"""GPU parity of the biased W8A8 epilogue, C = rne_bf16(acc * 2^(ea + ew) + b_j) rounded
once ("Deterministic LLM Inference Across GPU Kernels ...", §II "Pipeline and alibi": the
epilogue is the one rounding of the exactly scaled accumulator; the bias joins the exact
value first), against the oracle bit for bit: the tensor-core engine (its fp32 round-down/up
form and its integer form), split-K, the decode-shaped kernels (whole-K and split chain),
and the fused linear layer with a bias; special biases (+-0, +-inf, NaN, subnormal,
huge, the negated output) in some columns."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import bf16_bits, cuda, dg, padded, poison_like, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda()


@pytest.fixture(scope="module")
def lib():
    return dg()


def _bf16(x: np.ndarray) -> np.ndarray:
    """round-to-nearest-even fp32 -> bf16 bit patterns (input generation only)."""
    b = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def _bias(seed, N, scale, neg_of=None):
    """bf16 biases of about the outputs' size; a few columns hold special values and, when
    neg_of (one output row, bf16 bits) is given, some hold that row's negated output so the
    sum cancels to a few units."""
    rng = np.random.default_rng(seed)
    b = _bf16(rng.standard_normal(N) * scale)
    special = [0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x8005, 0x6F00, 0xEF00]
    for j, v in enumerate(special[:N]):
        b[j] = v
    if neg_of is not None:
        for j in range(len(special), N, 5):
            b[j] = neg_of[j] ^ 0x8000
    return b


def _check(lib, dev, oracle_mod, A, W, ea, ew, bias, split=1):
    want = oracle_mod.w8a8_bias(A, W, ea, ew, bias)
    M, N = A.shape[0], W.shape[0]
    out = poison_like((M, N), torch.bfloat16, dev)
    tb = to_dev(bias.view(np.int16), dev).view(torch.bfloat16)
    got = lib.w8a8(to_dev(A, dev), to_dev(W, dev), to_dev(ea, dev), to_dev(ew, dev), split_k=split, out=out,
                   bias=tb)
    g = bf16_bits(got)
    bad = np.argwhere(g != want)
    assert bad.size == 0, (A.shape, W.shape, split, bad[:5], g[tuple(bad[0])] if bad.size else None)
    return g


# (M, N, K, split): tensor-core engine (M > 64) incl. split-K and ragged edges; decode
# kernels (M <= 64): whole K (K <= 4096) and the split chain (K > 4096)
SHAPES = [(300, 264, 1024, 1), (512, 768, 1024, 3), (257, 520, 2048, 1), (130, 100, 208, 1),
          (65, 72, 4096, 2), (16, 256, 512, 1), (64, 304, 4096, 1), (17, 100, 5008, 1), (1, 33, 4112, 1)]


@pytest.mark.parametrize("M,N,K,split", SHAPES)
def test_bias_typical_exponents(lib, dev, oracle_mod, M, N, K, split):
    A, W, ea, ew = synthetic.w8a8_normal(300 + M, M, N, K, 25.0, 35.0, -14, -6)
    plain = oracle_mod.w8a8(A, W, ea, ew)
    scale = float(np.sqrt(K) * 25.0 * 35.0 * 2.0 ** -20)  # about |acc| * 2^E at E = -20
    bias = _bias(M + N, N, scale, neg_of=plain[0])
    _check(lib, dev, oracle_mod, A, W, ea, ew, bias, split)


@pytest.mark.parametrize("M,N,K", [(300, 264, 1024), (16, 256, 512)])
def test_bias_extreme_exponents_and_large_accumulators(lib, dev, oracle_mod, M, N, K):
    # exponents outside the fast range and |acc| >= 2^24: the engine's integer form
    rng = np.random.default_rng(M * 7 + K)
    A = np.where(rng.random((M, K)) < 0.5, 127, -127).astype(np.int8)
    W = np.where(rng.random((N, K)) < 0.5, 127, -127).astype(np.int8)
    A[: M // 2, :] = 127
    W[: N // 3, :] = 127  # |acc| = K * 127^2 > 2^24 in the top-left block
    ea = rng.integers(-150, 70, M).astype(np.int32)
    ew = rng.integers(-60, 60, N).astype(np.int32)
    # in-range exponents for two whole warps of rows and one 128-column group, so that the
    # engine's fast form meets large accumulators and hands them to the integer form
    ea[: min(M, 64)] = rng.integers(-20, -5, min(M, 64))
    ew[: min(N, 128)] = rng.integers(-20, -5, min(N, 128))
    bias = _bf16(rng.standard_normal(N).astype(np.float32) * np.exp2(rng.integers(-120, 120, N)).astype(np.float32))
    bias[:4] = [0x4F00, 0xCF00, 0x0001, 0x8000]
    _check(lib, dev, oracle_mod, A, W, ea, ew, bias)


def test_bias_rows_identical_across_batch_and_split(lib, dev, oracle_mod):
    # a row's biased output does not depend on M (engine or decode kernels) or on split-K
    A, W, ea, ew = synthetic.w8a8_normal(77, 520, 384, 2048, 25.0, 35.0, -14, -6)
    bias = _bias(5, 384, 2.0 ** -6)
    full = _check(lib, dev, oracle_mod, A, W, ea, ew, bias, 1)
    full3 = _check(lib, dev, oracle_mod, A, W, ea, ew, bias, 4)
    assert (full == full3).all()
    for m in (1, 40, 64, 65, 300):
        part = _check(lib, dev, oracle_mod, A[:m], W, ea[:m], ew, bias)
        assert (part == full[:m]).all(), m


@pytest.mark.parametrize("M,N,K,split,w16", [(8, 96, 512, 1, False), (100, 200, 2048, 1, False),
                                             (300, 264, 1024, 2, True), (64, 128, 5008, 1, False)])
def test_linear_with_bias(lib, dev, oracle_mod, M, N, K, split, w16):
    rng = np.random.default_rng(M + K)
    X = (rng.standard_normal((M, K)) * 2.0).astype(np.float32)
    W = synthetic.normal_i8(21, 1, (N, K), 40.0)
    ew = synthetic.uniform_i32(21, 3, (N,), -14, -6)
    Q, ea = oracle_mod.quantize_pow2(X, 0)
    bias = _bias(N, N, 0.5)
    want = oracle_mod.w8a8_bias(Q, W, ea, ew, bias)
    tW = to_dev(W, dev)
    W16 = lib.widen_i8_f16(tW) if w16 else None
    tb = to_dev(bias.view(np.int16), dev).view(torch.bfloat16)
    got = lib.linear_w8a8(to_dev(X, dev), tW, to_dev(ew, dev), W16=W16, split_k=split, bias=tb)
    assert (bf16_bits(got) == want).all()


def test_bias_with_strided_operands(lib, dev, oracle_mod):
    A, W, ea, ew = synthetic.w8a8_normal(91, 200, 136, 1000, 25.0, 35.0, -14, -6)
    bias = _bias(3, 136, 2.0 ** -8)
    want = oracle_mod.w8a8_bias(A, W, ea, ew, bias)
    tA, tW = padded(A, dev, 1024), padded(W, dev, 1040)
    tb = to_dev(bias.view(np.int16), dev).view(torch.bfloat16)
    got = lib.w8a8(tA, tW, to_dev(ea, dev), to_dev(ew, dev), bias=tb)
    assert (bf16_bits(got) == want).all()
