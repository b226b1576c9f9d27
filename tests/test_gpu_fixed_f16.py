"""GPU parity of the fixed-order fp16/bf16 GEMM (detgemm_gemm_fixed_f16) with the oracle's
tensor-core block-FMA model ("GPU Arithmetic Emulator" README, "Tensor Core Matmul"; the
descriptor of "Taming Bitwise Behavior in GPU Kernels with Tensor Core", §3.2.1-§3.2.2: K
walked in 16-wide blocks in order, never split). Bit-exact fp32 comparisons; rows identical
across M; ragged shapes with K tails; a 4096^3 bf16 case on sampled rows and on every row
of sampled columns."""
import numpy as np
import pytest
import torch

from gpu_util import cuda, dg, padded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda()


@pytest.fixture(scope="module")
def lib():
    return dg()


def _bits(x, tdt):
    return torch.from_numpy(np.asarray(x, np.float32)).to(tdt).view(torch.int16).numpy().view(np.uint16)


def _data(rng, M, N, K, spread, tdt, cancel=False):
    a = rng.standard_normal((M, K)) * np.exp2(rng.integers(-spread, spread + 1, (M, K)))
    w = rng.standard_normal((N, K)) * np.exp2(rng.integers(-spread, spread + 1, (N, K)))
    if cancel:  # neighbouring products nearly cancel
        a[:, 1::2] = a[:, 0::2][:, : a[:, 1::2].shape[1]]
        w[:, 1::2] = -w[:, 0::2][:, : w[:, 1::2].shape[1]] * (1 + 2.0 ** -7)
    return _bits(a, tdt), _bits(w, tdt)


def _run(lib, dev, A, W, tdt, ld=None):
    M, K = A.shape
    ld = ld or (K + 7) // 8 * 8
    tA = padded(A.view(np.int16), dev, ld).view(tdt)
    tW = padded(W.view(np.int16), dev, ld).view(tdt)
    out = lib.gemm_fixed_f16(tA, tW)
    return out.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("tdt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("M,N,K,spread,cancel", [
    (1, 1, 1, 0, False), (7, 13, 33, 4, False), (128, 256, 64, 0, False), (130, 257, 1000, 6, False),
    (300, 100, 517, 3, True), (257, 64, 4096, 5, False), (64, 300, 2048, 0, True)])
def test_bitexact_against_the_block_fma_model(lib, dev, oracle_mod, tdt, M, N, K, spread, cancel):
    rng = np.random.default_rng(M * 7 + N + K + spread)
    if tdt == torch.float16:
        spread = min(spread, 5)  # keep fp16 values and fp32 sums in range
    A, W = _data(rng, M, N, K, spread, tdt, cancel)
    dt = oracle_mod.BF16 if tdt == torch.bfloat16 else oracle_mod.F16
    want = oracle_mod.gemm_blockfma(A, W, dtype=dt)
    got = _run(lib, dev, A, W, tdt)
    assert (got == want).all(), int((got != want).sum())


def test_rows_identical_across_M(lib, dev, oracle_mod):
    rng = np.random.default_rng(9)
    A, W = _data(rng, 1024, 512, 1536, 8, torch.bfloat16)
    want = oracle_mod.gemm_blockfma(A, W)
    for M in (1, 5, 64, 200, 1024):
        got = _run(lib, dev, np.ascontiguousarray(A[:M]), W, torch.bfloat16)
        assert (got == want[:M]).all(), M


def test_4096_cube_sampled(lib, dev, oracle_mod):
    rng = np.random.default_rng(10)
    A, W = _data(rng, 4096, 4096, 4096, 2, torch.bfloat16)
    got = _run(lib, dev, A, W, torch.bfloat16)
    rows = [0, 1, 255, 256, 2047, 4095] + rng.integers(0, 4096, 4).tolist()
    assert (got[rows] == oracle_mod.gemm_blockfma(np.ascontiguousarray(A[rows]), W)).all()
    cols = sorted({0, 255, 256, 4095} | {256 * t + int(rng.integers(0, 256)) for t in range(16)})
    want = oracle_mod.gemm_blockfma(A, np.ascontiguousarray(W[cols]))
    assert (got[:, cols] == want).all()
