"""GPU parity of the Ozaki-scheme fp32 GEMM against the CPU oracle (bit-exact), plus the
error bound |C - C_fp64| <= 4 * 2^-24 * (|A||B|)_ij on the full-size workload."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import cuda, dg, f32_bits, padded, poison_like, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda()


@pytest.fixture(scope="module")
def lib():
    return dg()


def run(lib, dev, A, B, split=1, nslices=7, max_diag=8, lda=None, ldb=None):
    M, K = A.shape
    N = B.shape[1]
    tA = padded(A, dev, lda) if lda else to_dev(A, dev)
    tB = padded(B, dev, ldb) if ldb else to_dev(B, dev)
    out = poison_like((M, N), torch.float32, dev)
    lib.ozaki_f32(tA, tB, nslices=nslices, max_diag=max_diag, split_k=split, out=out)
    return f32_bits(out)


@pytest.mark.parametrize("M,N,K,split,nslices,max_diag", [
    (64, 96, 256, 1, 7, 8), (33, 17, 100, 2, 7, 8), (130, 129, 513, 3, 7, 8), (1, 1, 1, 1, 7, 8),
    (70, 40, 300, 1, 4, 5), (20, 24, 64, 1, 7, 14), (257, 65, 1024, 4, 7, 8)])
def test_small_bitexact(lib, dev, oracle_mod, M, N, K, split, nslices, max_diag):
    rng = np.random.default_rng(M + 7 * N + K)
    A = (rng.standard_normal((M, K)) * np.exp2(rng.integers(-8, 9, size=(M, K)))).astype(np.float32)
    B = (rng.standard_normal((K, N)) * np.exp2(rng.integers(-8, 9, size=(K, N)))).astype(np.float32)
    lda = (K + 3) // 4 * 4
    ldb = (N + 3) // 4 * 4
    want = oracle_mod.ozaki_f32(A, B, nslices, max_diag).view(np.uint32)
    got = run(lib, dev, A, B, split, nslices, max_diag, lda, ldb)
    assert (got == want).all(), int((got != want).sum())


def test_combine_order_case(lib, dev):
    # the hand-worked cancellation case: the defined order g = 8..2 gives +0.0
    K = 130
    x = np.full((1, K), 0.5, np.float32)
    x[0, 129] = 2.0 ** -7
    y = np.full((K, 1), -(2.0 ** -8), np.float32)
    y[0, 0] = 0.5
    y[129, 0] = 2.0 ** -49
    got = run(lib, dev, x, y, lda=132, ldb=4)
    assert got[0, 0] == 0


def _tile_columns(N, seed):
    """One column at a random offset inside every 256-wide tile column, plus the edges."""
    rng = np.random.default_rng(seed)
    cols = {0, 1, 127, 128, 255, N - 256, N - 129, N - 1}
    for t in range((N + 255) // 256):
        cols.add(min(N - 1, 256 * t + int(rng.integers(0, 256))))
    return sorted(cols)


def test_ozaki_workload_bitexact_sampled_and_error_bound_everywhere(lib, dev, oracle_mod):
    """4096^3: ten whole rows and every row of one column per 256-wide tile column
    bit-exact against the oracle; the bound |C - AB| <= 4 * 2^-24 * (|A||B|)_ij on every
    element (checked against an fp64 product, whose own error, at most K * 2^-53 * (|A||B|)_ij,
    is taken off the allowance)."""
    A, B = synthetic.ozaki(4096)
    tA, tB = to_dev(A, dev), to_dev(B, dev)
    out = poison_like((4096, 4096), torch.float32, dev)
    lib.ozaki_f32(tA, tB, out=out)
    C = out.cpu().numpy()
    rows = [0, 1, 127, 128, 2047, 4094, 4095] + np.random.default_rng(3).integers(0, 4096, 3).tolist()
    want = oracle_mod.ozaki_f32(A, B, rows=rows)
    assert (C[rows].view(np.uint32) == want.view(np.uint32)).all()
    cols = _tile_columns(4096, 8)
    want = oracle_mod.ozaki_f32(A, np.ascontiguousarray(B[:, cols]))
    got = np.ascontiguousarray(C[:, cols])
    assert (got.view(np.uint32) == want.view(np.uint32)).all(), int((got != want).sum())
    A64, B64 = A.astype(np.float64), B.astype(np.float64)
    ref = A64 @ B64
    absab = np.abs(A64) @ np.abs(B64)
    allowance = (4 * 2.0 ** -24 - 4096 * 2.0 ** -52) * absab
    assert (np.abs(C.astype(np.float64) - ref) <= allowance).all()


def test_ozaki_workload_identical_across_real_cuts(lib, dev, oracle_mod):
    """4096^3 with every diagonal's K range cut into exactly 1 and 3 parts (reported by the
    call): byte-identical to the plain call, and bit-exact against the oracle on sampled rows."""
    A, B = synthetic.ozaki(4096)
    tA, tB = to_dev(A, dev), to_dev(B, dev)
    out = poison_like((4096, 4096), torch.float32, dev)
    lib.ozaki_f32(tA, tB, out=out)
    rows = [0, 255, 256, 3000, 4095]
    want = oracle_mod.ozaki_f32(A, B, rows=rows).view(np.uint32)
    for parts in (1, 3):
        out2 = poison_like((4096, 4096), torch.float32, dev)
        _, run = lib.ozaki_f32_split_exact(tA, tB, split_k=parts, out=out2)
        assert run == parts
        assert torch.equal(out.view(torch.int32), out2.view(torch.int32)), parts
        assert (f32_bits(out2)[rows] == want).all(), parts


def test_small_real_cuts(lib, dev, oracle_mod):
    """Small Ozaki problems at cuts up to one 64-wide K block per part of the lightest
    diagonal, bit-exact against the oracle."""
    for M, N, K, split in [(130, 129, 513, 9), (257, 65, 1024, 16), (33, 17, 100, 2)]:
        rng = np.random.default_rng(M + N + K)
        A = (rng.standard_normal((M, K)) * np.exp2(rng.integers(-8, 9, size=(M, K)))).astype(np.float32)
        B = (rng.standard_normal((K, N)) * np.exp2(rng.integers(-8, 9, size=(K, N)))).astype(np.float32)
        tA = padded(A, dev, (K + 3) // 4 * 4)
        tB = padded(B, dev, (N + 3) // 4 * 4)
        out = poison_like((M, N), torch.float32, dev)
        _, run = lib.ozaki_f32_split_exact(tA, tB, split_k=split, out=out)
        assert run == split
        want = oracle_mod.ozaki_f32(A, B).view(np.uint32)
        assert (f32_bits(out) == want).all(), (M, N, K, split)


def _diagonals(rng, nd, M, N):
    # full-range, small, and trailing-zero-heavy sums: every rounding of the combine,
    # including exact ties at the 53-bit boundary, is reached
    full = rng.integers(-2 ** 31 + 1, 2 ** 31, size=(nd, M, N), dtype=np.int64)
    small = rng.integers(-3000, 3001, size=(nd, M, N), dtype=np.int64)
    shifted = rng.integers(-2 ** 10, 2 ** 10, size=(nd, M, N), dtype=np.int64) << rng.integers(0, 20, size=(nd, M, N))
    pick = rng.integers(0, 3, size=(nd, M, N))
    T = np.where(pick == 0, full, np.where(pick == 1, small, shifted))
    return np.clip(T, -2 ** 31 + 1, 2 ** 31 - 1).astype(np.int32)


@pytest.mark.parametrize("max_diag", [2, 3, 5, 8, 9, 13, 14, 18])
def test_combine_step_bitexact(lib, dev, oracle_mod, max_diag):
    """detgemm_ozaki_combine against the oracle's fp64 loop, element by element: ragged N
    (the scalar tail), a padded row stride, and exponents reaching fp32 subnormals and
    overflow."""
    rng = np.random.default_rng(100 + max_diag)
    M, N, ldT = 37, 1003, 1012
    T = _diagonals(rng, max_diag - 1, M, N)
    e = rng.integers(-40, 41, size=M).astype(np.int32)
    f = rng.integers(-40, 41, size=N).astype(np.int32)
    e[:4] = [-150, -120, 100, 140]
    f[:6] = [-160, -60, 0, 60, 130, 2 ** 31 - 1]
    f[6] = -2 ** 31
    tT = torch.zeros((max_diag - 1, M, ldT), dtype=torch.int32, device=dev)[:, :, :N]
    tT.copy_(torch.from_numpy(T))
    out = poison_like((M, N), torch.float32, dev)
    lib.ozaki_combine(tT, to_dev(e, dev), to_dev(f, dev), out=out)
    got = f32_bits(out)
    want = oracle_mod.ozaki_combine(T, e, f).view(np.uint32)
    assert (got == want).all(), int((got != want).sum())
    assert lib.device_status() == lib.OK
