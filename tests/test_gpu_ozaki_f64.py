"""GPU parity of the fp64-target Ozaki GEMM (DGEMM emulation on exact integer slice
products), its fp64 slicer and its fp64-output combine against the CPU oracle, bit for bit,
plus the error bound on the 4096-size workload."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import cuda, dg, padded, poison_like, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda()


@pytest.fixture(scope="module")
def lib():
    return dg()


def f64_bits(t):
    return t.cpu().numpy().view(np.uint64)


def _operands(rng, M, N, K, spread):
    A = rng.standard_normal((M, K)) * np.exp2(rng.integers(-spread, spread + 1, size=(M, K)))
    B = rng.standard_normal((K, N)) * np.exp2(rng.integers(-spread, spread + 1, size=(K, N)))
    if M > 3:
        A[2] = 0.0                      # a zero row
        A[3, ::3] = 5e-324 * 7          # subnormals inside a row of normal values
    if N > 2:
        B[:, 1] = 0.0                   # a zero column
    return A, B


@pytest.mark.parametrize("M,N,K,split,nslices,max_diag,spread", [
    (64, 96, 256, 1, 8, 9, 8), (33, 17, 100, 2, 8, 9, 20), (130, 129, 513, 3, 8, 9, 4), (1, 1, 1, 1, 8, 9, 0),
    (70, 40, 300, 1, 11, 12, 30), (20, 24, 64, 1, 6, 12, 8), (257, 65, 1024, 4, 8, 9, 8), (40, 50, 200, 1, 9, 14, 10)])
def test_small_bitexact(lib, dev, oracle_mod, M, N, K, split, nslices, max_diag, spread):
    rng = np.random.default_rng(M + 7 * N + K + nslices)
    A, B = _operands(rng, M, N, K, spread)
    want = oracle_mod.ozaki_f64(A, B, nslices, max_diag).view(np.uint64)
    tA = padded(A, dev, (K + 1) // 2 * 2)
    tB = padded(B, dev, (N + 1) // 2 * 2)
    out = poison_like((M, N), torch.float64, dev)
    lib.ozaki_f64(tA, tB, nslices=nslices, max_diag=max_diag, split_k=split, out=out)
    got = f64_bits(out)
    assert (got == want).all(), int((got != want).sum())
    assert lib.device_status() == lib.OK


@pytest.mark.parametrize("nslices", [8, 12])
@pytest.mark.parametrize("rows,cols", [(37, 100), (64, 64), (5, 3)])
def test_slice_f64_rows_and_cols(lib, dev, oracle_mod, nslices, rows, cols):
    rng = np.random.default_rng(rows * cols + nslices)
    X, _ = _operands(rng, rows, 1, cols, 40)
    for axis in (0, 1):
        Sw, ew = oracle_mod.slice_f64(X, axis, nslices)
        S, e = lib.slice_f64(padded(X, dev, (cols + 1) // 2 * 2), axis, nslices)
        assert (e.cpu().numpy() == ew).all()
        assert (S.cpu().numpy() == Sw).all()


@pytest.mark.parametrize("max_diag", [2, 9, 13, 14, 18])
def test_combine_step_f64_bitexact(lib, dev, oracle_mod, max_diag):
    rng = np.random.default_rng(200 + max_diag)
    M, N = 29, 515
    T = rng.integers(-2 ** 31 + 1, 2 ** 31, size=(max_diag - 1, M, N)).astype(np.int32)
    T[:, :, ::5] = (T[:, :, ::5] >> 12) << 12  # trailing zeros: ties at the 53-bit boundary
    e = rng.integers(-600, 600, size=M).astype(np.int32)
    f = rng.integers(-600, 600, size=N).astype(np.int32)
    e[:3] = [-1080, -1040, 1000]   # fp64 subnormal results, and overflow
    f[:3] = [-20, 30, 90]
    tT = torch.zeros((max_diag - 1, M, 516), dtype=torch.int32, device=dev)[:, :, :N]
    tT.copy_(torch.from_numpy(T))
    out = poison_like((M, N), torch.float64, dev)
    lib.ozaki_combine(tT, to_dev(e, dev), to_dev(f, dev), out=out, dtype=torch.float64)
    got = f64_bits(out)
    want = oracle_mod.ozaki_combine_f64(T, e, f).view(np.uint64)
    assert (got == want).all(), int((got != want).sum())


def test_ozaki_f64_workload_sampled_and_error_bound(lib, dev, oracle_mod):
    A, B = synthetic.ozaki_f64(4096)
    tA, tB = to_dev(A, dev), to_dev(B, dev)
    out = poison_like((4096, 4096), torch.float64, dev)
    lib.ozaki_f64(tA, tB, out=out)
    C = out.cpu().numpy()
    rows = [0, 1, 127, 2048, 4095]
    want = oracle_mod.ozaki_f64(A, B, rows=rows)
    assert (C[rows].view(np.uint64) == want.view(np.uint64)).all()
    # error bound against an fp64 GEMM (whose own error is at most K 2^-53 (|A||B|)_ij)
    _, e = oracle_mod.slice_f64(A[rows], 0, 8)
    _, f = oracle_mod.slice_f64(B, 1, 8)
    ref = A[rows] @ B
    absab = np.abs(A[rows]) @ np.abs(B)
    K = A.shape[1]
    bound = 2.0 ** -53 * np.abs(C[rows]) + 10 * K * np.exp2(e[:, None] + f[None, :] - 53.0) + K * 2.0 ** -53 * absab
    assert (np.abs(C[rows] - ref) <= bound).all()
    out2 = poison_like((4096, 4096), torch.float64, dev)
    lib.ozaki_f64(tA, tB, split_k=5, out=out2)
    assert torch.equal(out.view(torch.int64), out2.view(torch.int64))


def test_ozaki_f64_nonfinite_reported(lib, dev):
    A = np.ones((4, 8))
    A[1, 3] = np.nan
    lib.ozaki_f64(to_dev(A, dev), to_dev(np.ones((8, 2)), dev))
    assert lib.device_status() == lib.ERR_NONFINITE
