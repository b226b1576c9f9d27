"""detgemm_w8a8_noalloc, called through the C ABI, against detgemm_w8a8 and the oracle.

The allocation-free entry point serves callers that cannot allocate device memory at
call time (a plugin handed only its input and output tensors, a serving loop that bans
cudaMalloc because it can stall the device). It must return the very same bits as the
regular entry point, including when called twice in a row, since its scratch array
keeps the previous call's contents. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthetic
from gpu_util import bf16_bits, cuda, dg, padded, to_dev

pytestmark = pytest.mark.gpu


def _noalloc(lib, A, W, ea, ew, C, split):
    M, K = A.shape
    N = W.shape[0]
    return lib.detgemm_w8a8_noalloc(A.data_ptr(), A.stride(0), W.data_ptr(), W.stride(0), ea.data_ptr(),
                                    ew.data_ptr(), C.data_ptr(), C.stride(0), M, N, K, split,
                                    torch.cuda.current_stream().cuda_stream)


def _run_and_compare(m, lib, dev, A, W, ea, ew, splits, ld=None, oracle_mod=None):
    """Two noalloc calls in a row per split against detgemm_w8a8 (and the oracle if given)."""
    M, K = A.shape
    N = W.shape[0]
    if ld is None:
        tA, tW = to_dev(A, dev), to_dev(W, dev)
    else:
        tA, tW = padded(A, dev, ld), padded(W, dev, ld)
    tea, tew = to_dev(ea, dev), to_dev(ew, dev)
    want = oracle_mod.w8a8(A, W, ea, ew) if oracle_mod is not None else None
    for split in splits:
        ref = m.w8a8(tA, tW, tea, tew, split_k=split)
        if want is not None:
            assert (bf16_bits(ref) == want).all(), split
        for _ in range(2):  # two calls in a row share the scratch array
            C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
            assert _noalloc(lib, tA, tW, tea, tew, C, split) == m.OK
            torch.cuda.synchronize()
            assert torch.equal(C.view(torch.int16), ref.view(torch.int16)), split
            if want is not None:
                assert (bf16_bits(C) == want).all(), split


@pytest.mark.parametrize("case", ["skinny", "tile"])
def test_noalloc_matches_w8a8_twice(case, oracle_mod):
    dev = cuda()
    m = dg()
    lib = m.load()
    if case == "skinny":
        A, W, ea, ew = synthetic.skinny()
        _run_and_compare(m, lib, dev, A, W, ea, ew, (8, 32), oracle_mod=oracle_mod)
    else:
        rng = np.random.default_rng(11)
        A = rng.integers(-128, 128, size=(300, 3008), dtype=np.int8)
        W = rng.integers(-128, 128, size=(1000, 3008), dtype=np.int8)
        ea = rng.integers(-14, -6, size=300, dtype=np.int32)
        ew = rng.integers(-14, -6, size=1000, dtype=np.int32)
        _run_and_compare(m, lib, dev, A, W, ea, ew, (3, 1), oracle_mod=oracle_mod)


def test_noalloc_tile_kernel_k_tail(oracle_mod):
    """Above 64 rows the call runs the int8 warp-MMA tile kernel; K = 3000 (padded rows of
    3008) leaves a partial last K block, at one and several K parts."""
    dev = cuda()
    m = dg()
    lib = m.load()
    rng = np.random.default_rng(12)
    A = rng.integers(-128, 128, size=(300, 3000), dtype=np.int8)
    W = rng.integers(-128, 128, size=(1000, 3000), dtype=np.int8)
    ea = rng.integers(-14, -6, size=300, dtype=np.int32)
    ew = rng.integers(-14, -6, size=1000, dtype=np.int32)
    _run_and_compare(m, lib, dev, A, W, ea, ew, (1, 3, 7), ld=3008, oracle_mod=oracle_mod)


def test_noalloc_refuses_by_its_own_scratch_size(oracle_mod):
    """The refusal follows detgemm_w8a8_noalloc_scratch_size, the scratch the call uses: a
    split problem needing 16 MiB is refused; the 2048-row sweep GEMM at split 1 needs none
    (detgemm_w8a8 would need ~28 MiB for its fp16 operand copies) and runs, bit-exact."""
    dev = cuda()
    m = dg()
    lib = m.load()
    M, N, K = 1024, 4096, 256  # split-K scratch 16 MiB > the fixed 8 MiB array
    need = lib.detgemm_w8a8_noalloc_scratch_size(M, N, K, 2)
    assert need >= M * N * 4 > m.NOALLOC_SCRATCH_BYTES
    A = torch.zeros((M, K), dtype=torch.int8, device=dev)
    W = torch.zeros((N, K), dtype=torch.int8, device=dev)
    e = torch.zeros((max(M, N),), dtype=torch.int32, device=dev)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    assert _noalloc(lib, A, W, e, e, C, 2) == m.ERR_WORKSPACE
    A, W, ea, ew = synthetic.sweep(2048)
    assert lib.detgemm_w8a8_noalloc_scratch_size(2048, 6144, 2048, 1) == 0
    assert m.w8a8_workspace_size(2048, 6144, 2048, 1) > m.NOALLOC_SCRATCH_BYTES
    _run_and_compare(m, lib, dev, A, W, ea, ew, (1,), oracle_mod=oracle_mod)
