"""detgemm_w8a8_noalloc, called through the C ABI, against detgemm_w8a8.

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
from gpu_util import cuda, dg, to_dev

pytestmark = pytest.mark.gpu


def _noalloc(lib, A, W, ea, ew, C, split):
    M, K = A.shape
    N = W.shape[0]
    return lib.detgemm_w8a8_noalloc(A.data_ptr(), A.stride(0), W.data_ptr(), W.stride(0), ea.data_ptr(),
                                    ew.data_ptr(), C.data_ptr(), C.stride(0), M, N, K, split,
                                    torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("case", ["skinny", "tile"])
def test_noalloc_matches_w8a8_twice(case):
    dev = cuda()
    m = dg()
    lib = m.load()
    if case == "skinny":
        A, W, ea, ew = synthetic.skinny()
        splits = (8, 32)
    else:
        rng = np.random.default_rng(11)
        A = rng.integers(-128, 128, size=(300, 3008), dtype=np.int8)
        W = rng.integers(-128, 128, size=(1000, 3008), dtype=np.int8)
        ea = rng.integers(-14, -6, size=300, dtype=np.int32)
        ew = rng.integers(-14, -6, size=1000, dtype=np.int32)
        splits = (3, 1)
    tA, tW, tea, tew = (to_dev(x, dev) for x in (A, W, ea, ew))
    M, N = A.shape[0], W.shape[0]
    for split in splits:
        ref = m.w8a8(tA, tW, tea, tew, split_k=split)
        for _ in range(2):  # two calls in a row share the scratch array
            C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
            assert _noalloc(lib, tA, tW, tea, tew, C, split) == m.OK
            torch.cuda.synchronize()
            assert torch.equal(C.view(torch.int16), ref.view(torch.int16)), (case, split)


def test_noalloc_refuses_oversized_problem():
    dev = cuda()
    m = dg()
    lib = m.load()
    M, N, K = 1024, 4096, 256  # split-K scratch 16 MiB > the fixed 8 MiB array
    assert m.w8a8_workspace_size(M, N, K, 2) > m.NOALLOC_SCRATCH_BYTES
    A = torch.zeros((M, K), dtype=torch.int8, device=dev)
    W = torch.zeros((N, K), dtype=torch.int8, device=dev)
    e = torch.zeros((max(M, N),), dtype=torch.int32, device=dev)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    assert _noalloc(lib, A, W, e, e, C, 2) == m.ERR_WORKSPACE
