"""Stream ordering of the library's launches. Several of its kernels are launched as
programmatic dependents of the kernel before them on the stream and wait for it inside the
kernel; these tests produce every input with a GPU kernel queued immediately before the call
(behind a spin kernel, so that the library's launches are issued while the producers are
still pending) and read the output with a kernel queued immediately after, with no host
synchronisation in between, and compare the bits with the oracle."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import bf16_bits, cuda, dg, f32_bits, to_dev

pytestmark = pytest.mark.gpu

SPIN_CYCLES = 2_000_000  # about a millisecond of GPU time ahead of the producers


@pytest.fixture(scope="module")
def dev():
    return cuda()


@pytest.fixture(scope="module")
def lib():
    return dg()


def _produced(src: torch.Tensor, filler) -> torch.Tensor:
    """A buffer holding other values whose contents a kernel (an elementwise add, not a
    copy engine transfer) replaces with src, queued on the current stream."""
    dst = torch.full_like(src, filler)
    return dst, lambda: torch.add(src, 0, out=dst)


@pytest.mark.parametrize("M,N,K,split", [(16, 512, 1024, 1), (64, 304, 4096, 1), (40, 200, 5008, 1),
                                         (300, 520, 2048, 1), (512, 768, 1024, 3), (257, 6144, 2048, 1)])
def test_w8a8_inputs_written_just_before(lib, dev, oracle_mod, M, N, K, split):
    A, W, ea, ew = synthetic.w8a8_normal(80 + M, M, N, K, 25.0, 35.0, -14, -6)
    want = oracle_mod.w8a8(A, W, ea, ew)
    srcs = [to_dev(x, dev) for x in (A, W, ea, ew)]
    bufs = [_produced(s, f) for s, f in zip(srcs, (77, -5, 3, 3))]
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(lib.w8a8_workspace_size(M, N, K, split), 1), dtype=torch.uint8, device=dev)
    C.fill_(0)
    torch.cuda.synchronize()
    for rep in range(2):
        torch.cuda._sleep(SPIN_CYCLES)
        for _, produce in bufs:
            produce()
        lib.w8a8(*(b for b, _ in bufs), split_k=split, out=C, ws=ws)
        C2 = C.clone()  # a kernel that reads the output right after the call
        assert (bf16_bits(C2) == want).all(), (M, N, K, split, rep)
        for b, _ in bufs:  # poison the inputs again for the next round
            b.fill_(-7)


@pytest.mark.parametrize("M,N,K", [(8, 96, 512), (300, 264, 1024)])
def test_linear_activations_written_just_before(lib, dev, oracle_mod, M, N, K):
    X = (np.random.default_rng(M + K).standard_normal((M, K)) * 2.0).astype(np.float32)
    W = synthetic.normal_i8(11, 1, (N, K), 40.0)
    ew = synthetic.uniform_i32(11, 3, (N,), -14, -6)
    Q, ea = oracle_mod.quantize_pow2(X, 0)
    want = oracle_mod.w8a8(Q, W, ea, ew)
    tX, produce = _produced(to_dev(X, dev), 1.0e30)
    tW, tew = to_dev(W, dev), to_dev(ew, dev)
    torch.cuda.synchronize()
    torch.cuda._sleep(SPIN_CYCLES)
    produce()
    C = lib.linear_w8a8(tX, tW, tew)
    assert (bf16_bits(C.clone()) == want).all()


def test_ozaki_operands_written_just_before(lib, dev, oracle_mod):
    rng = np.random.default_rng(5)
    A = (rng.standard_normal((130, 300)) * np.exp2(rng.integers(-8, 9, size=(130, 300)))).astype(np.float32)
    B = (rng.standard_normal((300, 96)) * np.exp2(rng.integers(-8, 9, size=(300, 96)))).astype(np.float32)
    want = oracle_mod.ozaki_f32(A, B, 7, 8).view(np.uint32)
    (tA, pa), (tB, pb) = _produced(to_dev(A, dev), 3.0), _produced(to_dev(B, dev), -2.0)
    torch.cuda.synchronize()
    torch.cuda._sleep(SPIN_CYCLES)
    pa()
    pb()
    C = lib.ozaki_f32(tA, tB)
    assert (f32_bits(C.clone()) == want).all()
