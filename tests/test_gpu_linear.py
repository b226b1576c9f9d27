"""GPU parity of the fused W8A8 linear layer (pow2 quantization of bf16/fp32 activations +
the exact W8A8 GEMM) against the oracle's two steps, bit for bit: both the decode-shaped
path (M <= 64) and the tensor-core path, with and without a pre-widened weight, across
split-K counts, ragged K and N, and a sampled check at the 8B-class FFN gate/up size."""
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


def _acts(seed, M, K, dtype):
    X = synthetic.normal_f32(seed, 0, (M, K), 3.0)
    X = X * np.exp2(np.arange(M) % 9 - 4)[:, None].astype(np.float32)  # rows of different scale
    if M > 2:
        X[1] = 0.0  # a zero row: e = 0, Q = 0
    return (_bf16(X), torch.bfloat16) if dtype == "bf16" else (X.astype(np.float32), torch.float32)


def _dev_x(X, tdt, dev, ld):
    if tdt == torch.bfloat16:
        return padded(X.view(np.int16), dev, ld).view(torch.bfloat16)
    return padded(X, dev, ld)


@pytest.mark.parametrize("M,N,K,split,dtype,mode,w16", [
    (1, 96, 512, 1, "bf16", 0, False),
    (7, 200, 1000, 2, "f32", 1, False),
    (64, 256, 4096, 4, "bf16", 0, False),
    (65, 130, 1000, 1, "bf16", 0, False),
    (100, 200, 2048, 1, "bf16", 0, True),
    (128, 96, 4096, 2, "f32", 1, False),
    (257, 300, 2048, 2, "f32", 0, True),
    (300, 256, 777, 1, "bf16", 1, True),
    (512, 512, 4096, 3, "bf16", 0, False),
])
def test_linear_matches_quantize_then_w8a8(lib, dev, oracle_mod, M, N, K, split, dtype, mode, w16):
    X, tdt = _acts(M * 31 + K, M, K, dtype)
    W = synthetic.normal_i8(9, 1, (N, K), 40.0)
    ew = synthetic.uniform_i32(9, 3, (N,), -14, -6)
    Qw, eaw = oracle_mod.quantize_pow2(X, mode)
    want = oracle_mod.w8a8(Qw, W, eaw, ew)
    ldx = (K + 15) // 16 * 16
    tX = _dev_x(X, tdt, dev, ldx)
    tW = padded(W, dev, (K + 15) // 16 * 16)
    tW16 = lib.widen_i8_f16(tW) if w16 else None
    out = poison_like((M, N), torch.bfloat16, dev)
    ea = torch.full((M,), 12345, dtype=torch.int32, device=dev)
    lib.linear_w8a8(tX, tW, to_dev(ew, dev), mode=mode, W16=tW16, split_k=split, out=out, ea_out=ea)
    assert (ea.cpu().numpy() == eaw).all()
    got = bf16_bits(out)
    assert (got == want).all(), int((got != want).sum())
    assert lib.device_status() == lib.OK


def test_linear_nonfinite_row_reported(lib, dev, oracle_mod):
    X = synthetic.normal_f32(3, 0, (80, 256), 1.0)
    X[5, 17] = np.inf
    W = synthetic.normal_i8(3, 1, (64, 256), 40.0)
    ew = np.zeros(64, np.int32)
    out = lib.linear_w8a8(to_dev(X, dev), to_dev(W, dev), to_dev(ew, dev))
    assert lib.device_status() == lib.ERR_NONFINITE
    got = bf16_bits(out)
    assert (got[5] == 0).all()  # the non-finite row is quantized to zero
    Qw, eaw = oracle_mod.quantize_pow2(np.delete(X, 5, axis=0), 0)
    want = oracle_mod.w8a8(Qw, W, eaw, ew)
    assert (np.delete(got, 5, axis=0) == want).all()


def test_linear_ffn_gate_up_sampled(lib, dev, oracle_mod):
    """8B-class FFN gate/up size (M=8192, K=4096, N=12288) on bf16 activations: sampled
    rows bit-exact against the oracle; identical bits with a pre-widened weight and at
    split-K 2."""
    M, K, N = 8192, 4096, 12288
    X = _bf16(synthetic.normal_f32(21, 0, (M, K), 2.0))
    W = synthetic.normal_i8(2, 1, (N, K), 30.0)
    ew = synthetic.uniform_i32(2, 3, (N,), -14, -6)
    tX = to_dev(X.view(np.int16), dev).view(torch.bfloat16)
    tW, tew = to_dev(W, dev), to_dev(ew, dev)
    ea = torch.empty((M,), dtype=torch.int32, device=dev)
    out = lib.linear_w8a8(tX, tW, tew, ea_out=ea)
    rows = [0, 1, 255, 256, 4097, 8191]
    Qw, eaw = oracle_mod.quantize_pow2(X[rows], 0)
    want = oracle_mod.w8a8(Qw, W, eaw, ew)
    assert (bf16_bits(out)[rows] == want).all()
    assert (ea.cpu().numpy()[rows] == eaw).all()
    out2 = lib.linear_w8a8(tX, tW, tew, W16=lib.widen_i8_f16(tW), split_k=2)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
