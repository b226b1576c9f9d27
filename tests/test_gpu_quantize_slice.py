"""GPU parity of the pow2 quantizer and the Ozaki slicer against the CPU oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import cuda, dg, padded, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda()


@pytest.fixture(scope="module")
def lib():
    return dg()


def _special_rows(cols, rng):
    X = (rng.standard_normal((12, cols)) * np.exp2(rng.integers(-30, 30, size=(12, 1)))).astype(np.float32)
    X[0] = 0.0                                      # zero row
    X[1] = np.float32(2.0 ** -149) * rng.integers(-5, 6, size=cols)  # subnormals only
    X[2, :] = 1.0
    X[2, 0] = 127.0 * 2.0 ** 0.5                    # nearest/ceil boundary region
    X[3] = rng.integers(-127, 128, size=cols) * np.float32(2.0 ** -7)  # already quantized
    X[4] = (rng.standard_normal(cols) * 3.0e37).astype(np.float32)   # near the top of the range
    X[5, ::2] = 0.5
    X[5, 1::2] = -0.25                              # ties after scaling
    return X


def _bf16(x: np.ndarray) -> np.ndarray:
    """round-to-nearest-even fp32 -> bf16 bit patterns (input generation only)."""
    b = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("cols,ld", [(4096, 4096), (1000, 1008), (24, 32), (1, 16)])
def test_quantize_fp32(lib, dev, oracle_mod, mode, cols, ld):
    rng = np.random.default_rng(cols + mode)
    X = np.concatenate([_special_rows(cols, rng),
                        synthetic.normal_f32(7, 0, (300, cols), 2.5)]).astype(np.float32)
    Qw, ew = oracle_mod.quantize_pow2(X, mode)
    Q, e = lib.quantize_pow2(padded(X, dev, ld), mode)
    assert (e.cpu().numpy() == ew).all()
    assert (Q.cpu().numpy() == Qw).all()


@pytest.mark.parametrize("mode", [0, 1])
def test_quantize_bf16(lib, dev, oracle_mod, mode):
    rng = np.random.default_rng(40 + mode)
    X = np.concatenate([_special_rows(2048, rng), synthetic.normal_f32(8, 0, (500, 2048), 30.0)])
    Xb = _bf16(X)
    Qw, ew = oracle_mod.quantize_pow2(Xb, mode)
    tX = to_dev(Xb.view(np.int16), dev).view(torch.bfloat16)
    Q, e = lib.quantize_pow2(tX, mode)
    assert (e.cpu().numpy() == ew).all()
    assert (Q.cpu().numpy() == Qw).all()


def test_quantize_nonfinite_reported(lib, dev):
    X = np.ones((3, 64), np.float32)
    X[1, 5] = np.inf
    assert lib.device_status() == lib.OK
    Q, e = lib.quantize_pow2(to_dev(X, dev), 0)
    assert lib.device_status() == lib.ERR_NONFINITE
    assert lib.device_status() == lib.OK  # cleared by the read
    q = Q.cpu().numpy()
    assert (q[1] == 0).all() and (q[0] == q[2]).all() and (q[0] != 0).all()


@pytest.mark.parametrize("nslices", [7, 4, 9])
@pytest.mark.parametrize("rows,cols", [(64, 512), (33, 100), (1, 5), (130, 257)])
def test_slice_rows_and_cols(lib, dev, oracle_mod, nslices, rows, cols):
    rng = np.random.default_rng(rows * cols + nslices)
    X = (rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-8, 9, size=(rows, cols)))).astype(np.float32)
    if rows > 3:
        X[2] = 0.0
        X[3] = np.float32(2.0 ** -149) * rng.integers(-3, 4, size=cols)
    ld = (cols + 3) // 4 * 4
    for axis in (0, 1):
        Sw, ew = oracle_mod.slice_f32(X, axis, nslices)
        S, e = lib.slice_f32(padded(X, dev, ld), axis, nslices)
        assert (e.cpu().numpy() == ew).all(), axis
        assert (S.cpu().numpy() == Sw).all(), axis


def test_slice_ozaki_workload(lib, dev, oracle_mod):
    A, B = synthetic.ozaki(1024)
    for axis, X in ((0, A), (1, B)):
        Sw, ew = oracle_mod.slice_f32(X, axis, 7)
        S, e = lib.slice_f32(to_dev(X, dev), axis, 7)
        assert (e.cpu().numpy() == ew).all()
        assert (S.cpu().numpy() == Sw).all()


def test_slice_nonfinite_reported(lib, dev):
    X = np.ones((4, 32), np.float32)
    X[2, 3] = np.nan
    lib.device_status()
    lib.slice_f32(to_dev(X, dev), 0, 7)
    assert lib.device_status() == lib.ERR_NONFINITE
    lib.slice_f32(to_dev(X, dev), 1, 7)
    assert lib.device_status() == lib.ERR_NONFINITE
