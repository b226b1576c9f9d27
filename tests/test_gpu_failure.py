"""Failure detection without a GPU fault: a bounded device-side wait that expires is
reported through the status word and leaves the context usable."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import bf16_bits, cuda, dg, to_dev

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives(oracle_mod):
    dev = cuda()
    lib = dg()
    assert lib.device_status() == lib.OK
    lib.selftest_timeout(50)  # a wait on a barrier nothing arrives on, limited to 50 ms
    assert lib.device_status() == lib.ERR_TIMEOUT
    assert lib.device_status() == lib.OK  # cleared by the read
    A, W, ea, ew = synthetic.tiny()
    A = np.concatenate([A, A])  # M = 128: the tensor-core engine
    ea = np.concatenate([ea, ea])
    C = lib.w8a8(to_dev(A, dev), to_dev(W, dev), to_dev(ea, dev), to_dev(ew, dev))
    assert (bf16_bits(C) == oracle_mod.w8a8(A, W, ea, ew)).all()
    assert lib.device_status() == lib.OK


def test_selftest_limit_validated():
    cuda()
    lib = dg()
    with pytest.raises(lib.DetGemmError):
        lib.selftest_timeout(0)
    with pytest.raises(lib.DetGemmError):
        lib.selftest_timeout(5000)
