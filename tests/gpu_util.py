"""Helpers shared by the GPU parity tests (no arithmetic of the method here)."""
import numpy as np
import pytest
import torch


def cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return torch.device("cuda:0")


def dg():
    """The product binding; the library must be built (a missing .so fails loudly)."""
    import deterministic_detgemm_w8a8_gb300 as m
    from deterministic_detgemm_w8a8_gb300 import build as b
    b.build()
    m.load()
    return m


def to_dev(a: np.ndarray, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def padded(a: np.ndarray, dev, ld: int):
    """2-D device tensor view [rows, cols] with row stride ld (>= cols); padding poisoned."""
    rows, cols = a.shape
    dtype = torch.from_numpy(a[:0]).dtype
    buf = torch.full((rows, ld), 0x5A if a.dtype == np.int8 else 0, dtype=dtype, device=dev)
    buf[:, :cols] = to_dev(a, dev)
    return buf[:, :cols]


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def f32_bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


def poison_like(shape, dtype, dev):
    """Output buffer (16-byte aligned row stride) filled with 0xFF bytes."""
    rows, cols = shape
    esize = torch.empty((), dtype=dtype).element_size()
    per = 16 // esize
    ld = max(per, (cols + per - 1) // per * per)
    t = torch.empty((rows, ld), dtype=dtype, device=dev)
    t.view(torch.uint8).fill_(0xFF)
    return t[:, :cols]
