"""GPU parity of detgemm_w8a8_host (operands in host memory; copies, computation and copy
back pipelined over chunks of rows) against detgemm_w8a8 on device operands and the CPU
oracle, bit for bit: the decode-shaped and tensor-core paths, one and several chunks, a
ragged last chunk, host row strides wider than K, pageable and pinned memory."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import bf16_bits, cuda, dg, padded, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda()


@pytest.fixture(scope="module")
def lib():
    return dg()


def _host(a, pinned, ld=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if ld is not None and ld != a.shape[1]:
        buf = torch.zeros((a.shape[0], ld), dtype=t.dtype)
        buf[:, :a.shape[1]] = t
        t = buf[:, :a.shape[1]]
    return t.pin_memory() if pinned and ld is None else t


@pytest.mark.parametrize("M,N,K,pinned,ld", [
    (16, 300, 1000, True, None), (64, 256, 4096, False, None), (65, 130, 700, True, None),
    (1000, 520, 2048, True, None), (2304, 768, 1024, False, 1040), (8192, 1024, 4096, True, None)])
def test_host_matches_device_and_oracle(lib, dev, oracle_mod, M, N, K, pinned, ld):
    A, W, ea, ew = synthetic.w8a8_normal(31 + M, M, N, K, 25.0, 35.0, -14, -6)
    C = lib.w8a8_host(_host(A, pinned, ld), _host(W, pinned), _host(ea, pinned), _host(ew, pinned))
    got = C.view(torch.int16).numpy().view(np.uint16)
    k16 = (K + 15) // 16 * 16
    Cd = lib.w8a8(padded(A, dev, k16), padded(W, dev, k16), to_dev(ea, dev), to_dev(ew, dev))
    assert (got == bf16_bits(Cd)).all()
    rows = sorted({0, M // 2, M - 1})
    assert (got[rows] == oracle_mod.w8a8(A, W, ea, ew, rows=rows)).all()


def test_host_async_then_sync(lib, dev):
    A, W, ea, ew = synthetic.w8a8_normal(7, 600, 300, 512, 25.0, 35.0, -14, -6)
    out = torch.empty((600, 300), dtype=torch.bfloat16).pin_memory()
    out.view(torch.int16).fill_(-1)
    s = torch.cuda.Stream()
    buf = torch.empty(lib.w8a8_host_buffer_size(600, 300, 512), dtype=torch.uint8, device=dev)
    args = [torch.from_numpy(x).pin_memory() for x in (A, W, ea, ew)]
    for _ in range(2):  # the second call reuses the buffer after the first one on the stream
        lib.w8a8_host(*args, out=out, buf=buf, stream=s, sync=False)
    s.synchronize()
    want = lib.w8a8(*(torch.from_numpy(x).to(dev) for x in (A, W, ea, ew)))
    assert (out.view(torch.int16).numpy().view(np.uint16) == bf16_bits(want)).all()


def test_host_two_streams_share_copy_streams(lib, dev):
    """Two independent problems issued on two streams go through the same library copy
    streams and events (re-recorded by the second call); every step's results equal those
    of the calls made one after the other."""
    probs = [synthetic.w8a8_normal(11, 1500, 640, 1024, 25.0, 35.0, -14, -6),
             synthetic.w8a8_normal(12, 700, 256, 2560, 25.0, 35.0, -14, -6)]
    want = [bf16_bits(lib.w8a8(*(torch.from_numpy(x).to(dev) for x in p))) for p in probs]
    hosts = [[torch.from_numpy(x).pin_memory() for x in p] for p in probs]
    outs = [torch.empty((p[0].shape[0], p[1].shape[0]), dtype=torch.bfloat16).pin_memory() for p in probs]
    bufs = [torch.empty(lib.w8a8_host_buffer_size(p[0].shape[0], p[1].shape[0], p[0].shape[1]),
                        dtype=torch.uint8, device=dev) for p in probs]
    main = torch.cuda.current_stream()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for step in range(3):
        for o in outs:
            o.view(torch.int16).fill_(-1)
        for s in streams:
            s.wait_stream(main)
        for h, o, b, s in zip(hosts, outs, bufs, streams):
            lib.w8a8_host(*h, out=o, buf=b, stream=s, sync=False)
        for s in streams:
            main.wait_stream(s)
        main.synchronize()
        for o, w in zip(outs, want):
            assert (o.view(torch.int16).numpy().view(np.uint16) == w).all(), step
