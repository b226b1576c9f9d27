"""The library's calls captured in a CUDA graph and replayed: the tensor-core W8A8 path, the
decode-shaped path (its programmatic-dependent-launch chain), split-K, the fused linear layer
and the Ozaki GEMMs give the same bits on replay as direct calls, replay after replay.
Buffers (outputs and workspaces) are allocated before the capture; the library allocates
nothing during it."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import cuda, dg, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda()


@pytest.fixture(scope="module")
def lib():
    return dg()


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32) if t.dtype == torch.float32 \
        else t.view(torch.int64)


def _check_graph(fn, outs):
    """fn() writes into the tensors of outs; compare direct results with graph replays."""
    fn()
    torch.cuda.synchronize()
    want = [_bits(o).clone() for o in outs]
    for o in outs:
        _bits(o).fill_(-1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.synchronize()
    for _ in range(3):
        for o in outs:
            _bits(o).fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        for w, o in zip(want, outs):
            assert torch.equal(w, _bits(o))


def test_graph_w8a8_paths(lib, dev):
    outs, calls = [], []
    for (M, N, K, split) in [(16, 4096, 8192, 1), (300, 768, 1024, 1), (512, 512, 2048, 3)]:
        A, W, ea, ew = (to_dev(x, dev) for x in synthetic.w8a8_normal(60 + M, M, N, K, 25.0, 35.0, -14, -6))
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(lib.w8a8_workspace_size(M, N, K, split), 1), dtype=torch.uint8, device=dev)
        outs.append(C)
        calls.append((A, W, ea, ew, split, C, ws))

    def fn():
        for (A, W, ea, ew, split, C, ws) in calls:
            lib.w8a8(A, W, ea, ew, split_k=split, out=C, ws=ws)
    _check_graph(fn, outs)


def test_graph_linear_and_ozaki(lib, dev):
    X = synthetic.normal_f32(8, 0, (256, 512), 2.0)
    tX = to_dev(X, dev)
    W = to_dev(synthetic.normal_i8(8, 1, (384, 512), 30.0), dev)
    ew = to_dev(synthetic.uniform_i32(8, 3, (384,), -14, -6), dev)
    Y = torch.empty((256, 384), dtype=torch.bfloat16, device=dev)
    wsl = torch.empty(lib.load().detgemm_linear_w8a8_workspace_size(256, 384, 512, 1, 0), dtype=torch.uint8,
                      device=dev)
    Af, Bf = (to_dev(x, dev) for x in synthetic.ozaki(256))
    Cf = torch.empty((256, 256), dtype=torch.float32, device=dev)
    wso = torch.empty(lib.ozaki_workspace_size(256, 256, 256), dtype=torch.uint8, device=dev)
    Ad, Bd = (to_dev(x, dev) for x in synthetic.ozaki_f64(256))
    Cd = torch.empty((256, 256), dtype=torch.float64, device=dev)
    wsd = torch.empty(lib.ozaki_f64_workspace_size(256, 256, 256), dtype=torch.uint8, device=dev)

    def fn():
        lib.linear_w8a8(tX, W, ew, out=Y, ws=wsl)
        lib.ozaki_f32(Af, Bf, out=Cf, ws=wso)
        lib.ozaki_f64(Ad, Bd, out=Cd, ws=wsd)
    _check_graph(fn, [Y, Cf, Cd])
