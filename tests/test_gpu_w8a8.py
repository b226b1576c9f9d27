"""GPU parity of the W8A8 GEMM and its exact int32 accumulator against the CPU oracle.

Every comparison is bit-exact (uint16 bf16 patterns / int32 values). Inputs come
from the seeded generators of the workloads (tiny, sweep, ffn, skinny), plus ragged
shapes, tail sentinels, the all-ones probe and the worst-case magnitude bound.
"""
import os

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


def run_w8a8(lib, dev, A, W, ea, ew, split=1, lda=None, ldw=None):
    M, K = A.shape
    N = W.shape[0]
    tA = padded(A, dev, lda) if lda else to_dev(A, dev)
    tW = padded(W, dev, ldw) if ldw else to_dev(W, dev)
    out = poison_like((M, N), torch.bfloat16, dev)
    lib.w8a8(tA, tW, to_dev(ea, dev), to_dev(ew, dev), split_k=split, out=out)
    return bf16_bits(out)


def run_i32(lib, dev, A, W, split=1, lda=None, ldw=None):
    M, K = A.shape
    N = W.shape[0]
    tA = padded(A, dev, lda) if lda else to_dev(A, dev)
    tW = padded(W, dev, ldw) if ldw else to_dev(W, dev)
    out = poison_like((M, N), torch.int32, dev)
    lib.gemm_s8_i32(tA, tW, split_k=split, out=out)
    return out.cpu().numpy()


def test_tiny_workload(lib, dev, oracle_mod):
    A, W, ea, ew = synthetic.tiny()
    want = oracle_mod.w8a8(A, W, ea, ew)
    assert (run_w8a8(lib, dev, A, W, ea, ew) == want).all()
    assert (run_i32(lib, dev, A, W) == oracle_mod.gemm_s8_i32(A, W)).all()


@pytest.mark.parametrize("M,N,K,split,lda", [
    (1, 1, 1, 1, 16), (7, 13, 33, 1, 48), (16, 200, 100, 2, 112), (33, 257, 1000, 3, 1008),
    (64, 130, 1001, 5, 1008), (65, 129, 64, 1, 64), (129, 131, 1000, 1, 1008),
    (200, 300, 4100, 7, 4112), (257, 64, 130, 3, 144), (300, 17, 3, 1, 16)])
def test_ragged_shapes(lib, dev, oracle_mod, M, N, K, split, lda):
    rng = np.random.default_rng(M * 1000 + N + K)
    A = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    W = rng.integers(-128, 128, size=(N, K), dtype=np.int8)
    ea = rng.integers(-20, -2, size=M, dtype=np.int32)
    ew = rng.integers(-20, -2, size=N, dtype=np.int32)
    got = run_w8a8(lib, dev, A, W, ea, ew, split=split, lda=lda, ldw=lda)
    assert (got == oracle_mod.w8a8(A, W, ea, ew)).all()
    got = run_i32(lib, dev, A, W, split=split, lda=lda, ldw=lda)
    assert (got == oracle_mod.gemm_s8_i32(A, W)).all()


def _bytes(out):
    return bf16_bits(out).tobytes()


def test_sweep_workload_rows_identical_across_M_and_real_cuts(lib, dev, oracle_mod):
    """Each row's bits are the oracle's at every M, with split_k honoured exactly: the
    split-exact entry runs 1, 2, 4 and 8 contiguous K parts (it reports how many), on the
    engine for M = 257 and 2048 and on the decode kernels' split form for M <= 64; the
    plain call (its own cut) is compared too."""
    A, W, ea, ew = synthetic.sweep(2048)
    want = oracle_mod.w8a8(A, W, ea, ew)
    tW = to_dev(W, dev)
    tew = to_dev(ew, dev)
    for M in (1, 7, 64, 257, 2048):
        tA = to_dev(A[:M], dev)
        tea = to_dev(ea[:M], dev)
        out = poison_like((M, 6144), torch.bfloat16, dev)
        lib.w8a8(tA, tW, tea, tew, split_k=1, out=out)
        ref = _bytes(out)
        assert (bf16_bits(out) == want[:M]).all(), M
        for parts in (1, 2, 4, 8):
            out = poison_like((M, 6144), torch.bfloat16, dev)
            _, run = lib.w8a8_split_exact(tA, tW, tea, tew, split_k=parts, out=out)
            assert run == parts, (M, parts, run)
            got = bf16_bits(out)
            assert (got == want[:M]).all(), (M, parts, int((got != want[:M]).sum()))
            assert _bytes(out) == ref, (M, parts)


def test_skinny_workload_deep_split_real_cuts(lib, dev, oracle_mod):
    """M = 16, K = 65536: 8, 16 and 32 contiguous K parts per 128-row block of W (reported
    by the call), each bit-exact against the oracle and byte-identical to the others and to
    the plain call's own cut."""
    A, W, ea, ew = synthetic.skinny()
    want = oracle_mod.w8a8(A, W, ea, ew)
    tA, tW, tea, tew = (to_dev(x, dev) for x in (A, W, ea, ew))
    out = poison_like((16, 4096), torch.bfloat16, dev)
    lib.w8a8(tA, tW, tea, tew, split_k=8, out=out)
    assert (bf16_bits(out) == want).all()
    ref = _bytes(out)
    for parts in (8, 16, 32):
        out = poison_like((16, 4096), torch.bfloat16, dev)
        _, run = lib.w8a8_split_exact(tA, tW, tea, tew, split_k=parts, out=out)
        assert run == parts
        assert (bf16_bits(out) == want).all(), parts
        assert _bytes(out) == ref, parts


def test_split_exact_reports_the_cut(lib, dev, oracle_mod):
    """Ragged shapes through the split-exact entry: the parts run are split_k on the engine
    and min(split_k, ceil(K / 128)) on the decode kernels, and the bits are the oracle's."""
    for M, N, K, split, want_parts in [(65, 300, 1000, 15, 15), (300, 17, 130, 3, 3), (16, 200, 300, 5, 3),
                                       (64, 129, 4100, 33, 33), (1, 1, 1, 1, 1), (3, 40, 4097, 2, 2)]:
        rng = np.random.default_rng(M * 7 + N + K)
        A = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
        W = rng.integers(-128, 128, size=(N, K), dtype=np.int8)
        ea = rng.integers(-20, -2, size=M, dtype=np.int32)
        ew = rng.integers(-20, -2, size=N, dtype=np.int32)
        ld = (K + 15) // 16 * 16
        out = poison_like((M, N), torch.bfloat16, dev)
        _, run = lib.w8a8_split_exact(padded(A, dev, ld), padded(W, dev, ld), to_dev(ea, dev), to_dev(ew, dev),
                                      split_k=split, out=out)
        assert run == want_parts, (M, N, K, split, run)
        assert (bf16_bits(out) == oracle_mod.w8a8(A, W, ea, ew)).all(), (M, N, K, split)


def _tile_columns(N, seed):
    """One column at a random offset inside every 256-wide tile column, plus the edges."""
    rng = np.random.default_rng(seed)
    cols = {0, 1, 127, 128, 255, N - 256, N - 129, N - 1}
    for t in range((N + 255) // 256):
        cols.add(min(N - 1, 256 * t + int(rng.integers(0, 256))))
    return sorted(cols)


@pytest.mark.parametrize("which", ["gate_up", "down"])
def test_ffn_workload_sampled_rows_and_all_rows_of_sampled_columns(lib, dev, oracle_mod, which):
    """8192-row FFN GEMMs: sixteen whole rows, and every row of one column per 256-wide tile
    column (so every tile row, TMEM lane and epilogue warp of the persistent raster)."""
    A, W, ea, ew = synthetic.ffn_gate_up() if which == "gate_up" else synthetic.ffn_down()
    M = A.shape[0]
    out = poison_like((M, W.shape[0]), torch.bfloat16, dev)
    lib.w8a8(to_dev(A, dev), to_dev(W, dev), to_dev(ea, dev), to_dev(ew, dev), out=out)
    rows = sorted({0, 1, 127, 128, 129, 4095, 4096, M - 129, M - 128, M - 1} |
                  set(np.random.default_rng(5).integers(0, M, 6).tolist()))
    got = bf16_bits(out)
    assert (got[rows] == oracle_mod.w8a8(A, W, ea, ew, rows=rows)).all()
    cols = _tile_columns(W.shape[0], 6 if which == "gate_up" else 7)
    want = oracle_mod.w8a8(A, np.ascontiguousarray(W[cols]), ea, np.ascontiguousarray(ew[cols]))
    assert (got[:, cols] == want).all(), int((got[:, cols] != want).sum())


def test_all_ones_probe(lib, dev):
    # all-ones operands: every accumulator equals K exactly (8648, not 8640)
    M, N, K = 4, 8, 8648
    A = np.ones((M, K), np.int8)
    W = np.ones((N, K), np.int8)
    for split in (1, 3, 8):
        assert (run_i32(lib, dev, A, W, split=split, lda=8656, ldw=8656) == 8648).all()
        got = run_w8a8(lib, dev, A, W, np.zeros(M, np.int32), np.zeros(N, np.int32), split=split,
                       lda=8656, ldw=8656)
        assert (got == 0x4607).all()


def test_tail_sentinel_walk(lib, dev):
    # one nonzero per row at k*, walked over block, split and tail boundaries
    K = 1000
    ks = [0, 1, 15, 16, 63, 64, 127, 128, 333, 500, 511, 512, 959, 960, 975, 976, 991, 992, 998, 999]
    A = np.zeros((len(ks), K), np.int8)
    for i, k in enumerate(ks):
        A[i, k] = (i % 120) + 3
    W = np.ones((24, K), np.int8)
    W[5] = -1
    for split in (1, 2, 5, 16):
        C = run_i32(lib, dev, A, W, split=split, lda=1008, ldw=1008)
        want = np.outer(np.arange(len(ks)) % 120 + 3, np.where(np.arange(24) == 5, -1, 1))
        assert (C == want).all(), split


def test_worst_case_magnitude_bound(lib, dev):
    # K = 131071 is the largest K with K * 128^2 < 2^31; all -128 operands
    K = 131071
    A = np.full((2, K), -128, np.int8)
    W = np.full((3, K), -128, np.int8)
    for split in (1, 7, 64):
        C = run_i32(lib, dev, A, W, split=split, lda=131072, ldw=131072)
        assert (C == K * 16384).all()
    A[1] = 127
    C = run_i32(lib, dev, A, W, split=3, lda=131072, ldw=131072)
    assert (C[1] == -K * 127 * 128).all()


def _row_for_acc(acc, K):
    """int8 rows (a, w) of length K with sum a*w == acc (|acc| <= K * 16256)."""
    a = np.zeros(K, np.int8)
    w = np.zeros(K, np.int8)
    s = 1 if acc >= 0 else -1
    big = 16384 if s > 0 else 16256  # (-128)(-128) or (-128)(127)
    q, r = divmod(abs(acc), big)
    a[:q] = -128
    w[:q] = -128 if s > 0 else 127
    i = q
    while r > 0:
        d = min(r, 127)
        a[i], w[i] = d, s
        r -= d
        i += 1
    return a, w


def test_golden_epilogue_cases(lib, dev):
    path = os.path.join(os.path.dirname(__file__), "golden", "w8a8_epilogue_cases.txt")
    rows = []
    for line in open(path):
        line = line.split("#")[0].strip()
        if line:
            acc, e, bits = line.split()[:3]
            rows.append((int(acc), int(e), int(bits, 16)))
    K = 2048
    rows = [r for r in rows if abs(r[0]) <= K * 16384]  # accumulators reachable at this K
    assert len(rows) >= 14
    A = np.zeros((len(rows), K), np.int8)
    W = np.zeros((len(rows), K), np.int8)
    for i, (acc, e, _) in enumerate(rows):
        A[i], W[i] = _row_for_acc(acc, K)
    ea = np.array([e for _, e, _ in rows], np.int32)
    C = run_w8a8(lib, dev, A, W, ea, np.zeros(len(rows), np.int32))
    got = np.diag(C)
    want = np.array([b for _, _, b in rows], np.uint16)
    assert (got == want).all(), [(r, hex(g)) for r, g in zip(rows, got) if g != r[2]]
    # the exponent may sit on either operand (only ea_i + ew_j matters)
    C2 = run_w8a8(lib, dev, A, W, np.zeros(len(rows), np.int32), ea)
    assert (np.diag(C2) == want).all()


def test_rows_independent_of_M_and_repeatable(lib, dev, oracle_mod):
    rng = np.random.default_rng(9)
    A = rng.integers(-128, 128, size=(300, 512), dtype=np.int8)
    W = rng.integers(-128, 128, size=(192, 512), dtype=np.int8)
    ea = rng.integers(-14, -6, size=300, dtype=np.int32)
    ew = rng.integers(-14, -6, size=192, dtype=np.int32)
    full = run_w8a8(lib, dev, A, W, ea, ew)
    for M in (1, 2, 17, 64, 65, 128, 299):
        for split in (1, 4):
            assert (run_w8a8(lib, dev, A[:M], W, ea[:M], ew, split=split) == full[:M]).all()
    assert (run_w8a8(lib, dev, A, W, ea, ew) == full).all()


def test_tc_engine_chunk_boundary_worst_case(lib, dev):
    # all -128 operands: every 1024-long fp32 chunk reaches exactly 2^24 on the
    # tensor-core path (M > 64), the largest value the chunked accumulation must hold
    for M, N, K, split in [(130, 260, 16384, 1), (65, 8, 131071, 1), (200, 300, 131071, 7)]:
        A = np.full((M, K), -128, np.int8)
        W = np.full((N, K), -128, np.int8)
        ld = (K + 15) // 16 * 16
        C = run_i32(lib, dev, A, W, split=split, lda=ld, ldw=ld)
        assert (C == K * 16384).all(), (M, N, K, split)


def test_tc_epilogue_large_accumulators(lib, dev, oracle_mod):
    # accumulators of 26-28 bits (well past fp32's 24-bit significand) with random low
    # bits: the tensor-core epilogue's rounding must still match the oracle bit for bit
    rng = np.random.default_rng(21)
    M, N, K = 130, 257, 10000
    A = rng.integers(90, 128, size=(M, K), dtype=np.int8)
    W = rng.integers(90, 128, size=(N, K), dtype=np.int8)
    A[::3] = -A[::3]
    ea = rng.integers(-40, -10, size=M, dtype=np.int32)
    ew = rng.integers(-40, -10, size=N, dtype=np.int32)
    acc = oracle_mod.gemm_s8_i32(A, W)
    assert np.abs(acc).max() > 2 ** 26
    got = run_w8a8(lib, dev, A, W, ea, ew, lda=10000, ldw=10000)
    assert (got == oracle_mod.w8a8(A, W, ea, ew)).all()


def test_tc_epilogue_extreme_exponents(lib, dev, oracle_mod):
    # exponents that push results into bf16 subnormals, to zero, near the largest finite
    # value and to infinity, mixed within warps, on the tensor-core path (M > 64)
    rng = np.random.default_rng(22)
    M, N, K = 200, 300, 700
    A = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    W = rng.integers(-128, 128, size=(N, K), dtype=np.int8)
    ea = rng.integers(-160, 130, size=M, dtype=np.int32)
    ew = rng.integers(-40, 40, size=N, dtype=np.int32)
    ea[:40] = rng.integers(-20, 0, size=40)  # some rows entirely in the common range
    got = run_w8a8(lib, dev, A, W, ea, ew, lda=704, ldw=704)
    want = oracle_mod.w8a8(A, W, ea, ew)
    assert (got == want).all(), int((got != want).sum())
    # golden cases on the tensor-core path: rows of the hand-worked table, repeated to M > 64
    path = os.path.join(os.path.dirname(__file__), "golden", "w8a8_epilogue_cases.txt")
    cases = []
    for line in open(path):
        line = line.split("#")[0].strip()
        if line:
            a, e, b = line.split()[:3]
            cases.append((int(a), int(e), int(b, 16)))
    cases = [c for c in cases if abs(c[0]) <= 2048 * 16256]
    rows = (cases * 10)[:130]
    A = np.zeros((len(rows), 2048), np.int8)
    W = np.zeros((len(rows), 2048), np.int8)
    for i, (acc, e, _) in enumerate(rows):
        A[i], W[i] = _row_for_acc(acc, 2048)
    C = run_w8a8(lib, dev, A, W, np.array([e for _, e, _ in rows], np.int32), np.zeros(len(rows), np.int32))
    assert (np.diag(C) == np.array([b for _, _, b in rows], np.uint16)).all()


@pytest.mark.parametrize("M,N,K,split", [(300, 520, 1000, 1), (64, 256, 2048, 4), (1000, 130, 70, 1)])
def test_prewidened_operands_give_the_same_bits(lib, dev, M, N, K, split):
    rng = np.random.default_rng(M + N + K)
    A = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    W = rng.integers(-128, 128, size=(N, K), dtype=np.int8)
    ea = rng.integers(-20, -2, size=M, dtype=np.int32)
    ew = rng.integers(-20, -2, size=N, dtype=np.int32)
    ld = (K + 15) // 16 * 16
    tA, tW = padded(A, dev, ld), padded(W, dev, ld)
    A16, W16 = lib.widen_i8_f16(tA), lib.widen_i8_f16(tW)
    assert torch.equal(A16.float().cpu(), torch.from_numpy(A).float())
    ref = lib.w8a8(tA, tW, to_dev(ea, dev), to_dev(ew, dev), split_k=split)
    got = lib.w8a8_f16ops(A16, W16, to_dev(ea, dev), to_dev(ew, dev), split_k=split)
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("rows,cols", [(3, 256), (3, 250), (5, 200), (2, 33), (7, 1)])
def test_widening_is_exact_and_zero_pads(lib, dev, rows, cols):
    # every int8 value appears; the row stride (cols rounded up to 8 halves) is either a
    # multiple of 16 (two-operand kernel) or only of 8 (the narrow kernel)
    X = ((np.arange(rows * cols, dtype=np.int64) * 37 + 11) % 256 - 128).astype(np.int8).reshape(rows, cols)
    tX = padded(X, dev, (cols + 15) // 16 * 16)
    Y = lib.widen_i8_f16(tX)
    assert torch.equal(Y.float().cpu(), torch.from_numpy(X).float())
    full = torch.as_strided(Y, (rows, Y.stride(0)), (Y.stride(0), 1))
    assert (full[:, cols:].float().cpu() == 0).all()
    assert (full.view(torch.int16)[:, cols:].cpu() == 0).all()  # +0, not -0


def test_skinny_many_ctas_repeated(lib, dev, oracle_mod):
    # many co-resident CTAs streaming W through the shared-memory ring: repeated runs at
    # deep splits must all be exact (guards the stage-release ordering under load)
    A, W, ea, ew = synthetic.skinny()
    want = oracle_mod.gemm_s8_i32(A, W)
    tA, tW = to_dev(A, dev), to_dev(W, dev)
    for split in (16, 32, 64, 64, 128):
        out = poison_like((16, 4096), torch.int32, dev)
        lib.gemm_s8_i32(tA, tW, split_k=split, out=out)
        assert (out.cpu().numpy() == want).all(), split


@pytest.mark.parametrize("M,N,K", [(64, 40, 4096), (17, 100, 4096), (1, 33, 4097), (48, 70, 3969), (64, 96, 5000),
                                   (65, 100, 2048), (128, 64, 4096), (100, 33, 1000), (128, 70, 4097),
                                   (16, 100, 4096), (1, 40, 4096), (5, 77, 384), (16, 130, 640), (9, 65, 128)])
def test_decode_short_and_long_k(lib, dev, oracle_mod, M, N, K):
    # up to K = 4096 the decode path (M <= 64) keeps whole rows of W per CTA (each warp's fp32
    # partials hold at most 1024 products); longer K splits K over the SMs; M > 64 runs on
    # the tensor cores. Worst case first: every product 128^2, so each warp's partial sums
    # reach 2^24 exactly.
    ld = (K + 15) // 16 * 16
    A = np.full((M, K), -128, np.int8)
    W = np.full((N, K), -128, np.int8)
    assert (run_i32(lib, dev, A, W, lda=ld, ldw=ld) == K * 16384).all()
    rng = np.random.default_rng(M * 7 + N + K)
    A = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    W = rng.integers(-128, 128, size=(N, K), dtype=np.int8)
    ea = rng.integers(-24, -2, size=M, dtype=np.int32)
    ew = rng.integers(-24, -2, size=N, dtype=np.int32)
    assert (run_w8a8(lib, dev, A, W, ea, ew, lda=ld, ldw=ld) == oracle_mod.w8a8(A, W, ea, ew)).all()
    assert (run_i32(lib, dev, A, W, lda=ld, ldw=ld) == oracle_mod.gemm_s8_i32(A, W)).all()


@pytest.mark.parametrize("M,N,K", [(8192, 4096, 1024), (2048, 6144, 2048), (4096, 4096, 4096), (3000, 2056, 1008)])
def test_epilogue_geometries_agree(lib, dev, oracle_mod, M, N, K):
    # the launcher picks sixteen epilogue warps for short K or few rounds (the first two
    # shapes, and the ragged last one) and eight otherwise (the third); every geometry gives
    # the oracle's bits on sampled rows, and rows computed alone (decode path or one-round
    # tiles) agree with them
    rng = np.random.default_rng(M + N + K)
    A = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    W = rng.integers(-128, 128, size=(N, K), dtype=np.int8)
    ea = rng.integers(-20, -4, size=M, dtype=np.int32)
    ew = rng.integers(-20, -4, size=N, dtype=np.int32)
    tW, tew = to_dev(W, dev), to_dev(ew, dev)
    out = poison_like((M, N), torch.bfloat16, dev)
    lib.w8a8(to_dev(A, dev), tW, to_dev(ea, dev), tew, out=out)
    full = bf16_bits(out)
    rows = sorted({0, 31, 32, 255, 256, M // 2, M - 1} | set(rng.integers(0, M, 5).tolist()))
    assert (full[rows] == oracle_mod.w8a8(A, W, ea, ew, rows=rows)).all()
    few = rows[:3]
    part = lib.w8a8(to_dev(A[few], dev), tW, to_dev(ea[few], dev), tew)
    assert (bf16_bits(part) == full[few]).all()
