"""GPU parity of the gated-linear-unit epilogue rne_bf16(SiLU(g) * u) with the oracle
(binary128 evaluation, pinned to mpmath), bit for bit: random accumulators over the whole
int32 range and exponent domain, inputs within 2^-20 and 2^-52 of a bf16 rounding boundary
(the float-float, fp64 and double-double evaluations), large gates whose product sits on a midpoint, deep
negative gates, subnormal and overflowing outputs, exponents outside the domain (NaN and
DETGEMM_ERR_RANGE), and the composition with the library's exact int32 GEMM."""
import os

import numpy as np
import pytest
import torch

from gpu_util import bf16_bits, cuda, dg, to_dev

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def dev():
    return cuda()


@pytest.fixture(scope="module")
def lib():
    return dg()


def _run(lib, dev, G, U, ea, ewg, ewu):
    return bf16_bits(lib.swiglu_bf16(to_dev(G, dev), to_dev(U, dev), to_dev(ea, dev), to_dev(ewg, dev),
                                     to_dev(ewu, dev)))


def _want(oracle_mod, G, U, ea, ewg, ewu):
    M, N = G.shape
    return np.array([[oracle_mod.silu_mul_bf16(int(G[i, j]), int(U[i, j]), int(ea[i] + ewg[j]), int(ea[i] + ewu[j]))
                      for j in range(N)] for i in range(M)], np.uint16)


@pytest.mark.parametrize("kind", ["ffn", "full", "large", "deep"])
def test_random_accumulators(lib, dev, oracle_mod, kind):
    rng = np.random.default_rng({"ffn": 1, "full": 2, "large": 3, "deep": 4}[kind])
    M, N = 48, 160
    if kind == "ffn":
        G = rng.integers(-2 ** 22, 2 ** 22, (M, N)); U = rng.integers(-2 ** 22, 2 ** 22, (M, N))
        ea = rng.integers(-12, -6, M); ewg = rng.integers(-12, -6, N); ewu = rng.integers(-12, -6, N)
    elif kind == "full":
        G = rng.integers(-2 ** 31 + 1, 2 ** 31, (M, N)); U = rng.integers(-2 ** 31 + 1, 2 ** 31, (M, N))
        ea = rng.integers(-30, -10, M); ewg = rng.integers(-30, 5, N); ewu = rng.integers(-30, 50, N)
    elif kind == "large":  # gates from ~30 to ~2^40
        G = rng.integers(2 ** 10, 2 ** 31, (M, N)) * rng.choice([-1, 1], (M, N))
        U = rng.integers(-2 ** 16, 2 ** 16, (M, N))
        ea = rng.integers(-5, 0, M); ewg = rng.integers(-25, 10, N); ewu = rng.integers(-20, 0, N)
    else:  # gates around -40 .. -2000: tiny, subnormal and zero outputs
        G = -rng.integers(2 ** 20, 2 ** 30, (M, N)); U = rng.integers(1, 2 ** 31, (M, N))
        ea = rng.integers(-20, -15, M); ewg = rng.integers(-8, 0, N); ewu = rng.integers(15, 55, N)
    G, U = G.astype(np.int32), U.astype(np.int32)
    ea, ewg, ewu = (x.astype(np.int32) for x in (ea, ewg, ewu))
    got = _run(lib, dev, G, U, ea, ewg, ewu)
    want = _want(oracle_mod, G, U, ea, ewg, ewu)
    assert (got == want).all(), int((got != want).sum())
    assert lib.device_status() == lib.OK


def test_inputs_near_rounding_boundaries(lib, dev, oracle_mod):
    rows = [line.split() for line in open(os.path.join(HERE, "golden", "swiglu_hard_inputs.txt"))
            if not line.startswith("#")]
    n = len(rows)
    G = np.array([[int(r[0]) for r in rows]], np.int32)
    U = np.array([[int(r[1]) for r in rows]], np.int32)
    ea = np.zeros(1, np.int32)
    ewg = np.array([int(r[2]) for r in rows], np.int32)
    ewu = np.array([int(r[3]) for r in rows], np.int32)
    got = _run(lib, dev, G, U, ea, ewg, ewu)
    want = _want(oracle_mod, G, U, ea, ewg, ewu)
    assert (got == want).all(), [rows[j] for j in np.nonzero(got[0] != want[0])[0]]
    assert lib.device_status() == lib.OK
    assert sum(r[4] == "fp64-ambiguous" for r in rows) >= 10 and n >= 50


def test_special_values(lib, dev, oracle_mod):
    # large gates with g * u on a midpoint; zero operands; deep negative gates; subnormal and
    # overflowing outputs
    cases = [(128, 259, 0, -7), (128, -259, 0, -7), (96, 1029, 0, -3), (2 ** 20, 513, -10, 0),
             (0, 5, 0, 0), (7, 0, 0, 0), (-1400, 3, -1, 0), (-(2 ** 30), 2 ** 30, -20, 40),
             (-90, 2 ** 30, 0, -40), (-88, 1, 0, 30), (2 ** 30, 2 ** 30, 40, 30), (-(2 ** 30), 2 ** 30, 40, 30),
             (1, 1, 0, 0), (-3, 5, -2, -1), (80, 3, 0, 0), (-80, 3, 0, 0), (64, 129, 0, 0), (63, 129, 0, 0)]
    G = np.array([[c[0] for c in cases]], np.int32)
    U = np.array([[c[1] for c in cases]], np.int32)
    ewg = np.array([c[2] for c in cases], np.int32)
    ewu = np.array([c[3] for c in cases], np.int32)
    ea = np.zeros(1, np.int32)
    got = _run(lib, dev, G, U, ea, ewg, ewu)
    want = _want(oracle_mod, G, U, ea, ewg, ewu)
    assert (got == want).all(), [(cases[j], hex(got[0, j]), hex(want[0, j])) for j in np.nonzero(got[0] != want[0])[0]]
    assert got[0, 0] == 0x4381 and got[0, 10] == 0x7F80


def test_exponents_outside_the_domain(lib, dev):
    G = np.array([[5, 5, 5]], np.int32)
    U = np.array([[3, 3, 3]], np.int32)
    got = _run(lib, dev, G, U, np.zeros(1, np.int32), np.array([41, 0, 0], np.int32), np.array([0, -61, 0], np.int32))
    assert got[0, 0] == 0x7FC0 and got[0, 1] == 0x7FC0 and got[0, 2] != 0x7FC0
    assert lib.device_status() == lib.ERR_RANGE
    assert lib.device_status() == lib.OK  # read and cleared


def test_composition_with_the_int32_gemm(lib, dev, oracle_mod):
    rng = np.random.default_rng(6)
    M, N, K = 96, 320, 1000
    A = np.clip(np.rint(rng.standard_normal((M, K)) * 30), -127, 127).astype(np.int8)
    Wg = np.clip(np.rint(rng.standard_normal((N, K)) * 30), -127, 127).astype(np.int8)
    Wu = np.clip(np.rint(rng.standard_normal((N, K)) * 30), -127, 127).astype(np.int8)
    ea = rng.integers(-14, -6, M).astype(np.int32)
    ewg = rng.integers(-14, -6, N).astype(np.int32)
    ewu = rng.integers(-14, -6, N).astype(np.int32)
    pad = lambda x: torch.nn.functional.pad(torch.from_numpy(x), (0, 8)).to(dev)[:, :K]
    G = lib.gemm_s8_i32(pad(A), pad(Wg))
    U = lib.gemm_s8_i32(pad(A), pad(Wu))
    got = bf16_bits(lib.swiglu_bf16(G, U, to_dev(ea, dev), to_dev(ewg, dev), to_dev(ewu, dev)))
    assert (got == oracle_mod.w8a8_swiglu(A, Wg, Wu, ea, ewg, ewu)).all()


@pytest.mark.parametrize("M,N,K", [(1, 64, 64), (64, 130, 1000), (300, 257, 520), (1024, 512, 4096)])
def test_fused_w8a8_swiglu(lib, dev, oracle_mod, M, N, K):
    rng = np.random.default_rng(M + N + K)
    A = np.clip(np.rint(rng.standard_normal((M, K)) * 30), -127, 127).astype(np.int8)
    Wg = np.clip(np.rint(rng.standard_normal((N, K)) * 30), -127, 127).astype(np.int8)
    Wu = np.clip(np.rint(rng.standard_normal((N, K)) * 30), -127, 127).astype(np.int8)
    ea = rng.integers(-14, -6, M).astype(np.int32)
    ewg = rng.integers(-14, -6, N).astype(np.int32)
    ewu = rng.integers(-14, -6, N).astype(np.int32)
    ld = (K + 15) // 16 * 16
    from gpu_util import padded
    out = lib.w8a8_swiglu(padded(A, dev, ld), padded(Wg, dev, ld), padded(Wu, dev, ld), to_dev(ea, dev),
                          to_dev(ewg, dev), to_dev(ewu, dev))
    got = bf16_bits(out)
    want = oracle_mod.w8a8_swiglu(A, Wg, Wu, ea, ewg, ewu)
    assert (got == want).all(), int((got != want).sum())
    assert lib.device_status() == lib.OK


def test_fused_ffn_gate_up_sampled(lib, dev, oracle_mod):
    # the 8B-class FFN's gate and up projections at 8192 tokens (K = 4096, N = 12288 each):
    # every row of one column per 128-wide output tile column, and sixteen whole rows
    import synthetic
    A, Wg, ea, ewg = synthetic.ffn_gate_up()
    Wu = synthetic.normal_i8(2, 9, Wg.shape, 30.0)
    ewu = synthetic.uniform_i32(2, 10, (Wg.shape[0],), -14, -6)
    got = bf16_bits(lib.w8a8_swiglu(to_dev(A, dev), to_dev(Wg, dev), to_dev(Wu, dev), to_dev(ea, dev),
                                    to_dev(ewg, dev), to_dev(ewu, dev)))
    rng = np.random.default_rng(12)
    rows = sorted({0, 255, 256, 8191} | set(rng.integers(0, 8192, 12).tolist()))
    assert (got[rows] == oracle_mod.w8a8_swiglu(A, Wg, Wu, ea, ewg, ewu, rows=rows)).all()
    cols = sorted({0, 127, 128, 12287} | {128 * t + int(rng.integers(0, 128)) for t in range(0, 96, 3)})
    want = oracle_mod.w8a8_swiglu(A, np.ascontiguousarray(Wg[cols]), np.ascontiguousarray(Wu[cols]), ea,
                                  np.ascontiguousarray(ewg[cols]), np.ascontiguousarray(ewu[cols]))
    assert (got[:, cols] == want).all()


def test_fused_second_pass_paths(lib, dev, oracle_mod):
    """The fused epilogue's out-of-line evaluations, which random FFN-like inputs rarely reach:
    (1) exponents of magnitude above 2^20 whose sums stay in the domain (the whole warp's
    outputs go to the second pass); (2) gates of magnitude >= 64 on nearly every output (more
    than four output columns of a warp left to the second pass, so the accumulator buffer is
    held through it); (3) zero activation rows (+0 whatever the exponents); (4) exponent sums
    outside the domain on two columns (NaN there, DETGEMM_ERR_RANGE, every other output exact)."""
    from gpu_util import padded
    rng = np.random.default_rng(41)
    M, N, K = 300, 260, 64
    mk = lambda *s: np.clip(np.rint(rng.standard_normal(s) * 30), -127, 127).astype(np.int8)
    A, Wg, Wu = mk(M, K), mk(N, K), mk(N, K)
    A[7] = 0
    A[200] = 0
    dA, dWg, dWu = padded(A, dev, K), padded(Wg, dev, K), padded(Wu, dev, K)

    def run(ea, ewg, ewu):
        return bf16_bits(lib.w8a8_swiglu(dA, dWg, dWu, to_dev(ea, dev), to_dev(ewg, dev), to_dev(ewu, dev)))

    # (1) and (3): large exponents, in-range sums
    ea = (2 ** 21 + rng.integers(-14, -6, M)).astype(np.int32)
    ewg = (-(2 ** 21) + rng.integers(-4, 4, N)).astype(np.int32)
    ewu = (-(2 ** 21) + rng.integers(-4, 4, N)).astype(np.int32)
    got = run(ea, ewg, ewu)
    assert (got == oracle_mod.w8a8_swiglu(A, Wg, Wu, ea, ewg, ewu)).all()
    assert (got[7] == 0).all() and (got[200] == 0).all()
    assert lib.device_status() == lib.OK
    # (2): g = the accumulator itself, |g| in the thousands
    ea = np.zeros(M, np.int32)
    ewg = np.zeros(N, np.int32)
    ewu = rng.integers(-12, -4, N).astype(np.int32)
    G = A.astype(np.int64) @ Wg.astype(np.int64).T
    assert (np.abs(G) >= 64).mean() > 0.9
    got = run(ea, ewg, ewu)
    assert (got == oracle_mod.w8a8_swiglu(A, Wg, Wu, ea, ewg, ewu)).all()
    assert lib.device_status() == lib.OK
    # (4): columns 5 and 131 with a gate exponent sum of 100
    ea = rng.integers(-14, -6, M).astype(np.int32)
    ewg = rng.integers(-14, -6, N).astype(np.int32)
    ewu = rng.integers(-14, -6, N).astype(np.int32)
    bad = [5, 131]
    ewg_bad = ewg.copy()
    ewg_bad[bad] = 100 - ea.max()
    got = run(ea, ewg_bad, ewu)
    assert lib.device_status() == lib.ERR_RANGE
    good = [j for j in range(N) if j not in bad]
    want = oracle_mod.w8a8_swiglu(A, np.ascontiguousarray(Wg[good]), np.ascontiguousarray(Wu[good]), ea,
                                  np.ascontiguousarray(ewg[good]), np.ascontiguousarray(ewu[good]))
    assert (got[:, good] == want).all()
    U = A.astype(np.int64) @ Wu.astype(np.int64).T
    for j in bad:
        # exponent sums 100 - max(ea) + ea_i lie outside [-60, 40] for every row: NaN where both
        # accumulators are nonzero, +0 where one is zero
        nz = (G[:, j] != 0) & (U[:, j] != 0)
        assert (got[nz, j] == 0x7FC0).all() and (got[~nz, j] == 0).all()
