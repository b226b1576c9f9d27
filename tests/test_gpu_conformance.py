"""The conformance instrument on the GPU: epilogue faults injected into the library's own
W8A8 path and the checks that can or cannot see them ("Deterministic LLM Inference Across
GPU Kernels ...", §III "Nine Faults", §IV "How much can a tolerance see?").

The exact int32 accumulators come from the product GEMM (detgemm_gemm_s8_i32); the injector
applies the correct epilogue or a fault (F1 scale precision, F2 double rounding, F3
multiplication order, F4 truncation) to the outputs a severity selects. Each injected output
is first compared element by element with the CPU reading of the same fault (exact rationals
and numpy fp32 arithmetic). The scorecard then checks the pages' findings on these kernels:
the null fault fires nothing; under power-of-two scales F1-F3 change no output while F4 is
seen only by the power-of-two identity; under real scales every epilogue fault that changes
an output stays within one spacing and passes every check; an operand fault is caught by the shared-operand check
and exceeds the tolerance; a precondition violation is refused and flagged.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import synthetic
from deterministic_detgemm_w8a8_gb300 import conformance as conf
from exact import bf16_bits_to_fraction, rne_bf16_exact, rne_f32_exact
from gpu_util import bf16_bits, cuda, dg, to_dev

pytestmark = pytest.mark.gpu

FAULTS = ("F1", "F2", "F3", "F4")


@pytest.fixture(scope="module")
def dev():
    return cuda()


@pytest.fixture(scope="module")
def lib():
    return dg()


def _rne_bf16_f32(x):
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _cpu_reading(acc, sa, sw, exact_vals):
    """CPU readings of every fault for every element (sa, sw: fp32 scales per row / column;
    exact_vals: the exact Fractions acc * sa * sw)."""
    f32acc = acc.astype(np.float32)
    SA = np.broadcast_to(sa[:, None], acc.shape).astype(np.float32)
    SW = np.broadcast_to(sw[None, :], acc.shape).astype(np.float32)
    exact = np.array([rne_bf16_exact(v) for v in exact_vals.ravel()], np.uint16).reshape(acc.shape)
    f2 = np.array([rne_f32_exact(v) for v in exact_vals.ravel()], np.float32).reshape(acc.shape)
    f4 = exact.copy()
    flat = exact_vals.ravel()
    for i in range(f4.size):
        r = bf16_bits_to_fraction(int(f4.flat[i]))
        if abs(r) > abs(flat[i]):
            f4.flat[i] -= 1
    return {
        "none": exact,
        "F1": _rne_bf16_f32(f32acc * (SA * SW)),
        "F2": _rne_bf16_f32(f2),
        "F3": _rne_bf16_f32((f32acc * SA) * SW),
        "F4": f4,
    }


@pytest.fixture(scope="module")
def case(lib, dev, oracle_mod):
    A, W, ea, ew = synthetic.w8a8_normal(31, 64, 256, 512, 30.0, 30.0, -14, -6)
    tA, tW = to_dev(A, dev), to_dev(W, dev)
    acc = lib.gemm_s8_i32(tA, tW)
    acc_np = acc.cpu().numpy().astype(np.int64)
    assert (acc_np == oracle_mod.gemm_s8_i32(A, W)).all()
    assert np.abs(acc_np).max() < 2 ** 24  # the regime where fp32 holds every accumulator
    rng = np.random.default_rng(32)
    sa_real = (rng.uniform(1.0, 2.0, 64) * np.exp2(rng.integers(-14, -6, 64))).astype(np.float32)
    sw_real = (rng.uniform(1.0, 2.0, 256) * np.exp2(rng.integers(-14, -6, 256))).astype(np.float32)
    exact_pow2 = np.array([[Fraction(int(a)) * Fraction(2) ** int(ea[i] + ew[j]) for j, a in enumerate(row)]
                           for i, row in enumerate(acc_np)], dtype=object)
    exact_real = np.array([[Fraction(int(a)) * Fraction(float(sa_real[i])) * Fraction(float(sw_real[j]))
                            for j, a in enumerate(row)] for i, row in enumerate(acc_np)], dtype=object)
    return {
        "A": A, "W": W, "ea": ea, "ew": ew, "acc": acc, "acc_np": acc_np,
        "pow2": (to_dev(ea, dev), to_dev(ew, dev),
                 _cpu_reading(acc_np, np.exp2(ea).astype(np.float32), np.exp2(ew).astype(np.float32), exact_pow2)),
        "real": (to_dev(sa_real, dev), to_dev(sw_real, dev), _cpu_reading(acc_np, sa_real, sw_real, exact_real)),
        "product": bf16_bits(lib.w8a8(tA, tW, to_dev(ea, dev), to_dev(ew, dev))),
        "oracle": oracle_mod.w8a8(A, W, ea, ew),
    }


@pytest.mark.parametrize("regime", ["pow2", "real"])
@pytest.mark.parametrize("severity", [0, 1, 2])
def test_injector_matches_the_cpu_readings(lib, case, regime, severity):
    sa, sw, want = case[regime]
    none = bf16_bits(lib.epilogue_inject(case["acc"], sa, sw, fault=lib.FAULT_NONE, severity=severity, seed=11))
    assert (none == want["none"]).all()
    for k, name in enumerate(FAULTS, start=1):
        got = bf16_bits(lib.epilogue_inject(case["acc"], sa, sw, fault=k, severity=severity, seed=11))
        mask = conf.faulted_mask(64, 256, severity, 11)
        expect = np.where(mask, want[name], want["none"])
        assert (got == expect).all(), (regime, severity, name, int((got != expect).sum()))


def test_null_fault_is_the_product_epilogue(lib, case):
    sa, sw, _ = case["pow2"]
    got = bf16_bits(lib.epilogue_inject(case["acc"], sa, sw, fault=lib.FAULT_NONE))
    assert (got == case["product"]).all() and (got == case["oracle"]).all()


def _cell(out, reference, A, W, A_ref, W_ref, scales_pow2):
    checks = conf.run_checks(out, reference, digest_arm=conf.operand_digest(A, W),
                             digest_reference=conf.operand_digest(A_ref, W_ref), A=A, W=W, scales_pow2=scales_pow2)
    observable = not np.array_equal(out, reference)
    return observable, checks


def test_scorecard(lib, dev, case):
    A, W = case["A"], case["W"]
    card = {}
    for regime in ("pow2", "real"):
        sa, sw, want = case[regime]
        reference = want["none"]
        for k, name in enumerate(("none",) + FAULTS):
            for severity in (0, 1, 2):
                out = bf16_bits(lib.epilogue_inject(case["acc"], sa, sw, fault=k, severity=severity, seed=3))
                card[(regime, name, severity)] = _cell(out, reference, A, W, A, W, regime == "pow2")
    for (regime, name, severity), (observable, checks) in card.items():
        fired = {c for c, v in checks.items() if v == conf.FIRE}
        assert checks["token_level"] == conf.NA
        if name == "none":
            assert not observable and not fired  # the null fault never fires
        elif regime == "pow2" and name in ("F1", "F2", "F3"):
            assert not observable  # power-of-two scales leave precision and order faults invisible
        elif regime == "pow2":  # F4
            if severity == 2:
                assert observable
            if observable:
                assert fired == {"pow2_identity"}  # the only check that sees a wrong rounding mode
        else:  # real scales: every epilogue fault passes every check
            assert checks["pow2_identity"] == conf.NA and not fired, (name, severity, fired)
            if severity == 2 and name == "F4":
                # truncation changes about half the outputs; F1-F3 change one only where an
                # fp32 intermediate crosses a bf16 rounding boundary (rare at |acc| < 2^24),
                # and an unobservable cell counts for no check
                assert observable
    # operand fault (F9): one int8 activation shifted by one, next to an exactly cancelling sum
    A9, W9 = A.copy(), W.copy()
    W9[5] = 0
    W9[5, 17], W9[5, 18] = 100, -100
    A9[3, 18] = A9[3, 17]
    tW9 = to_dev(W9, dev)
    ea_d, ew_d, _ = case["pow2"]
    reference = bf16_bits(lib.w8a8(to_dev(A9, dev), tW9, ea_d, ew_d))
    assert reference[3, 5] == 0  # the cancelling sum
    A9f = A9.copy()
    A9f[3, 17] = A9f[3, 17] + 1 if A9f[3, 17] < 127 else A9f[3, 17] - 1
    out = bf16_bits(lib.w8a8(to_dev(A9f, dev), tW9, ea_d, ew_d))
    observable, checks = _cell(out, reference, A9f, W9, A9, W9, True)
    assert observable
    assert checks["shared_operands"] == conf.FIRE and checks["tolerance_1_spacing"] == conf.FIRE
    assert conf.bf16_spacings(out, reference).max() > 100
    # precondition violation: a K beyond the exact-accumulation bound is refused by the
    # library and flagged by the precondition check
    Kbig = conf.MAX_K + 1
    Ab = torch.zeros((1, Kbig + 15), dtype=torch.int8, device=dev)[:, :Kbig]
    Wb = torch.zeros((8, Kbig + 15), dtype=torch.int8, device=dev)[:, :Kbig]
    with pytest.raises(lib.DetGemmError) as ei:
        lib.w8a8(Ab, Wb, torch.zeros(1, dtype=torch.int32, device=dev), torch.zeros(8, dtype=torch.int32, device=dev))
    assert ei.value.status == lib.ERR_PRECONDITION
    assert conf.check_exactness_preconditions(np.full((1, Kbig), 127, np.int8), np.full((8, Kbig), 127, np.int8)) \
        == conf.FIRE


def test_double_rounding_seen_beyond_fp32_accumulators(lib, dev):
    # |acc| >= 2^24 leaves fp32's exact range: acc = 2^24 + 2^16 + 1 rounds to 0x4B81 once,
    # but to fp32 first (a tie at 2^24 + 2^16, to even) and then to bf16 (a tie, to even) it
    # gives 0x4B80, one spacing off, which the power-of-two identity sees
    acc = torch.tensor([[2 ** 24 + 2 ** 16 + 1, -(2 ** 24 + 2 ** 16 + 1), 3, 0]], dtype=torch.int32, device=dev)
    z1 = torch.zeros(1, dtype=torch.int32, device=dev)
    z4 = torch.zeros(4, dtype=torch.int32, device=dev)
    good = bf16_bits(lib.epilogue_inject(acc, z1, z4, fault=lib.FAULT_NONE))
    bad = bf16_bits(lib.epilogue_inject(acc, z1, z4, fault=lib.FAULT_F2_DOUBLE_ROUNDING))
    assert good.tolist() == [[0x4B81, 0xCB81, 0x4040, 0x0000]]
    assert bad.tolist() == [[0x4B80, 0xCB80, 0x4040, 0x0000]]
    assert conf.check_pow2_identity(bad, good, True) == conf.FIRE
    assert conf.check_tolerance(bad, good) == conf.SILENT
