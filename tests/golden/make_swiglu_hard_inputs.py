"""Writes swiglu_hard_inputs.txt: gated-linear-unit epilogue inputs (gacc, uacc, Eg, Eu) whose
value y = SiLU(g) * u, g = gacc 2^Eg, u = uacc 2^Eu, lies very close to a bfloat16 rounding
boundary (a midpoint between neighbours): within 2^-20 of it relative to y (an fp32 evaluation
cannot place it) and within 2^-52 (nor can an fp64 one). Inputs only: the expected outputs
come from the oracle at test time. Search: for a gate g and exponent Eu, c = SiLU(g) / g * g
is computed in extended precision and uacc chosen so that c * uacc * 2^Eu is nearest to a
midpoint; candidates are kept when mpmath at 300 bits confirms the distance. Run from the
repository root: python tests/golden/make_swiglu_hard_inputs.py"""
import os

import mpmath
import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
mpmath.mp.prec = 300


def distance(gacc, uacc, eg, eu):
    """relative distance of y to the nearest bf16 midpoint, at 300 bits"""
    g = mpmath.mpf(gacc) * mpmath.mpf(2) ** eg
    y = abs(g * mpmath.mpf(uacc) * mpmath.mpf(2) ** eu / (1 + mpmath.exp(-g)))
    e = int(mpmath.floor(mpmath.log(y, 2)))
    m = y / mpmath.mpf(2) ** (e - 7)  # in [128, 256)
    return abs(m - mpmath.floor(m) - mpmath.mpf(0.5)) / m


def search(rng, n, thresh):
    out = []
    ld = np.longdouble
    gacc = rng.integers(-2 ** 24, 2 ** 24, n)
    gacc[gacc == 0] = 1
    eg = rng.integers(-24, -18, n)
    g = gacc.astype(ld) * np.exp2(eg.astype(ld))
    c = g / (ld(1) + np.exp(-g))  # y = c * u
    eu = rng.integers(-40, -20, n)
    # a midpoint near c * 2^30 * 2^eu: pick odd j with 9 significant bits in that binade
    target = np.abs(c) * np.exp2(ld(30) + eu.astype(ld))
    e = np.floor(np.log2(target.astype(np.float64))).astype(np.int64)
    j = rng.integers(128, 256, n) * 2 + 1  # odd, 9 bits: a midpoint
    mid = j.astype(ld) * np.exp2((e - 8).astype(ld))
    x = mid / (np.abs(c) * np.exp2(eu.astype(ld)))
    uacc = np.rint(x)
    rel = np.abs(uacc - x) / x
    keep = (rel < thresh) & (uacc < 2 ** 31 - 1) & (uacc > 0)
    for i in np.nonzero(keep)[0]:
        ua = int(uacc[i]) * (1 if rng.random() < 0.5 else -1)
        cand = (int(gacc[i]), ua, int(eg[i]), int(eu[i]))
        d = distance(*cand)
        out.append((cand, float(d)))
    return out


def main():
    rng = np.random.default_rng(20260101)
    fp32_hard, fp64_hard = [], []
    while len(fp32_hard) < 40:
        fp32_hard += [c for c, d in search(rng, 20000, 2.0 ** -24) if 2.0 ** -40 < d < 2.0 ** -20]
    while len(fp64_hard) < 12:
        fp64_hard += [c for c, d in search(rng, 4_000_000, 2.0 ** -53) if d < 2.0 ** -52]
    with open(os.path.join(HERE, "swiglu_hard_inputs.txt"), "w") as f:
        f.write("# written by make_swiglu_hard_inputs.py (see its docstring); gacc uacc Eg Eu tier\n")
        for c in fp32_hard[:40]:
            f.write(" ".join(map(str, c)) + " fp32-ambiguous\n")
        for c in fp64_hard[:12]:
            f.write(" ".join(map(str, c)) + " fp64-ambiguous\n")


if __name__ == "__main__":
    main()
