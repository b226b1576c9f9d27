"""The seeded input generators: deterministic, in range, with the stated distributions."""
import numpy as np


def test_deterministic_and_seed_dependent(synth):
    a = synth.uniform_i8(0, 0, (1000,))
    b = synth.uniform_i8(0, 0, (1000,))
    c = synth.uniform_i8(1, 0, (1000,))
    d = synth.uniform_i8(0, 1, (1000,))
    assert (a == b).all() and (a != c).any() and (a != d).any()


def test_uniform_ranges(synth):
    x = synth.uniform_i8(5, 0, (200000,), -127, 127)
    assert x.min() == -127 and x.max() == 127
    assert abs(x.astype(np.float64).mean()) < 1.0
    e = synth.uniform_i32(5, 2, (100000,), -12, -4)
    assert set(np.unique(e).tolist()) == set(range(-12, -3))


def test_rounded_normal(synth):
    x = synth.normal_i8(2, 0, (400000,), 30.0).astype(np.float64)
    assert abs(x.mean()) < 0.2 and abs(x.std() - 30.0) < 0.3
    y = synth.normal_i8(2, 0, (100000,), 200.0)
    assert y.min() == -127 and y.max() == 127  # clipped


def test_normal_pow2(synth):
    x = synth.normal_pow2_f32(4, 0, (100000,), -8, 8)
    m, e = np.frexp(np.abs(x[x != 0]).astype(np.float64))
    assert np.isfinite(x).all() and e.max() <= 12 and e.min() >= -30


def test_prefix_rows_of_sweep(synth):
    A, W, ea, ew = synth.sweep(64)
    A2, W2, ea2, ew2 = synth.sweep(2048)
    assert (A == A2[:64]).all() and (ea == ea2[:64]).all() and (W == W2).all()
