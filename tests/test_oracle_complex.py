"""Pins of the complex-A SSD oracle (oracle/complex_ssd.py) against facts fixed outside it:
hand-worked values, the chunkwise/naive equivalence the page states, the independent C
oracle of the real recurrence, symmetries of the bilinear form, and split invariance."""
import math
import os

import numpy as np
import pytest

from oracle import complex_ssd as cx
from oracle import sequential

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "complex_ssd.txt")
DT_ONE = math.log(math.e - 1.0)            # softplus(DT_ONE) = 1
A_HALF_I = complex(-math.log(2.0), math.pi / 2)   # exp(A) = i/2


def rel(a, b):
    return np.linalg.norm(np.ravel(a - b)) / max(np.linalg.norm(np.ravel(b)), 1e-300)


def golden():
    rows = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        case, t, re, im = line.split()
        rows[(case, t)] = complex(float(re), float(im))
    return rows


def unit(T, x=1.0, B=1.0, C=1.0, eta=None):
    sh = (1, T, 1, 1)
    init = None if eta is None else np.full((1, 1, 1, 1), eta, dtype=np.complex128)
    return dict(x=np.full(sh, x, dtype=np.complex128), A=np.array([A_HALF_I]),
                B=np.full(sh, B, dtype=np.complex128), C=np.full(sh, C, dtype=np.complex128),
                dt=np.full((1, T, 1), DT_ONE), init=init)


def rand_problem(rng, Bt=2, T=37, H=3, D=4, N=5, init=True):
    def c(*s):
        return (rng.standard_normal(s) + 1j * rng.standard_normal(s)) / math.sqrt(2)
    A = -np.exp(rng.uniform(math.log(0.3), math.log(3.0), H)) + 1j * rng.uniform(-math.pi, math.pi, H)
    return dict(x=c(Bt, T, H, D), A=A, B=c(Bt, T, H, N), C=c(Bt, T, H, N),
                dt=rng.standard_normal((Bt, T, H)), init=0.3 * c(Bt, H, D, N) if init else None)


def test_golden_geometric_rotation():
    g = golden()
    y, f = cx.naive(**unit(80))
    for t in range(5):
        assert abs(y[0, t, 0, 0] - g[("unit", str(t))]) < 1e-15
    assert abs(y[0, -1, 0, 0] - g[("unit", "inf")]) < 1e-15
    assert abs(f[0, 0, 0, 0] - g[("unit", "inf")]) < 1e-15
    y, _ = cx.naive(**unit(4, eta=2.0))
    for t in range(4):
        assert abs(y[0, t, 0, 0] - g[("init", str(t))]) < 1e-15
    y, _ = cx.naive(**unit(2, x=1 - 1j, B=2.0, C=1j))
    for t in range(2):
        assert abs(y[0, t, 0, 0] - g[("mixed", str(t))]) < 1e-15
    # the chunkwise path returns the real part of the same numbers
    yc = cx.chunkwise(**unit(80), Q=16)
    assert abs(yc[0, 3, 0, 0] - g[("unit", "3")].real) < 1e-15


@pytest.mark.parametrize("Q", [1, 2, 4, 16, 37])
def test_chunkwise_equals_naive_real_part(Q):
    """Chunk-length invariance with time-varying dt, an initial state and a ragged tail."""
    p = rand_problem(np.random.default_rng(Q))
    y, _ = cx.naive(**p)
    yc = cx.chunkwise(Q=Q, **p)
    assert yc.dtype == np.float64
    assert rel(yc, y.real) < 1e-12


def test_planted_window_mistake_is_seen():
    p = rand_problem(np.random.default_rng(9), T=40)
    y, _ = cx.naive(**p)
    assert rel(cx.chunkwise(Q=8, **p), y.real) < 1e-12
    assert rel(cx.chunkwise(Q=8, _window_shift=0, **p), y.real) > 1e-3


def test_real_special_case_matches_the_c_oracle():
    """Im(A) = 0 and real x, B, C: the real recurrence with input term dt*x*B, fed x/dt."""
    rng = np.random.default_rng(4)
    T, H, D, N = 29, 3, 4, 5
    x = rng.standard_normal((1, T, H, D))
    B = rng.standard_normal((1, T, H, N))
    C = rng.standard_normal((1, T, H, N))
    dt = rng.standard_normal((1, T, H))
    A = -np.exp(rng.uniform(-1, 1, H))
    init = rng.standard_normal((1, H, D, N))
    y, f = cx.naive(x, A + 0j, B, C, dt, init=init)
    sp = cx.softplus(dt)
    ys, fs = sequential.forward(x=(x / sp[..., None])[0], dt_raw=dt[0], A=A, B=B[0], C=C[0], init=init)
    assert np.abs(y.imag).max() == 0.0
    assert rel(y.real[0], ys) < 1e-12
    assert rel(f.real, fs) < 1e-12


def test_bilinear_phase_and_conjugation():
    rng = np.random.default_rng(5)
    p = rand_problem(rng)
    y, f = cx.naive(**p)
    ph = np.exp(1j * rng.uniform(-math.pi, math.pi, size=p["B"].shape))
    q = dict(p, B=p["B"] * ph, C=p["C"] / ph)
    q["init"] = None
    y0, _ = cx.naive(**dict(p, init=None))
    y1, _ = cx.naive(**q)
    # per-position phases do not cancel in general; a global phase per (b, h, n) does
    ph_g = np.exp(1j * rng.uniform(-math.pi, math.pi, size=(2, 1, 3, 5)))
    y2, _ = cx.naive(**dict(p, init=None, B=p["B"] * ph_g, C=p["C"] / ph_g))
    assert rel(y2, y0) < 1e-13
    assert rel(y1, y0) > 1e-3
    yc, fc = cx.naive(x=p["x"].conj(), A=p["A"].conj(), B=p["B"].conj(), C=p["C"].conj(), dt=p["dt"],
                      init=p["init"].conj())
    assert rel(yc, y.conj()) < 1e-13 and rel(fc, f.conj()) < 1e-13


def test_linear_in_x_and_affine_in_init():
    rng = np.random.default_rng(6)
    p = rand_problem(rng)
    p2 = rand_problem(np.random.default_rng(7))
    a, b = 0.7 - 0.2j, -1.3 + 0.5j
    ya, _ = cx.naive(**dict(p, init=None))
    yb, _ = cx.naive(**dict(p, x=p2["x"], init=None))
    yab, _ = cx.naive(**dict(p, x=a * p["x"] + b * p2["x"], init=None))
    assert rel(yab, a * ya + b * yb) < 1e-13
    yi, _ = cx.naive(**dict(p, x=0 * p["x"]))
    y, _ = cx.naive(**p)
    assert rel(y, ya + yi) < 1e-13


@pytest.mark.parametrize("T1", [1, 20, 36])
def test_split_walk_bit_exact(T1):
    p = rand_problem(np.random.default_rng(8))
    y, f = cx.naive(**p)
    cut = lambda k, a, b: p[k][:, a:b]
    y1, f1 = cx.naive(cut("x", 0, T1), p["A"], cut("B", 0, T1), cut("C", 0, T1), cut("dt", 0, T1), init=p["init"])
    y2, f2 = cx.naive(cut("x", T1, None), p["A"], cut("B", T1, None), cut("C", T1, None), cut("dt", T1, None),
                      init=f1)
    assert np.array_equal(np.concatenate([y1, y2], axis=1), y)
    assert np.array_equal(f2, f)
