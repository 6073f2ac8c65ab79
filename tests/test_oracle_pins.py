"""Pins of the float64 oracle against facts fixed by the mathematics (CPU only).

Each test ties the sequential oracle (or one of its sibling forms) to something
other than itself: a hand-worked closed form, the independent materialised
quadratic form, the chunkwise decomposition at many chunk sizes, split-sequence
invariance, linearity, and a textbook IIR filter (scipy.signal.lfilter).
"""
import math
import os

import numpy as np
import pytest

from oracle import sequential, quadratic, chunked64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "geometric_series.txt")


def rand_problem(rng, T=40, H=4, P=5, G=2, N=3, S=1, z=True, D=True, bias=True, init=True,
                 dt_scale=0.5, A_range=(1.0, 16.0), cu=None):
    x = rng.standard_normal((T, H, P))
    dt_raw = dt_scale * rng.standard_normal((T, H))
    A = -np.exp(rng.uniform(math.log(A_range[0]), math.log(A_range[1]), H))
    B = rng.standard_normal((T, G, N))
    C = rng.standard_normal((T, G, N))
    u = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), H))
    p = dict(x=x, dt_raw=dt_raw, A=A, B=B, C=C,
             D=rng.standard_normal(H) if D else None,
             z=rng.standard_normal((T, H, P)) if z else None,
             dt_bias=(u + np.log(-np.expm1(-u))) if bias else None,
             init=0.1 * rng.standard_normal((S, H, P, N)) if init else None,
             cu=cu if cu is not None else [0, T])
    return p


def rel(a, b):
    return np.linalg.norm(np.ravel(a - b)) / max(np.linalg.norm(np.ravel(b)), 1e-300)


# --- pin 1: the materialised semiseparable form ------------------------------------------
@pytest.mark.parametrize("G", [1, 2])
@pytest.mark.parametrize("feat", [(True, True, True, True), (False, False, False, False), (True, False, True, False)])
def test_sequential_matches_quadratic_form(G, feat):
    z, D, bias, init = feat
    rng = np.random.default_rng(1 + G)
    p = rand_problem(rng, T=48, H=4, P=6, G=G, N=5, z=z, D=D, bias=bias, init=init)
    y, f = sequential.forward(**p)
    yq, fq = quadratic.forward(**p)
    assert rel(y, yq) < 1e-12
    assert rel(f, fq) < 1e-12


def test_quadratic_form_multi_sequence():
    rng = np.random.default_rng(7)
    cu = [0, 9, 9, 30, 47]          # includes an empty sequence
    p = rand_problem(rng, T=47, H=3, P=4, G=1, N=6, S=4, cu=cu)
    y, f = sequential.forward(**p)
    yq, fq = quadratic.forward(**p)
    assert rel(y, yq) < 1e-12
    assert rel(f, fq) < 1e-12
    # empty sequence: final state is the initial state
    assert np.array_equal(f[1], p["init"][1])


# --- pin 2: hand-worked geometric series ----------------------------------------------------
def _golden():
    rows = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        k, v = line.split()
        rows[k] = float(v)
    return rows


def _unit_problem(T, eta=None, Dv=None):
    one = np.ones((T, 1, 1))
    return dict(x=one, dt_raw=np.zeros((T, 1)), A=np.array([-1.0]), B=one, C=one,
                D=None if Dv is None else np.array([Dv]), z=None, dt_bias=np.zeros(1),
                init=None if eta is None else np.full((1, 1, 1, 1), eta))


def test_geometric_series_golden():
    g = _golden()
    y, f = sequential.forward(**_unit_problem(200))
    for t in range(5):
        assert abs(y[t, 0, 0] - g[str(t)]) <= 1e-15 * g[str(t)] * 4
    assert abs(y[-1, 0, 0] - g["inf"]) < 1e-14
    assert abs(f[0, 0, 0, 0] - g["inf"]) < 1e-14


def test_geometric_series_with_init_and_D():
    T, eta, Dv = 30, 0.37, -1.25
    y, f = sequential.forward(**_unit_problem(T, eta=eta, Dv=Dv))
    t = np.arange(T)
    expect = 2 * math.log(2) * (1 - 2.0 ** -(t + 1)) + eta * 2.0 ** -(t + 1) + Dv
    assert np.max(np.abs(y[:, 0, 0] - expect)) < 1e-14


# --- pin 3: chunk-size invariance (time-varying dt) -----------------------------------------
@pytest.mark.parametrize("Q", [1, 2, 4, 16, 64, 75])
def test_chunked_matches_sequential(Q):
    rng = np.random.default_rng(11)
    p = rand_problem(rng, T=75, H=4, P=4, G=2, N=4, dt_scale=1.0)
    y, f = sequential.forward(**p)
    yc, fc = chunked64.forward(Q=Q, **p)
    assert rel(yc, y) < 1e-12
    assert rel(fc, f) < 1e-12


def test_chunked_propagation_uses_previous_chunk_total():
    """The carry-in of chunk z decays by exp(CD[z-1] - CD[c]); with time-varying dt
    a window one chunk too long (CD[z] - CD[c]) must be visibly wrong.  Planting that
    mistake in a copy of the oracle's propagation shows the invariance test can see it."""
    rng = np.random.default_rng(5)
    T, P, N, Q = 32, 3, 2, 4
    x = rng.standard_normal((T, P))
    dt = np.exp(rng.standard_normal(T))
    B = rng.standard_normal((T, N))
    C = rng.standard_normal((T, N))
    y, fin, inter = chunked64.forward_one(x, dt, -0.7, B, C, Q)
    # planted mistake: the same propagation with CD[z] in place of CD[z-1]
    cs = inter["cs"]
    states = inter["chunk_states"]
    CD = np.cumsum(cs[:, -1])
    n_c = cs.shape[0]
    wrong = np.zeros_like(inter["carry_in"])
    for zc in range(n_c):
        for c in range(zc):
            wrong[zc] += np.exp(CD[zc] - CD[c]) * states[c]
    assert rel(wrong, inter["carry_in"]) > 1e-2
    one = dict(x=x[:, None, :], dt_raw=np.log(np.expm1(dt))[:, None], A=np.array([-0.7]),
               B=B[:, None, :], C=C[:, None, :])
    ys, fs = sequential.forward(**one)
    assert rel(y, ys[:, 0, :]) < 1e-12


# --- pin 4: split-sequence invariance ----------------------------------------------------------
@pytest.mark.parametrize("L1", [1, 17, 40])
def test_split_sequence_bit_exact(L1):
    rng = np.random.default_rng(3)
    p = rand_problem(rng, T=64, H=3, P=4, G=1, N=5)
    y, f = sequential.forward(**p)
    a = {k: v for k, v in p.items() if k != "cu"}
    first = {k: (v[:L1] if k in ("x", "dt_raw", "B", "C", "z") and v is not None else v) for k, v in a.items()}
    second = {k: (v[L1:] if k in ("x", "dt_raw", "B", "C", "z") and v is not None else v) for k, v in a.items()}
    y1, f1 = sequential.forward(**first)
    second["init"] = f1
    y2, f2 = sequential.forward(**second)
    assert np.array_equal(np.concatenate([y1, y2], 0), y)
    assert np.array_equal(f2, f)


# --- pin 5: linearity and special cases ----------------------------------------------------------
def test_linear_in_x_and_affine_in_init():
    rng = np.random.default_rng(9)
    p = rand_problem(rng, T=30, H=2, P=3, G=1, N=4, z=False, D=True)
    x2 = rng.standard_normal(p["x"].shape)
    i2 = 0.1 * rng.standard_normal(p["init"].shape)
    ya, fa = sequential.forward(**p)
    q = dict(p, x=x2, init=i2)
    yb, fb = sequential.forward(**q)
    r = dict(p, x=2.0 * p["x"] - 3.0 * x2, init=2.0 * p["init"] - 3.0 * i2)
    yr, fr = sequential.forward(**r)
    assert rel(yr, 2 * ya - 3 * yb) < 1e-12
    assert rel(fr, 2 * fa - 3 * fb) < 1e-12


def test_A_zero_is_causal_linear_attention():
    rng = np.random.default_rng(2)
    p = rand_problem(rng, T=25, H=2, P=3, G=1, N=4, z=False, D=False, init=False)
    p["A"] = np.zeros(2)
    y, f = sequential.forward(**p)
    v = p["dt_raw"] + p["dt_bias"][None, :]
    dt = np.log1p(np.exp(v))
    for h in range(2):
        # h_t = sum_{s<=t} dt_s x_s (outer) B_s ; y_t = C_t . h_t
        outer = dt[:, h, None, None] * p["x"][:, h, :, None] * p["B"][:, 0, None, :]
        hs = np.cumsum(outer, 0)
        yt = np.einsum("tpn,tn->tp", hs, p["C"][:, 0, :])
        assert rel(y[:, h, :], yt) < 1e-12


def test_scalar_state_is_first_order_iir_filter():
    scipy_signal = pytest.importorskip("scipy.signal")
    rng = np.random.default_rng(4)
    T = 300
    x = rng.standard_normal((T, 1, 1))
    dt0 = 0.3
    A = -2.0
    p = dict(x=x, dt_raw=np.full((T, 1), math.log(math.expm1(dt0))), A=np.array([A]),
             B=np.ones((T, 1, 1)), C=np.ones((T, 1, 1)))
    y, _ = sequential.forward(**p)
    a = math.exp(dt0 * A)
    ref = scipy_signal.lfilter([dt0], [1.0, -a], x[:, 0, 0])
    assert np.max(np.abs(y[:, 0, 0] - ref)) < 1e-12


# --- pin 7: packed sequences equal separate runs -----------------------------------------------
def test_packed_equals_separate():
    rng = np.random.default_rng(8)
    cu = [0, 5, 5, 21, 40]
    p = rand_problem(rng, T=40, H=4, P=3, G=2, N=4, S=4, cu=cu)
    y, f = sequential.forward(**p)
    for s in range(4):
        t0, t1 = cu[s], cu[s + 1]
        q = {k: (v[t0:t1] if k in ("x", "dt_raw", "B", "C", "z") and v is not None else v) for k, v in p.items()}
        q["init"] = p["init"][s:s + 1]
        q["cu"] = [0, t1 - t0]
        ys, fs = sequential.forward(**q)
        assert np.array_equal(ys, y[t0:t1])
        assert np.array_equal(fs[0], f[s])


def test_head_subset_matches_full_run():
    rng = np.random.default_rng(12)
    p = rand_problem(rng, T=20, H=6, P=3, G=2, N=4)
    y, f = sequential.forward(**p)
    ys, fs = sequential.forward(heads=[1, 4], **p)
    assert np.array_equal(ys[:, [1, 4]], y[:, [1, 4]])
    assert np.array_equal(fs[:, [1, 4]], f[:, [1, 4]])
    assert not ys[:, 0].any()
