"""Pins of the oracle's adjoint (CPU only).

(a) Central finite differences in float64 of the sequential forward.
(b) torch float64 autograd of the independent quadratic form.
The case has z, D, dt_bias, an initial state and dfinal, H=6 heads in G=2
groups (3 heads per group), and two packed sequences.
"""
import numpy as np
import pytest

from oracle import sequential, quadratic


def make(rng, T=24, H=6, P=4, G=2, N=4, cu=(0, 11, 24)):
    S = len(cu) - 1
    u = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), H))
    return dict(
        x=rng.standard_normal((T, H, P)), dt_raw=0.5 * rng.standard_normal((T, H)),
        A=-np.exp(rng.uniform(0, np.log(16.0), H)), B=rng.standard_normal((T, G, N)),
        C=rng.standard_normal((T, G, N)), D=rng.standard_normal(H),
        z=rng.standard_normal((T, H, P)), dt_bias=u + np.log(-np.expm1(-u)),
        init=0.1 * rng.standard_normal((S, H, P, N)), cu=list(cu))


def loss(p, dy, dfinal):
    y, f = sequential.forward(**p)
    return float(np.sum(dy * y) + np.sum(dfinal * f))


GRAD_OF = dict(x="dx", dt_raw="ddt_raw", A="dA", B="dB", C="dC", D="dD", z="dz", dt_bias="ddt_bias", init="dinit")


@pytest.fixture(scope="module")
def case():
    rng = np.random.default_rng(0)
    p = make(rng)
    T, H, P = p["x"].shape
    dy = rng.standard_normal((T, H, P))
    dfinal = 0.1 * rng.standard_normal(p["init"].shape)
    g = sequential.backward(dy=dy, dfinal=dfinal, ckpt=5, **p)
    return p, dy, dfinal, g


@pytest.mark.parametrize("name", list(GRAD_OF))
def test_adjoint_matches_central_differences(case, name):
    p, dy, dfinal, g = case
    rng = np.random.default_rng(hash(name) % 1000)
    arr = p[name]
    flat = arr.reshape(-1)
    idx = rng.choice(flat.size, size=min(12, flat.size), replace=False)
    eps = 1e-6
    for i in idx:
        orig = flat[i]
        flat[i] = orig + eps
        lp = loss(p, dy, dfinal)
        flat[i] = orig - eps
        lm = loss(p, dy, dfinal)
        flat[i] = orig
        fd = (lp - lm) / (2 * eps)
        an = g[GRAD_OF[name]].reshape(-1)[i]
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, i, fd, an)


def test_adjoint_matches_torch_autograd_of_quadratic_form(case):
    torch = pytest.importorskip("torch")
    p, dy, dfinal, g = case
    cu = p["cu"]
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True)
         for k, v in p.items() if k != "cu"}
    total = 0.0
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        y, f = quadratic.forward_torch(t["x"][a:b], t["dt_raw"][a:b], t["A"], t["B"][a:b], t["C"][a:b],
                                       D=t["D"], z=t["z"][a:b], dt_bias=t["dt_bias"], init=t["init"][s])
        total = total + (y * torch.tensor(dy[a:b])).sum() + (f * torch.tensor(dfinal[s])).sum()
    total.backward()
    for name, gname in GRAD_OF.items():
        ref = t[name].grad.numpy()
        err = np.max(np.abs(ref - g[gname])) / max(np.max(np.abs(ref)), 1e-30)
        assert err < 1e-11, (name, err)


def test_checkpoint_interval_does_not_change_gradients(case):
    p, dy, dfinal, g = case
    g2 = sequential.backward(dy=dy, dfinal=dfinal, ckpt=128, **p)
    for k in g:
        assert np.allclose(g[k], g2[k], rtol=1e-13, atol=1e-15), k


def test_head_subset_backward():
    rng = np.random.default_rng(3)
    p = make(rng, H=4, G=2)
    T, H, P = p["x"].shape
    dy = rng.standard_normal((T, H, P))
    full = sequential.backward(dy=dy, **p)
    part = sequential.backward(dy=dy, heads=[2, 3], **p)   # all heads of group 1
    assert np.array_equal(part["dB"][:, 1], full["dB"][:, 1])
    assert np.array_equal(part["dx"][:, 2:], full["dx"][:, 2:])
