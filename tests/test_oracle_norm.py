"""Pins of the gated normalisation oracle (CPU): hand-worked values, closed forms and
invariants, finite differences and an independent autograd formulation, in every mode
(RMS or LayerNorm, the gate before or after the norm)."""
import os

import numpy as np
import pytest

from oracle import gated_norm as gn

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "gated_norm.txt")


def golden():
    d = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, *v = line.split()
            d[k] = [float(x) for x in v]
    return d


def test_hand_worked_values():
    g = golden()
    out, rstd = gn.forward(np.array([g["y"]]), np.array(g["w"]), 2, eps=g["eps"][0])
    assert np.allclose(rstd[0], g["rstd"], rtol=1e-15, atol=0)
    assert np.allclose(out[0], g["out"], rtol=1e-15, atol=0)
    out, rstd = gn.forward(np.array([g["y2"]]), np.ones(4), 2, eps=0.0)
    assert np.allclose(rstd[0], g["rstd2"], rtol=1e-15, atol=0)
    assert np.allclose(out[0], g["out2"], rtol=1e-15, atol=1e-300)


def rand(rng, rows=5, width=24, group=8, gate=True):
    y = rng.standard_normal((rows, width))
    z = rng.standard_normal((rows, width)) if gate else None
    w = rng.standard_normal(width)
    return y, z, w, group


@pytest.mark.parametrize("eps", [0.0, 1e-5, 0.3])
def test_mean_square_closed_form(eps):
    """With w = 1, each normalised group has mean square ms / (ms + eps)."""
    rng = np.random.default_rng(1)
    y, z, _, G = rand(rng)
    out, _ = gn.forward(y, np.ones(y.shape[1]), G, z=z, eps=eps)
    v = y * z / (1 + np.exp(-z))
    for g in range(y.shape[1] // G):
        ms = np.mean(v[:, g * G:(g + 1) * G] ** 2, axis=1)
        got = np.mean(out[:, g * G:(g + 1) * G] ** 2, axis=1)
        assert np.allclose(got, ms / (ms + eps), rtol=1e-13)


def test_scale_invariance_and_zero_gate():
    rng = np.random.default_rng(2)
    y, z, w, G = rand(rng)
    a, _ = gn.forward(y, w, G, z=z, eps=0.0)
    b, _ = gn.forward(7.5 * y, w, G, z=z, eps=0.0)
    assert np.allclose(a, b, rtol=1e-13)
    out, _ = gn.forward(y, w, G, z=np.zeros_like(y), eps=1e-5)   # silu(0) = 0: the gate closes
    assert np.all(out == 0)
    # without a gate the group structure alone decides: one group == the row's RMS norm
    o1, r1 = gn.forward(y, w, y.shape[1])
    assert np.allclose(o1, y / np.sqrt(np.mean(y * y, axis=1, keepdims=True) + 1e-5) * w, rtol=1e-13)


MODES = [dict(), dict(layer_norm=True), dict(gate_after=True), dict(layer_norm=True, gate_after=True)]


@pytest.mark.parametrize("eps", [0.0, 1e-5, 0.3])
def test_layer_norm_closed_form(eps):
    """LayerNorm, w = 1: each normalised group has mean 0 and mean square var / (var + eps)."""
    rng = np.random.default_rng(5)
    y, z, _, G = rand(rng)
    out, _ = gn.forward(y, np.ones(y.shape[1]), G, z=z, eps=eps, layer_norm=True)
    v = y * z / (1 + np.exp(-z))
    for g in range(y.shape[1] // G):
        seg = v[:, g * G:(g + 1) * G]
        var = np.var(seg, axis=1)
        o = out[:, g * G:(g + 1) * G]
        assert np.allclose(np.mean(o, axis=1), 0.0, atol=1e-13)
        assert np.allclose(np.mean(o * o, axis=1), var / (var + eps), rtol=1e-12)


def test_gate_after_and_shift_invariance():
    """The gate after the norm multiplies the ungated normalised rows; LayerNorm ignores a
    constant added to every feature of a group; without a gate the gate order is moot."""
    rng = np.random.default_rng(6)
    y, z, w, G = rand(rng)
    s = z / (1 + np.exp(-z))
    for ln in (False, True):
        a, ra = gn.forward(y, w, G, z=z, layer_norm=ln, gate_after=True)
        b, rb = gn.forward(y, w, G, layer_norm=ln)
        assert np.allclose(a, b * s, rtol=1e-13) and np.array_equal(ra, rb)
        c, _ = gn.forward(y, w, G, layer_norm=ln, gate_after=True)
        assert np.allclose(c, b, rtol=0, atol=0)
    shift = np.repeat(rng.standard_normal((y.shape[0], y.shape[1] // G)), G, axis=1)
    a, _ = gn.forward(y + shift, w, G, layer_norm=True, gate_after=True)
    b, _ = gn.forward(y, w, G, layer_norm=True, gate_after=True)
    assert np.allclose(a, b, rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("gate", [True, False])
def test_gradients_by_central_differences(gate, mode):
    rng = np.random.default_rng(3)
    y, z, w, G = rand(rng, rows=3, width=12, group=4, gate=gate)
    dout = rng.standard_normal(y.shape)
    eps = 1e-3
    dy, dz, dw = gn.backward(y, w, dout, G, z=z, eps=eps, **mode)
    h = 1e-6

    def loss(y_, z_, w_):
        return float(np.sum(gn.forward(y_, w_, G, z=z_, eps=eps, **mode)[0] * dout))

    def fd(arr, name):
        g = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += h
            a2[idx] -= h
            args1 = dict(y_=y, z_=z, w_=w)
            args2 = dict(y_=y, z_=z, w_=w)
            args1[name], args2[name] = a1, a2
            g[idx] = (loss(**args1) - loss(**args2)) / (2 * h)
        return g

    assert np.allclose(dy, fd(y, "y_"), rtol=1e-6, atol=1e-8)
    assert np.allclose(dw, fd(w, "w_"), rtol=1e-6, atol=1e-8)
    if gate:
        assert np.allclose(dz, fd(z, "z_"), rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("mode", MODES)
def test_gradients_by_autograd_of_a_tensor_formula(mode):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    y, z, w, G = rand(rng, rows=6, width=32, group=16)
    dout = rng.standard_normal(y.shape)
    yt = torch.tensor(y, requires_grad=True)
    zt = torch.tensor(z, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    ln, after = mode.get("layer_norm", False), mode.get("gate_after", False)
    s = torch.nn.functional.silu(zt)
    v = (yt if after else yt * s).reshape(6, 2, 16)
    if ln:
        o = torch.nn.functional.layer_norm(v, (16,), eps=1e-5)
    else:
        o = v * torch.rsqrt(v.pow(2).mean(-1, keepdim=True) + 1e-5)
    o = o.reshape(6, 32) * wt * (s if after else 1.0)
    (o * torch.tensor(dout)).sum().backward()
    dy, dz, dw = gn.backward(y, w, dout, G, z=z, **mode)
    assert np.allclose(dy, yt.grad.numpy(), rtol=1e-12, atol=1e-14)
    assert np.allclose(dz, zt.grad.numpy(), rtol=1e-12, atol=1e-14)
    assert np.allclose(dw, wt.grad.numpy(), rtol=1e-12, atol=1e-14)
    out, _ = gn.forward(y, w, G, z=z, **mode)
    assert np.allclose(out, o.detach().numpy(), rtol=1e-12, atol=1e-14)
