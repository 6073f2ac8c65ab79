"""Gated RMS normalisation over feature groups, float64 -- TEST INFRASTRUCTURE ONLY.

The normalisation that follows the SSD scan in a Mamba-2 block: the Helion pull request
for the Mamba-2 SSD path ("Summary", "Measurements": the gated-LayerNorm backward,
layernorm_gated.py, LayerNormFn / _layer_norm_bwd) names it without printing it.  Its
plainest reading (RMS normalisation with the gate applied before it, over groups of the
feature axis):

    v[t, i]   = y[t, i] * silu(z[t, i])            (v = y when no gate is given)
    rstd[t,g] = 1 / sqrt(mean_{i in group g} v[t, i]^2 + eps)
    out[t, i] = v[t, i] * rstd[t, g(i)] * w[i]

with g(i) = i // group_size.  The backward is the exact derivative of that map for an
upstream gradient dout: dy, dz (through the gate) and dw (summed over rows).

Pinned by tests/test_oracle_norm.py: a hand-worked example (tests/golden/gated_norm.txt),
the closed form of the normalised rows' mean square, scale invariance at eps = 0, the zero
gate, central finite differences of every gradient, and torch float64 autograd of a direct
tensor formula.
"""
import numpy as np


def _silu(z):
    return z / (1.0 + np.exp(-z))


def forward(y, w, group_size, z=None, eps=1e-5):
    """y, z: [rows, width]; w: [width].  Returns (out, rstd[rows, width // group_size])."""
    y = np.asarray(y, np.float64)
    rows, width = y.shape
    v = y * _silu(np.asarray(z, np.float64)) if z is not None else y.copy()
    ng = width // group_size
    out = np.empty_like(v)
    rstd = np.empty((rows, ng))
    for t in range(rows):
        for g in range(ng):
            seg = v[t, g * group_size:(g + 1) * group_size]
            r = 1.0 / np.sqrt(np.mean(seg * seg) + eps)
            rstd[t, g] = r
            out[t, g * group_size:(g + 1) * group_size] = seg * r * w[g * group_size:(g + 1) * group_size]
    return out, rstd


def backward(y, w, dout, group_size, z=None, eps=1e-5):
    """Gradients of sum(dout * out).  Returns (dy, dz or None, dw)."""
    y = np.asarray(y, np.float64)
    dout = np.asarray(dout, np.float64)
    rows, width = y.shape
    if z is not None:
        z = np.asarray(z, np.float64)
        sig = 1.0 / (1.0 + np.exp(-z))
        s = z * sig
        v = y * s
    else:
        v = y.copy()
    ng = width // group_size
    dv = np.empty_like(v)
    dw = np.zeros(width)
    for t in range(rows):
        for g in range(ng):
            sl = slice(g * group_size, (g + 1) * group_size)
            seg = v[t, sl]
            r = 1.0 / np.sqrt(np.mean(seg * seg) + eps)
            vhat = seg * r
            gw = dout[t, sl] * w[sl]
            # d out_i / d v_j = w_i (r delta_ij - v_i r^3 v_j / n)
            dv[t, sl] = r * (gw - vhat * np.mean(gw * vhat))
            dw[sl] += dout[t, sl] * vhat
    if z is None:
        return dv, None, dw
    dy = dv * s
    dz = dv * y * sig * (1.0 + z * (1.0 - sig))
    return dy, dz, dw
