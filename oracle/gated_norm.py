"""Gated normalisation over feature groups, float64 -- TEST INFRASTRUCTURE ONLY.

The normalisation that follows the SSD scan in a Mamba-2 block: the Helion pull request
for the Mamba-2 SSD path ("Summary", "Measurements": the gated-LayerNorm backward,
layernorm_gated.py, LayerNormFn / _layer_norm_bwd) names it without printing it.  Its
plainest reading, over groups of the feature axis, with s = silu(z) (s = 1 when no gate is
given) and g(i) = i // group_size:

    u[t, i]   = y[t, i] * s[t, i]   (the gate first, the default)   or   y[t, i]   (gate_after)
    mu[t, g]  = 0   (RMS normalisation, the default)   or   mean_{i in g} u[t, i]   (layer_norm)
    rstd[t,g] = 1 / sqrt(mean_{i in group g} (u[t, i] - mu[t, g])^2 + eps)
    out[t, i] = (u[t, i] - mu[t, g(i)]) * rstd[t, g(i)] * w[i]   (times s[t, i] with gate_after)

The backward is the exact derivative of that map for an upstream gradient dout: dy, dz
(through the gate) and dw (summed over rows).

Pinned by tests/test_oracle_norm.py: a hand-worked example (tests/golden/gated_norm.txt),
the closed forms of the normalised rows' mean square (RMS) and of their mean and variance
(LayerNorm), scale invariance at eps = 0, the zero gate, central finite differences of
every gradient in every mode, and torch float64 autograd of a direct tensor formula.
"""
import numpy as np


def _silu(z):
    return z / (1.0 + np.exp(-z))


def forward(y, w, group_size, z=None, eps=1e-5, layer_norm=False, gate_after=False):
    """y, z: [rows, width]; w: [width].  Returns (out, rstd[rows, width // group_size])."""
    y = np.asarray(y, np.float64)
    rows, width = y.shape
    s = _silu(np.asarray(z, np.float64)) if z is not None else np.ones_like(y)
    u = y.copy() if gate_after else y * s
    ng = width // group_size
    out = np.empty_like(u)
    rstd = np.empty((rows, ng))
    for t in range(rows):
        for g in range(ng):
            sl = slice(g * group_size, (g + 1) * group_size)
            seg = u[t, sl]
            c = seg - (np.mean(seg) if layer_norm else 0.0)
            r = 1.0 / np.sqrt(np.mean(c * c) + eps)
            rstd[t, g] = r
            out[t, sl] = c * r * w[sl] * (s[t, sl] if gate_after else 1.0)
    return out, rstd


def backward(y, w, dout, group_size, z=None, eps=1e-5, layer_norm=False, gate_after=False):
    """Gradients of sum(dout * out).  Returns (dy, dz or None, dw)."""
    y = np.asarray(y, np.float64)
    dout = np.asarray(dout, np.float64)
    rows, width = y.shape
    if z is not None:
        z = np.asarray(z, np.float64)
        sig = 1.0 / (1.0 + np.exp(-z))
        s = z * sig
        dsilu = sig * (1.0 + z * (1.0 - sig))
    else:
        s = np.ones_like(y)
    u = y.copy() if gate_after else y * s
    m = s if gate_after else np.ones_like(y)    # the factor after the norm
    ng = width // group_size
    du = np.empty_like(u)
    xhat = np.empty_like(u)
    dw = np.zeros(width)
    for t in range(rows):
        for g in range(ng):
            sl = slice(g * group_size, (g + 1) * group_size)
            seg = u[t, sl]
            c = seg - (np.mean(seg) if layer_norm else 0.0)
            r = 1.0 / np.sqrt(np.mean(c * c) + eps)
            xh = c * r
            xhat[t, sl] = xh
            gw = dout[t, sl] * w[sl] * m[t, sl]             # d sum(dout out) / d xhat
            # d xhat_i / d u_j = r (delta_ij - [layer_norm] / n - xhat_i xhat_j / n)
            du[t, sl] = r * (gw - (np.mean(gw) if layer_norm else 0.0) - xh * np.mean(gw * xh))
            dw[sl] += dout[t, sl] * xh * m[t, sl]
    if z is None:
        return du, None, dw
    if gate_after:
        return du, dout * w * xhat * dsilu, dw
    return du * s, du * y * dsilu, dw
