"""Causal depthwise convolution over the sequence axis with an optional SiLU -- TEST
INFRASTRUCTURE ONLY.

The step before the scan in a Mamba-2 block: the Helion pull request for the Mamba-2 SSD
path ("Summary": mamba_split_conv1d_scan_combined; "Testing": x, B and C are views of one
packed xBC buffer) runs it on the packed xBC = [x | B | C] channels and feeds the scan
slices of its output.  Its plainest reading, per channel c with kernel w[c, 0..K-1]:

    pre[t, c] = bias[c] + sum_{k=0}^{K-1} w[c, k] * u[t - (K-1) + k, c]
    out[t, c] = silu(pre[t, c])          (or pre itself without the activation)

where u[t'] = 0 for t' before the start of t's sequence (a batch row, or a packed sequence of
cu_seqlens): the window never reaches into another sequence.  The backward is its exact
derivative: du, dw (summed over tokens), dbias.

Pinned by tests/test_oracle_conv.py: the impulse response (the kernel reversed), the
identity kernel, torch's grouped conv1d on one sequence, packed == separate sequences, and
central finite differences of every gradient.
"""
import numpy as np


def _starts(T, cu):
    """Start of the sequence of every token on the flat axis."""
    st = np.zeros(T, np.int64)
    for s in range(len(cu) - 1):
        st[cu[s]:cu[s + 1]] = cu[s]
    return st


def forward(u, w, bias=None, cu=None, silu=True):
    """u: [T, channels] (T tokens on a flat axis, sequences given by cu, default one);
    w: [channels, K]; returns out [T, channels] and pre (before the activation)."""
    u = np.asarray(u, np.float64)
    T, Cn = u.shape
    K = w.shape[1]
    cu = [0, T] if cu is None else [int(c) for c in cu]
    st = _starts(T, cu)
    pre = np.zeros((T, Cn)) + (np.asarray(bias, np.float64) if bias is not None else 0.0)
    for t in range(T):
        for k in range(K):
            tp = t - (K - 1) + k
            if tp >= st[t]:
                pre[t] += w[:, k] * u[tp]
    out = pre / (1.0 + np.exp(-pre)) if silu else pre.copy()
    return out, pre


def backward(u, w, dout, bias=None, cu=None, silu=True):
    """Gradients of sum(dout * out): (du, dw, dbias)."""
    u = np.asarray(u, np.float64)
    T, Cn = u.shape
    K = w.shape[1]
    cu = [0, T] if cu is None else [int(c) for c in cu]
    st = _starts(T, cu)
    _, pre = forward(u, w, bias, cu, silu)
    if silu:
        sg = 1.0 / (1.0 + np.exp(-pre))
        g = np.asarray(dout, np.float64) * sg * (1.0 + pre * (1.0 - sg))
    else:
        g = np.asarray(dout, np.float64)
    du = np.zeros_like(u)
    dw = np.zeros((Cn, K))
    for t in range(T):
        for k in range(K):
            tp = t - (K - 1) + k
            if tp >= st[t]:
                du[tp] += w[:, k] * g[t]
                dw[:, k] += g[t] * u[tp]
    return du, dw, g.sum(axis=0)
