"""Materialised semiseparable ("quadratic") form of the SSD -- TEST INFRASTRUCTURE ONLY.

The Mamba-3-Lite "SSD Reference" page, section "Math: the recurrence both
functions implement", gives the closed form of the scan with zero initial state:

    y_t = sum_{s <= t} C_t^T ( prod_{u=s+1}^{t} abar_u ) B_s x_s ,   empty product = 1.

For the Mamba-2 recurrence (real A, dt on the input, initial state h_{-1},
D skip, silu(z) gate) the same unrolling gives

    y_t = sum_{s<=t} (C_t . B_s) exp(sum_{u=s+1}^{t} dt_u A) dt_s x_s
          + exp(sum_{u=0}^{t} dt_u A) C_t . h_{-1}  +  D x_t ,       then * silu(z_t)
    final = exp(sum_{u} dt_u A) h_{-1} + sum_s exp(sum_{u>s} dt_u A) dt_s x_s (outer) B_s

This module evaluates that formula directly: it builds the full T x T decay
matrix per (sequence, head), with no chunking and no recurrence, so it is an
independent check on the sequential loop (pinned against it in
tests/test_oracle_pins.py, and through torch autograd against the adjoint in
tests/test_oracle_grad.py).  Sizes: tiny inputs only (T up to a few hundred).
"""
import numpy as np


def _softplus(v):
    return np.where(v > 0, v + np.log1p(np.exp(-np.abs(v))), np.log1p(np.exp(np.minimum(v, 0.0))))


def forward(x, dt_raw, A, B, C, D=None, z=None, dt_bias=None, init=None, cu=None):
    """Float64 quadratic form; same array conventions as ``oracle.sequential``."""
    x = np.asarray(x, np.float64)
    T, H, P = x.shape
    B = np.asarray(B, np.float64)
    C = np.asarray(C, np.float64)
    G, N = B.shape[1], B.shape[2]
    hpg = H // G
    if cu is None:
        cu = [0, T]
    cu = [int(c) for c in cu]
    S = len(cu) - 1
    v = np.asarray(dt_raw, np.float64) + (0.0 if dt_bias is None else np.asarray(dt_bias, np.float64)[None, :])
    dt = _softplus(v)                                    # [T, H]
    y = np.zeros((T, H, P))
    fin = np.zeros((S, H, P, N))
    for s in range(S):
        t0, t1 = cu[s], cu[s + 1]
        n = t1 - t0
        for h in range(H):
            g = h // hpg
            if n == 0:
                fin[s, h] = 0.0 if init is None else init[s, h]
                continue
            la = dt[t0:t1, h] * A[h]                     # log decay of each step
            seg = np.cumsum(la)                          # seg[t] = sum_{u<=t} la_u
            # decay from token s to token t (excluding step s): exp(seg[t]-seg[s]) for s<=t
            diff = seg[:, None] - seg[None, :]
            causal = np.tril(np.ones((n, n), dtype=bool))
            Lmat = np.where(causal, np.exp(np.where(causal, diff, 0.0)), 0.0)
            CB = C[t0:t1, g, :] @ B[t0:t1, g, :].T       # [t, s]
            W = CB * Lmat * dt[t0:t1, h][None, :]        # [t, s]
            yh = W @ x[t0:t1, h, :]                      # [t, p]
            wend = np.exp(seg[-1] - seg) * dt[t0:t1, h]  # decay of token s to the end
            fh = (x[t0:t1, h, :] * wend[:, None]).T @ B[t0:t1, g, :]   # [p, n]
            if init is not None:
                h0 = np.asarray(init, np.float64)[s, h]  # [P, N]
                yh = yh + np.exp(seg)[:, None] * (C[t0:t1, g, :] @ h0.T)
                fh = fh + np.exp(seg[-1]) * h0
            if D is not None:
                yh = yh + D[h] * x[t0:t1, h, :]
            if z is not None:
                zz = np.asarray(z, np.float64)[t0:t1, h, :]
                yh = yh * zz / (1.0 + np.exp(-zz))
            y[t0:t1, h, :] = yh
            fin[s, h] = fh
    return y, fin


def forward_torch(x, dt_raw, A, B, C, D=None, z=None, dt_bias=None, init=None):
    """The same closed form written with torch float64 CPU ops (one sequence).

    Used only to obtain gradients by torch autograd, independently of the
    hand-written adjoint.  Shapes: x [T,H,P], dt_raw [T,H], A/D/dt_bias [H],
    B/C [T,G,N], z [T,H,P], init [H,P,N].  Returns (y, final).
    """
    import torch
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    hpg = H // G
    v = dt_raw + (dt_bias[None, :] if dt_bias is not None else 0.0)
    dt = torch.nn.functional.softplus(v)
    ys, fins = [], []
    causal = torch.tril(torch.ones(T, T, dtype=torch.bool))
    for h in range(H):
        g = h // hpg
        la = dt[:, h] * A[h]
        seg = torch.cumsum(la, 0)
        diff = seg[:, None] - seg[None, :]
        Lmat = torch.where(causal, torch.exp(torch.where(causal, diff, torch.zeros_like(diff))), torch.zeros_like(diff))
        CB = C[:, g, :] @ B[:, g, :].T
        W = CB * Lmat * dt[:, h][None, :]
        yh = W @ x[:, h, :]
        wend = torch.exp(seg[-1] - seg) * dt[:, h]
        fh = (x[:, h, :] * wend[:, None]).T @ B[:, g, :]
        if init is not None:
            yh = yh + torch.exp(seg)[:, None] * (C[:, g, :] @ init[h].T)
            fh = fh + torch.exp(seg[-1]) * init[h]
        if D is not None:
            yh = yh + D[h] * x[:, h, :]
        if z is not None:
            yh = yh * z[:, h, :] * torch.sigmoid(z[:, h, :])
        ys.append(yh)
        fins.append(fh)
    return torch.stack(ys, 1), torch.stack(fins, 0)
