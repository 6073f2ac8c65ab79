"""Chunkwise decomposition of the SSD in float64 -- TEST INFRASTRUCTURE ONLY.

Restates, for the real Mamba-2 recurrence (dt on the input, initial state, D,
silu(z)), the chunkwise path of the Mamba-3-Lite "SSD Reference" page
(section "ssd_complex_chunkwise -- the production scan"):

1. Padding rule: the sequence is right-padded to a multiple of the chunk
   length Q.  Here the pad is applied *after* softplus with dt := 0 (decay 1,
   zero input), so padding never changes real outputs or the final state.
2. Chunking and the discretised log-decay: dA = dt * A, A_cumsum = inclusive
   cumulative sum inside each chunk, decay_states[l] = exp(A_cumsum[Q-1] - A_cumsum[l]).
3. Intra-chunk outputs and chunk states: L[l, s] = exp(A_cumsum[l] - A_cumsum[s]) 1[l >= s];
   Y_diag = (L o (C B^T) o dt_s) X ;  S_c = X^T (decay_states o dt o B)   (state [P, N]).
4. Inter-chunk propagation: with CD[k] = sum_{u<=k} Lambda_u (Lambda = chunk total
   log-decay) and CD[-1] := 0, the carry-in state of chunk z is
       G_z = sum_{c<z} exp(CD[z-1] - CD[c]) S_c + exp(CD[z-1]) H_{-1}
   (the page's "fixed contract" decay_chunk[z, c] = exp(CD[z-1] - CD[c]) 1[z > c],
   and the initial-state term that decays one chunk longer than any S_c).
5. Readout: Y_off[l] = exp(A_cumsum[l]) C_l . G_z ; Y = Y_diag + Y_off (+ D x), gated,
   then sliced back to the real length.

The final state is the carry-in of the (virtual) chunk after the last one.
Pinned by chunk-size invariance against the sequential oracle for Q in
{1, 2, 4, 16, 64, T} with time-varying dt (tests/test_oracle_pins.py); Q=1 is
the sequential scan and Q=T the quadratic form.
"""
import numpy as np


def _softplus(v):
    return np.where(v > 0, v + np.log1p(np.exp(-np.abs(v))), np.log1p(np.exp(np.minimum(v, 0.0))))


def forward_one(x, dt, A, B, C, Q, init=None):
    """One sequence, one head.  x [T,P], dt [T] (post-softplus), A scalar,
    B/C [T,N], init [P,N] or None.  Returns (y_pre_without_D [T,P], final [P,N], inter)
    where ``inter`` holds the chunk intermediates (padded): dt, cs [n_c,Q],
    chunk_states [n_c,P,N], carry_in [n_c,P,N]."""
    T, P = x.shape
    N = B.shape[1]
    n_c = max(1, -(-T // Q))
    pad = n_c * Q - T
    xp = np.concatenate([x, np.zeros((pad, P))], 0).reshape(n_c, Q, P)
    Bp = np.concatenate([B, np.zeros((pad, N))], 0).reshape(n_c, Q, N)
    Cp = np.concatenate([C, np.zeros((pad, N))], 0).reshape(n_c, Q, N)
    dtp = np.concatenate([dt, np.zeros(pad)], 0).reshape(n_c, Q)
    dA = dtp * A
    cs = np.cumsum(dA, axis=1)                                  # A_cumsum
    decay_states = np.exp(cs[:, -1:] - cs)                      # [n_c, Q]
    causal = np.tril(np.ones((Q, Q), dtype=bool))
    Y_diag = np.zeros((n_c, Q, P))
    states = np.zeros((n_c, P, N))
    for c in range(n_c):
        seg = cs[c][:, None] - cs[c][None, :]
        Lm = np.where(causal, np.exp(np.where(causal, seg, 0.0)), 0.0)
        CB = Cp[c] @ Bp[c].T
        Y_diag[c] = (Lm * CB * dtp[c][None, :]) @ xp[c]
        states[c] = (xp[c] * (decay_states[c] * dtp[c])[:, None]).T @ Bp[c]
    Lam = cs[:, -1]                                             # chunk total log-decay
    CD = np.cumsum(Lam)
    CDm1 = np.concatenate([[0.0], CD[:-1]])                     # CD[z-1], CD[-1] = 0
    carry = np.zeros((n_c, P, N))
    for zc in range(n_c):
        acc = np.zeros((P, N))
        for c in range(zc):
            acc += np.exp(CDm1[zc] - CD[c]) * states[c]
        if init is not None:
            acc += np.exp(CDm1[zc]) * init
        carry[zc] = acc
    Y_off = np.zeros((n_c, Q, P))
    for c in range(n_c):
        Y_off[c] = np.exp(cs[c])[:, None] * (Cp[c] @ carry[c].T)
    # final state: carry-in of the chunk after the last one
    fin = np.zeros((P, N))
    for c in range(n_c):
        fin += np.exp(CD[-1] - CD[c]) * states[c]
    if init is not None:
        fin += np.exp(CD[-1]) * init
    y = (Y_diag + Y_off).reshape(n_c * Q, P)[:T]
    inter = dict(dt=dtp, cs=cs, chunk_states=states, carry_in=carry)
    return y, fin, inter


def forward(x, dt_raw, A, B, C, Q, D=None, z=None, dt_bias=None, init=None, cu=None):
    """Chunked float64 forward over all sequences/heads; same conventions as
    ``oracle.sequential.forward`` plus the chunk length ``Q``."""
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
    dt = _softplus(v)
    y = np.zeros((T, H, P))
    fin = np.zeros((S, H, P, N))
    for s in range(S):
        t0, t1 = cu[s], cu[s + 1]
        for h in range(H):
            g = h // hpg
            h0 = None if init is None else np.asarray(init, np.float64)[s, h]
            if t1 == t0:
                fin[s, h] = 0.0 if h0 is None else h0
                continue
            yh, fh, _ = forward_one(x[t0:t1, h], dt[t0:t1, h], float(A[h]), B[t0:t1, g], C[t0:t1, g], Q, h0)
            if D is not None:
                yh = yh + D[h] * x[t0:t1, h]
            if z is not None:
                zz = np.asarray(z, np.float64)[t0:t1, h]
                yh = yh * zz / (1.0 + np.exp(-zz))
            y[t0:t1, h] = yh
            fin[s, h] = fh
    return y, fin
