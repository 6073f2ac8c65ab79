"""Complex-A SSD scan (the Mamba-3-Lite variant) in complex128 -- TEST INFRASTRUCTURE ONLY.

Follows the Mamba-3-Lite "SSD Reference -- complex scan API & kernel contract" page:

* section "Math: the recurrence both functions implement": with the per-position decay
  abar_t = exp(softplus(dt_t) * A_h) (A a complex per-head scalar, dt real), the state
  h_t [N, D] of each (batch row, head) follows
      h_t = abar_t * h_{t-1} + B_t (outer) x_t ,     y_t = sum_n C_{t,n} h_{t,n}
  -- no dt factor on the input, no conjugation anywhere (C and B enter bilinearly);
* section "ssd_naive_complex -- the O(T) oracle": the literal walk over time, returning
  the complex output (imaginary part included);
* section "ssd_complex_chunkwise -- the production scan": pad to a multiple of the chunk
  length (zeros on x, B, C and on dt *before* softplus), the in-chunk cumulative log-decay,
  the causal decay matrix L, the intra-chunk output and the chunk's own right-edge state,
  the inter-chunk contract decay_chunk[z, c] = exp(CD[z-1] - CD[c]) 1[z > c] plus the
  initial-state term exp(CD[z-1]) H_{-1}, the readout exp(A_cumsum[l]) C_l . G_z, and the
  real part sliced back to the true length.  Its tensor-shape table fixes the state
  layout [D, N] ("P before N") of initial_states.

Layouts (complex128 NumPy): x [Bt, T, H, D]; B, C [Bt, T, H, N] (one projection per
head); dt [Bt, T, H] real; A [H] complex; states [Bt, H, D, N].

Pins (tests/test_oracle_complex.py): the hand-computed geometric series of
tests/golden/complex_ssd.txt; chunkwise == naive for chunk lengths 1, 2, 4, 16 and the
whole sequence with time-varying dt and an initial state; the real special case against
the independent float64 C oracle of the real recurrence; bilinear phase invariance,
conjugation symmetry, linearity in x, and bit-exact split invariance of the walk; a
planted one-chunk-too-long propagation window must fail.
"""
import numpy as np


def softplus(v):
    """log(1 + e^v), evaluated without overflow."""
    v = np.asarray(v, dtype=np.float64)
    return np.maximum(v, 0.0) + np.log1p(np.exp(-np.abs(v)))


def discretise(dt, A):
    """abar = exp(softplus(dt) * A) for dt [..., H] (real) and A [H] (complex)."""
    return np.exp(softplus(dt) * np.asarray(A, dtype=np.complex128))


def naive(x, A, B, C, dt, init=None):
    """The O(T) walk.  Returns (y [Bt, T, H, D] complex, final [Bt, H, D, N] complex),
    final being the state after the last token."""
    x = np.asarray(x, dtype=np.complex128)
    B = np.asarray(B, dtype=np.complex128)
    C = np.asarray(C, dtype=np.complex128)
    Bt, T, H, D = x.shape
    N = B.shape[-1]
    abar = discretise(dt, A)                                   # [Bt, T, H]
    h = np.zeros((Bt, H, N, D), dtype=np.complex128)           # state as [N, D] per head
    if init is not None:
        h = h + np.swapaxes(np.asarray(init, dtype=np.complex128), -1, -2)
    y = np.zeros((Bt, T, H, D), dtype=np.complex128)
    for t in range(T):
        h = abar[:, t, :, None, None] * h + B[:, t, :, :, None] * x[:, t, :, None, :]
        y[:, t] = (C[:, t, :, :, None] * h).sum(axis=-2)
    return y, np.swapaxes(h, -1, -2).copy()


def chunkwise(x, A, B, C, dt, Q, init=None, _window_shift=1):
    """The chunkwise decomposition in the page's order; returns Re(y) [Bt, T, H, D].

    ``_window_shift`` exists only so a test can plant the one-chunk-too-long window
    (CD[z] - CD[c]); the contract is 1 (CD[z-1] - CD[c])."""
    x = np.asarray(x, dtype=np.complex128)
    B = np.asarray(B, dtype=np.complex128)
    C = np.asarray(C, dtype=np.complex128)
    dt = np.asarray(dt, dtype=np.float64)
    A = np.asarray(A, dtype=np.complex128)
    Bt, T, H, D = x.shape
    N = B.shape[-1]
    pad = (Q - T % Q) % Q
    if pad:
        x = np.concatenate([x, np.zeros((Bt, pad, H, D))], axis=1)
        B = np.concatenate([B, np.zeros((Bt, pad, H, N))], axis=1)
        C = np.concatenate([C, np.zeros((Bt, pad, H, N))], axis=1)
        dt = np.concatenate([dt, np.zeros((Bt, pad, H))], axis=1)
    nc = (T + pad) // Q
    y = np.zeros((Bt, T + pad, H, D))
    for b in range(Bt):
        for h in range(H):
            a_log = softplus(dt[b, :, h]) * A[h]               # complex log-decay per position
            S = []                                             # each chunk's own right-edge state [D, N]
            lam = []                                           # each chunk's total log-decay
            ydiag = []
            cum = []
            for c in range(nc):
                sl = slice(c * Q, (c + 1) * Q)
                Xc, Bc, Cc = x[b, sl, h], B[b, sl, h], C[b, sl, h]
                cs = np.cumsum(a_log[sl])
                Lm = np.zeros((Q, Q), dtype=np.complex128)
                for l in range(Q):
                    for s in range(l + 1):
                        Lm[l, s] = np.exp(cs[l] - cs[s])
                ydiag.append((Lm * (Cc @ Bc.T)) @ Xc)
                decay_states = np.exp(cs[-1] - cs)
                S.append((Xc * decay_states[:, None]).T @ Bc)
                lam.append(cs[-1])
                cum.append(cs)
            CD = np.cumsum(np.array(lam))
            for z in range(nc):
                cd_prev = CD[z - _window_shift] if z - _window_shift >= 0 else 0.0
                G = np.zeros((D, N), dtype=np.complex128)
                for c in range(z):
                    G += np.exp(cd_prev - CD[c]) * S[c]
                if init is not None:
                    G += np.exp(cd_prev) * np.asarray(init[b, h], dtype=np.complex128)
                sl = slice(z * Q, (z + 1) * Q)
                yoff = np.exp(cum[z])[:, None] * (C[b, sl, h] @ G.T)
                y[b, sl, h] = (ydiag[z] + yoff).real
    return y[:, :T]
