"""Parity at the edges of the scan's parameter ranges (GPU), per head against the
float64 oracle, on the tensor-core and the SIMT paths, forward and backward.

The regimes the cuDNN frontend's Mamba-2 SSD engine validates ("Validation": strong,
zero and weak-positive recurrence rates; timestep values near the softplus branches
and in its negative tail), one per head so that each head's rel-L2 checks one regime:
  0  dt_raw + dt_bias straddling softplus's large-argument switch: 19.9, 20, 20.1, 40
  1  the far-negative tail: dt_raw + dt_bias around -30 (dt ~ 1e-13, the state barely moves)
  2  A = 0 (no decay: causal linear attention without normalisation)
  3  weak-positive A = +0.05 (a slowly growing state; short sequences only)
  4  the strongest decay of the workloads: A = -16 with dt = 0.3 on every token
  5, 6, 7  the workloads' own distributions
Token-level outputs and states are compared per head (rel-L2 of that head); where a
head's reference is below fp32's range (the initial-state gradient of head 0, whose
state decays by exp(-20 |A|) or more at the first step) the error is taken relative to
the whole tensor's norm; per-head scalars (dA, dD, ddt_bias) relative to their largest
reference value (the peak-normalised error the cuDNN engine's validation reports).
"""
import numpy as np
import pytest
import torch

from state_space_model_scan_gb300 import inputs as I
from helpers import TOL, rel_l2, gpu_forward, gpu_backward, oracle_forward, oracle_backward, flat

pytestmark = pytest.mark.gpu

H = 8


def edge_inputs(w, with_grad=False):
    inp = I.make_inputs(w, with_grad_inputs=with_grad, with_dfinal=with_grad)
    bias = inp["dt_bias"]
    L = w.seqlen
    t = torch.arange(L)
    v = (inp["dt_raw"] + bias[None, None, :]).clone()
    v[:, :, 0] = torch.tensor([19.9, 20.0, 20.1, 40.0])[t % 4]
    v[:, :, 1] = -30.0 + 0.5 * torch.sin(t.float())
    v[:, :, 4] = float(np.log(np.expm1(0.3)))            # softplus(v) = 0.3
    inp["dt_raw"] = (v - bias[None, None, :]).to(torch.float32)
    A = inp["A"].clone()
    A[2] = 0.0
    A[3] = 0.05
    A[4] = -16.0
    inp["A"] = A
    return inp


def cases():
    # (dtype, P, N, G, chunk, algo)
    return [("bf16", 64, 128, 2, 128, "fused"), ("bf16", 64, 128, 2, 64, "staged"), ("f32", 16, 16, 2, 64, "staged")]


def W(dtype, P, N, G, Q, L=300, B=1):
    return I.Workload("edge", B, L, H, P, G, N, Q, dtype, has_z=True, has_D=True, has_init=True)


@pytest.mark.parametrize("dtype,P,N,G,Q,algo", cases())
def test_edge_regimes_forward(dtype, P, N, G, Q, algo):
    w = W(dtype, P, N, G, Q)
    inp = edge_inputs(w)
    y, fin = gpu_forward(w, inp, algo=algo)
    yo, fo = oracle_forward(w, inp)
    yg, fg = flat(y, w.seqlen), fin.double().cpu().numpy()
    assert np.isfinite(yg).all() and np.isfinite(fg).all()
    errs = {h: (rel_l2(yg[:, h], yo[:, h]), rel_l2(fg[:, h], fo[:, h])) for h in range(H)}
    bad = {h: e for h, e in errs.items() if not (e[0] <= TOL[dtype] and e[1] <= TOL[dtype])}
    assert not bad, errs


@pytest.mark.parametrize("dtype,P,N,G,Q,algo", cases())
def test_edge_regimes_backward(dtype, P, N, G, Q, algo):
    w = W(dtype, P, N, G, Q, L=200)
    inp = edge_inputs(w, with_grad=True)
    g = gpu_backward(w, inp, algo=algo)
    o = oracle_backward(w, inp)
    T = w.seqlen
    errs = {}
    for h in range(H):
        for gn, on in (("dx", "dx"), ("dz", "dz"), ("ddt", "ddt_raw")):
            errs[(h, gn)] = rel_l2(flat(g[gn], T)[:, h], o[on][:, h])
        gi = g["dinitial_states"].double().cpu().numpy()
        errs[(h, "dinit")] = float(np.linalg.norm(gi[:, h] - o["dinit"][:, h]) / np.linalg.norm(o["dinit"]))
    for gn, on in (("dA", "dA"), ("dD", "dD"), ("ddt_bias", "ddt_bias")):
        a = g[gn].double().cpu().numpy()
        errs[gn] = rel_l2(a, o[on])
        for h in range(H):   # per-head scalars, peak-normalised
            errs[(h, gn)] = abs(a[h] - o[on][h]) / np.abs(o[on]).max()
    for gn in ("dB", "dC"):   # summed over the heads of a group: every regime's share inside
        errs[gn] = rel_l2(flat(g[gn], T), o[gn])
    tol = TOL[dtype]
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, bad
