"""Complex-A SSD forward (tensor cores, tf32) against the complex128 oracle walk.

Tolerance: rel-L2 <= 5e-3 per output.  The contractions take tf32 operands (10-bit
mantissa, truncated: up to 2^-10 relative per operand, biased towards zero), three chained
contractions (C B^T, then (L o Cb) X, and C S^T through the carried state) give a few times
2^-10 ~ 1e-3 in the worst direction (measured 1.5e-3); the carried state, the decays and the
accumulation are fp32."""
import numpy as np
import pytest
import torch

from oracle import complex_ssd as cx
from state_space_model_scan_gb300 import inputs as I
from state_space_model_scan_gb300.api import complex_ssd_forward

pytestmark = pytest.mark.gpu
TOL = 5e-3


def rel(a, b):
    return float(np.linalg.norm(np.ravel(a - b)) / max(np.linalg.norm(np.ravel(b)), 1e-300))


def npc(t):
    return None if t is None else t.cpu().numpy().astype(np.complex128)


def run(inp, **kw):
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    out = complex_ssd_forward(d["x"], d["A"], d["B"], d["C"], d["dt"], initial_states=d["initial_states"],
                              return_imag=True, return_final=True, **kw)
    torch.cuda.synchronize()
    return [o.cpu() for o in out]


def oracle(inp, b=None, h=None):
    sel = lambda t: t if b is None else t[b:b + 1, :, h:h + 1]
    x, B, C = npc(sel(inp["x"])), npc(sel(inp["B"])), npc(sel(inp["C"]))
    dt = sel(inp["dt"]).double().numpy()
    A = npc(inp["A"]) if h is None else npc(inp["A"][h:h + 1])
    init = None
    if inp["initial_states"] is not None:
        init = npc(inp["initial_states"]) if b is None else npc(inp["initial_states"][b:b + 1, h:h + 1])
    return cx.naive(x, A, B, C, dt, init=init)


@pytest.mark.parametrize("Bt,T,H,init", [(1, 1, 1, True), (2, 64, 2, False), (1, 200, 3, True), (2, 130, 2, True),
                                         (1, 640, 1, True)])
def test_complex_matches_oracle(Bt, T, H, init):
    inp = I.complex_inputs(Bt, T, H, seed=T + H, with_init=init)
    y_re, y_im, fin = run(inp)
    y, f = oracle(inp)
    assert rel(y_re.double().numpy(), y.real) <= TOL
    assert rel(y_im.double().numpy(), y.imag) <= TOL
    assert rel(npc(fin), f) <= TOL


def test_complex_434m_shape_sampled_heads():
    """8 x 2048 tokens x 16 heads (the 434M Mamba-3-Lite configuration): whole-kernel run,
    (batch row, head) pairs checked one by one against the oracle walk."""
    inp = I.complex_inputs(8, 2048, 16, seed=434)
    y_re, y_im, fin = run(inp)
    for b, h in [(0, 0), (3, 7), (7, 15), (5, 2)]:
        y, f = oracle(inp, b, h)
        assert rel(y_re[b:b + 1, :, h:h + 1].double().numpy(), y.real) <= TOL
        assert rel(y_im[b:b + 1, :, h:h + 1].double().numpy(), y.imag) <= TOL
        assert rel(npc(fin[b:b + 1, h:h + 1]), f) <= TOL


def test_complex_empty_sequence_returns_initial_state():
    inp = I.complex_inputs(2, 0, 3, seed=1)
    _, _, fin = run(inp)
    assert torch.equal(fin, inp["initial_states"])


def test_complex_real_special_case_has_no_imaginary_part():
    inp = I.complex_inputs(1, 150, 2, seed=3)
    for k in ("x", "B", "C", "initial_states"):
        inp[k] = torch.complex(inp[k].real, torch.zeros_like(inp[k].real))
    inp["A"] = torch.complex(inp["A"].real, torch.zeros_like(inp["A"].real))
    y_re, y_im, fin = run(inp)
    y, f = oracle(inp)
    assert float(y_im.abs().max()) == 0.0
    assert rel(y_re.double().numpy(), y.real) <= TOL


def test_complex_split_sequence():
    """Running [0, T1) then [T1, T) from the returned state equals the whole run (split off the chunk grid)."""
    inp = I.complex_inputs(1, 300, 2, seed=4)
    y_re, y_im, fin = run(inp)
    T1 = 137
    a = {k: (v[:, :T1] if k in ("x", "B", "C", "dt") else v) for k, v in inp.items()}
    y1, _, f1 = run(a)
    b = {k: (v[:, T1:] if k in ("x", "B", "C", "dt") else v) for k, v in inp.items()}
    b["initial_states"] = f1.to(torch.complex64)
    y2, _, f2 = run(b)
    assert rel(torch.cat([y1, y2], 1).double().numpy(), y_re.double().numpy()) <= TOL
    assert rel(npc(f2), npc(fin)) <= TOL


def test_complex_deterministic():
    inp = I.complex_inputs(2, 333, 4, seed=5)
    r1 = run(inp)
    r2 = run(inp)
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)


@pytest.mark.parametrize("T", [63, 65, 127, 129])
def test_complex_chunk_boundaries(T):
    """One token short of / past a chunk edge (the last chunk's rows past T are never stored)."""
    inp = I.complex_inputs(1, T, 2, seed=T)
    y_re, y_im, fin = run(inp)
    y, f = oracle(inp)
    assert rel(y_re.double().numpy(), y.real) <= TOL
    assert rel(y_im.double().numpy(), y.imag) <= TOL
    assert rel(npc(fin), f) <= TOL


@pytest.mark.parametrize("want_final", [True, False])
def test_complex_real_output_only(want_final):
    """Re y alone (the second MMA chain is then waited for by the state update only), with and
    without the final state."""
    inp = I.complex_inputs(2, 200, 2, seed=21)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    out = complex_ssd_forward(d["x"], d["A"], d["B"], d["C"], d["dt"], initial_states=d["initial_states"],
                              return_imag=False, return_final=want_final)
    torch.cuda.synchronize()
    y_re = out[0] if isinstance(out, (tuple, list)) else out
    y, f = oracle(inp)
    assert rel(y_re.cpu().double().numpy(), y.real) <= TOL
    if want_final:
        assert rel(npc(out[-1].cpu()), f) <= TOL


@pytest.mark.parametrize("regime", ["strong_decay", "weak_decay", "fast_rotation", "softplus_switch", "far_negative"])
def test_complex_decay_regimes(regime):
    """Decay and timestep regimes: Re A = -16 with dt near 3 (abar ~ e^-48 per step: every
    chunk forgets its past), Re A = -1e-4 (the state keeps everything), |Im A| = 3 pi (the
    phase turns by more than a half-turn per step), raw dt straddling softplus's switch at 20
    and raw dt near -30 (dt underflows towards 0)."""
    H, T = 3, 200
    inp = I.complex_inputs(1, T, H, seed=31)
    g = torch.Generator().manual_seed(77)
    A = inp["A"]
    dt = inp["dt"]
    if regime == "strong_decay":
        A = torch.complex(torch.full((H,), -16.0), A.imag)
        dt = 3.0 + 0.1 * torch.randn(1, T, H, generator=g)
    elif regime == "weak_decay":
        A = torch.complex(torch.full((H,), -1e-4), A.imag)
    elif regime == "fast_rotation":
        A = torch.complex(A.real, torch.tensor([3 * np.pi, -3 * np.pi, 2.5 * np.pi]))
    elif regime == "softplus_switch":
        vals = torch.tensor([19.9, 20.0, 20.1, 40.0])
        dt = vals[torch.randint(0, 4, (1, T, H), generator=g)]
        A = torch.complex(torch.full((H,), -0.05), A.imag)
    else:
        dt = -30.0 + torch.randn(1, T, H, generator=g)
    inp["A"] = A.to(torch.complex64)
    inp["dt"] = dt.to(torch.float32)
    y_re, y_im, fin = run(inp)
    y, f = oracle(inp)
    assert np.isfinite(y_re.numpy()).all() and np.isfinite(y_im.numpy()).all()
    assert rel(y_re.double().numpy(), y.real) <= TOL
    assert rel(y_im.double().numpy(), y.imag) <= TOL
    assert rel(npc(fin), f) <= TOL


def test_complex_more_rows_than_sms():
    """3 x 70 (batch row, head) pairs: more CTAs than SMs, each still one walk."""
    inp = I.complex_inputs(3, 70, 70, seed=41)
    y_re, y_im, fin = run(inp)
    y, f = oracle(inp)
    assert rel(y_re.double().numpy(), y.real) <= TOL
    assert rel(y_im.double().numpy(), y.imag) <= TOL
    assert rel(npc(fin), f) <= TOL
