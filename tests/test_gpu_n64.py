"""dstate 64, 32 and 16 (headdim 64, bf16) on the tensor-core path: the N = 128 tiles compute
them as their zero-extended part (TMA fills B/C past the caller's dstate with zeros; the states
are padded copies; dB/dC stores are clipped to the caller's columns), so the results are those
of the smaller problem.  Forward (single-pass and split), packed
sequences, kept chunk states, backward (whole-group items and head subsets), bf16 states,
against the float64 oracle."""
import pytest
import torch

from state_space_model_scan_gb300 import inputs as I
from state_space_model_scan_gb300 import _lib
from state_space_model_scan_gb300.api import ssd_forward
from helpers import TOL, rel_l2, gpu_forward, gpu_backward, oracle_forward, oracle_backward, flat, to_dev

pytestmark = pytest.mark.gpu


def W(B=1, L=700, H=8, G=2, N=64, **kw):
    kw.setdefault("has_init", True)
    return I.Workload("n%d" % N, B, L, H, 64, G, N, 128, "bf16", **kw)


def on_tensor_cores(w, inp):
    d = to_dev(inp)
    prob = _lib.problem(w.batch, w.seqlen, w.nheads, 64, w.ngroups, w.dstate, 128,
                        w.nseqs if d["cu_seqlens"] is not None else 0)
    y = torch.empty_like(d["x"])
    args = _lib.fwd_args(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], y, D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                         initial_states=d["initial_states"], cu_seqlens=d["cu_seqlens"])
    return _lib.chunk_states_size(prob, args) > 0   # the tensor-core path's kept-state format only


@pytest.mark.parametrize("N", [64, 32, 16])
@pytest.mark.parametrize("algo", ["auto", "split"])
@pytest.mark.parametrize("B,L,lens", [(2, 700, None), (1, 0, [130, 0, 300, 1, 269])])
def test_n64_forward(algo, B, L, lens, N):
    w = W(B=B, L=sum(lens) if lens else L, seqlens=lens, N=N)
    inp = I.make_inputs(w)
    assert on_tensor_cores(w, inp)
    y, fin = gpu_forward(w, inp, algo=algo)
    yo, fo = oracle_forward(w, inp)
    assert rel_l2(flat(y, w.tokens), yo) <= TOL["bf16"]
    assert rel_l2(fin.double().cpu().numpy(), fo) <= TOL["bf16"]


@pytest.mark.parametrize("N", [64, 32, 16])
@pytest.mark.parametrize("H,G", [(8, 2), (16, 1)])   # 4 heads per group; 16 (head subsets + reduction)
@pytest.mark.parametrize("kept", [False, True])
def test_n64_backward(H, G, kept, N):
    w = W(B=1, L=520, H=H, G=G, has_z=True, N=N)
    inp = I.make_inputs(w, with_grad_inputs=True, with_dfinal=True)
    kw = {}
    if kept:
        d = to_dev(inp)
        _, _, cs = ssd_forward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                               initial_states=d["initial_states"], chunk_size=128, keep_chunk_states=True)
        kw["chunk_states"] = cs
    g = gpu_backward(w, inp, **kw)
    o = oracle_backward(w, inp)
    T = w.tokens
    for k, ok in [("dx", "dx"), ("dz", "dz"), ("ddt", "ddt_raw"), ("dB", "dB"), ("dC", "dC")]:
        assert rel_l2(flat(g[k], T), o[ok]) <= TOL["bf16"], k
    for k, ok in [("dA", "dA"), ("dD", "dD"), ("ddt_bias", "ddt_bias"), ("dinitial_states", "dinit")]:
        assert rel_l2(g[k].double().cpu().numpy(), o[ok]) <= TOL["bf16"], k


def test_n64_bf16_states_match_fp32_states():
    w = W(B=2, L=400)
    inp = I.make_inputs(w)
    inp["initial_states"] = inp["initial_states"].to(torch.bfloat16).float()
    y32, f32 = gpu_forward(w, inp)
    b16 = dict(inp, initial_states=inp["initial_states"].to(torch.bfloat16))
    y16, f16 = gpu_forward(w, b16)
    assert torch.equal(y16, y32) and torch.equal(f16, f32.to(torch.bfloat16))
