"""bf16 storage of the initial/final states and their gradients: the kernels widen bf16
inputs and compute in fp32, so a bf16 run equals the fp32 run on the same rounded state
values exactly (y and every gradient bitwise, the bf16 outputs = the fp32 ones rounded to
nearest even), on every path; and against the float64 oracle on the rounded values."""
import pytest
import torch

from state_space_model_scan_gb300 import inputs as I
from helpers import TOL, rel_l2, gpu_forward, gpu_backward, oracle_forward, oracle_backward, flat

pytestmark = pytest.mark.gpu

CASES = {
    "fused": I.Workload("sf", 2, 700, 8, 64, 2, 128, 128, "bf16", has_z=True, has_init=True),
    "split": I.Workload("ss", 1, 900, 8, 64, 4, 128, 128, "bf16", has_z=True, has_init=True),
    "staged": I.Workload("st", 1, 333, 4, 32, 2, 64, 64, "f32", has_z=True, has_init=True),
    "varlen": I.Workload("sv", 1, 600, 4, 64, 2, 128, 128, "bf16", has_z=False, has_init=True,
                         seqlens=[150, 0, 200, 1, 249]),
}


def rounded_inputs(w, with_grad=False):
    inp = I.make_inputs(w, with_grad_inputs=with_grad, with_dfinal=with_grad)
    inp["initial_states"] = inp["initial_states"].to(torch.bfloat16).float()
    if with_grad:
        inp["dfinal_states"] = inp["dfinal_states"].to(torch.bfloat16).float()
    return inp


def as_bf16_states(inp):
    out = dict(inp)
    out["initial_states"] = inp["initial_states"].to(torch.bfloat16)
    if inp.get("dfinal_states") is not None:
        out["dfinal_states"] = inp["dfinal_states"].to(torch.bfloat16)
    return out


@pytest.mark.parametrize("case", list(CASES))
def test_bf16_states_forward(case):
    w = CASES[case]
    algo = "split" if case == "split" else "auto"
    inp = rounded_inputs(w)
    y32, f32 = gpu_forward(w, inp, algo=algo)
    y16, f16 = gpu_forward(w, as_bf16_states(inp), algo=algo)
    assert f16.dtype == torch.bfloat16
    assert torch.equal(y16, y32)
    assert torch.equal(f16, f32.to(torch.bfloat16))
    yo, fo = oracle_forward(w, inp)
    assert rel_l2(flat(y16, w.tokens), yo) <= TOL[w.dtype]
    assert rel_l2(f16.double().cpu().numpy(), fo) <= TOL["bf16"]


@pytest.mark.parametrize("case", ["fused", "staged", "varlen"])
def test_bf16_states_backward(case):
    w = CASES[case]
    inp = rounded_inputs(w, with_grad=True)
    g32 = gpu_backward(w, inp)
    g16 = gpu_backward(w, as_bf16_states(inp))
    assert g16["dinitial_states"].dtype == torch.bfloat16
    for k in g32:
        if k == "dinitial_states":
            assert torch.equal(g16[k], g32[k].to(torch.bfloat16))
        else:
            assert torch.equal(g16[k], g32[k]), k
    go = oracle_backward(w, inp)
    assert rel_l2(g16["dinitial_states"].double().cpu().numpy(), go["dinit"]) <= TOL["bf16"]
