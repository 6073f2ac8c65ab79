"""The split tensor-core forward (SSD_ALGO_SPLIT: chunk states, state passing and outputs
as three launches) against the float64 oracle (GPU): fixed-length batches, packed
sequences on grids whose chunks span sequences, head subsets of large groups, kept chunk
states and the backward that uses its state recompute."""
import numpy as np
import pytest
import torch

from state_space_model_scan_gb300 import inputs as I
from state_space_model_scan_gb300.api import ssd_forward
from helpers import TOL, rel_l2, gpu_forward, gpu_backward, oracle_forward, oracle_backward, flat, to_dev

pytestmark = pytest.mark.gpu


def W(B=1, L=300, H=8, G=2, **kw):
    return I.Workload("sp", B, L, H, 64, G, 128, 128, "bf16", **kw)


@pytest.mark.parametrize("w", [
    W(L=1000, has_z=True, has_init=True),
    W(B=2, L=333, H=4, G=1, has_z=False),
    W(L=1, H=2, G=1, has_init=True),
    W(B=3, L=129, H=6, G=2, has_D=False, has_dt_bias=False),          # 3 heads per group
    W(L=700, H=32, G=1, has_z=True, has_init=True),                   # 32 heads per group: subsets of 8
    I.Workload("spv", 1, 902, 8, 64, 2, 128, 128, "bf16", has_z=True, has_init=True,
               seqlens=[3, 200, 1, 0, 129, 127, 442]),               # chunks spanning sequences
], ids=lambda w: "B%d_L%d_H%d_G%d%s" % (w.batch, w.seqlen, w.nheads, w.ngroups, "_varlen" if w.seqlens else ""))
def test_split_forward_matches_oracle(w):
    inp = I.make_inputs(w)
    y, fin = gpu_forward(w, inp, algo="split")
    yo, fo = oracle_forward(w, inp)
    assert np.isfinite(flat(y, w.batch * w.seqlen)).all()
    assert rel_l2(flat(y, w.batch * w.seqlen), yo) <= TOL["bf16"]
    assert rel_l2(fin.double().cpu().numpy(), fo) <= TOL["bf16"]


def test_split_and_single_pass_agree():
    """Same function, same chunking: the two tensor-core forwards agree closely, and the
    split one is deterministic run to run."""
    w = W(L=1500, has_z=True, has_init=True)
    inp = I.make_inputs(w)
    y1, f1 = gpu_forward(w, inp, algo="split")
    y2, f2 = gpu_forward(w, inp, algo="fused")
    y3, f3 = gpu_forward(w, inp, algo="split")
    assert torch.equal(y1, y3) and torch.equal(f1, f3)
    assert rel_l2(y1.double().cpu(), y2.double().cpu()) < 5e-3
    assert rel_l2(f1.double().cpu(), f2.double().cpu()) < 5e-3


def test_split_kept_states_feed_the_backward():
    """The split forward keeps the carried states in the tile format the backward reads."""
    w = W(L=700, has_z=True, has_init=True)
    inp = I.make_inputs(w, with_grad_inputs=True, with_dfinal=True)
    d = to_dev(inp)
    _, _, cs = ssd_forward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                           initial_states=d["initial_states"], chunk_size=128, keep_chunk_states=True, algo="split")
    g = gpu_backward(w, inp, chunk_states=cs)
    o = oracle_backward(w, inp)
    for gn, on in (("dx", "dx"), ("dB", "dB"), ("dC", "dC"), ("ddt", "ddt_raw"), ("dz", "dz")):
        assert rel_l2(flat(g[gn], w.seqlen), o[on]) <= TOL["bf16"], gn
    assert rel_l2(g["dinitial_states"].double().cpu().numpy(), o["dinit"]) <= TOL["bf16"]


@pytest.mark.parametrize("lens", [None, [40, 0, 130, 1, 270, 128]])
def test_split_backward_recompute(lens):
    """The backward without kept states, its carried states recomputed by the split forward's
    first two launches."""
    if lens is None:
        w = W(L=640, has_z=True, has_init=True)
    else:
        w = I.Workload("spb", 1, sum(lens), 4, 64, 2, 128, 128, "bf16", has_z=True, has_init=True, seqlens=lens)
    inp = I.make_inputs(w, with_grad_inputs=True, with_dfinal=True)
    g = gpu_backward(w, inp, algo="split")
    o = oracle_backward(w, inp)
    T = w.batch * w.seqlen
    for gn, on in (("dx", "dx"), ("dB", "dB"), ("dC", "dC"), ("ddt", "ddt_raw"), ("dz", "dz")):
        assert rel_l2(flat(g[gn], T), o[on]) <= TOL["bf16"], gn
    for gn, on in (("dA", "dA"), ("dD", "dD"), ("dinitial_states", "dinit")):
        assert rel_l2(g[gn].double().cpu().numpy(), o[on]) <= TOL["bf16"], gn
