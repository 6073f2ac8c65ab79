"""Parity at the full sizes of the benchmarked workloads, in the launch
configuration bench.py times (AUTO path, default work units).  The float64
oracle computes a sample of heads (heads are independent, so each sampled head
is an exact reference for that head's outputs and final state)."""
import dataclasses

import numpy as np
import pytest
import torch

from state_space_model_scan_gb300 import inputs as I
from helpers import TOL, rel_l2, gpu_forward, gpu_backward, oracle_forward, oracle_backward, flat

pytestmark = pytest.mark.gpu


def check_sampled(w, heads):
    inp = I.make_inputs(w)
    y, fin = gpu_forward(w, inp)
    yo, fo = oracle_forward(w, inp, heads=heads)
    T = w.batch * w.seqlen
    yg = flat(y, T)[:, heads]
    fg = fin.double().cpu().numpy()[:, heads]
    assert np.isfinite(yg).all() and np.isfinite(fg).all()
    ey, ef = rel_l2(yg, yo[:, heads]), rel_l2(fg, fo[:, heads])
    assert ey <= TOL[w.dtype] and ef <= TOL[w.dtype], (w.name, ey, ef)
    return ey, ef


def test_nemotron_nano_fwd_full_size():
    """L=8192, 64 heads x 64, 8 groups, N=128, z + D, bf16."""
    check_sampled(I.named("nemotron_nano"), [0, 13, 37, 63])


@pytest.mark.parametrize("L", [1024, 8192, 32768])
def test_long_sequence_fwd_full_size(L):
    """128 heads x 64, 1 group, N=128, random initial states, final states returned."""
    check_sampled(I.named("long_seq", L), [0, 77, 127])


def test_varlen_fwd_full_size():
    """16 packed sequences, lengths U{512..8192}, 80 heads x 64, 1 group, own initial states."""
    check_sampled(I.named("varlen"), [0, 41, 79])


def test_varlen_fwd_full_size_chunk256():
    """The same packed workload at the 256-token chunks it is quoted with (the SIMT path; the
    chunk grid over the packed axis, so chunks that straddle two sequences)."""
    check_sampled(dataclasses.replace(I.named("varlen"), chunk_size=256), [0, 41, 79])


@pytest.mark.parametrize("kept", [False, True])
def test_nemotron_nano_bwd_full_size(kept):
    """fwd+bwd workload: gradients of one whole group (dB/dC sum over its 8 heads); with the
    chunk states recomputed, and kept by the forward as bench.py's training step runs it."""
    w = I.named("nemotron_nano")
    inp = I.make_inputs(w, with_grad_inputs=True)
    kw = {}
    if kept:
        from helpers import to_dev
        from state_space_model_scan_gb300.api import ssd_forward
        d = to_dev(inp)
        _, _, kw["chunk_states"] = ssd_forward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                               dt_bias=d["dt_bias"], chunk_size=w.chunk_size, keep_chunk_states=True)
    g = gpu_backward(w, inp, **kw)
    heads = list(range(8, 16))          # group 1
    o = oracle_backward(w, inp, heads=heads)
    T = w.seqlen
    errs = dict(
        dx=rel_l2(flat(g["dx"], T)[:, heads], o["dx"][:, heads]),
        dz=rel_l2(flat(g["dz"], T)[:, heads], o["dz"][:, heads]),
        ddt=rel_l2(flat(g["ddt"], T)[:, heads], o["ddt_raw"][:, heads]),
        dB=rel_l2(flat(g["dB"], T)[:, 1], o["dB"][:, 1]),
        dC=rel_l2(flat(g["dC"], T)[:, 1], o["dC"][:, 1]),
        dA=rel_l2(g["dA"].double().cpu().numpy()[heads], o["dA"][heads]),
        dD=rel_l2(g["dD"].double().cpu().numpy()[heads], o["dD"][heads]),
        ddt_bias=rel_l2(g["ddt_bias"].double().cpu().numpy()[heads], o["ddt_bias"][heads]),
    )
    bad = {k: v for k, v in errs.items() if not v <= TOL["bf16"]}
    assert not bad, errs


def test_long_sequence_bwd_one_group_of_128_heads():
    """The long-sequence shape (128 heads in one B/C group) through the backward, with the
    forward's kept chunk states: the gradient kernel covers the group in head subsets whose
    dB/dC shares are summed afterwards."""
    from helpers import to_dev
    from state_space_model_scan_gb300.api import ssd_forward
    w = I.Workload("long_bwd", 1, 1024, 128, 64, 1, 128, 128, "bf16", has_z=False, has_init=True)
    inp = I.make_inputs(w, with_grad_inputs=True, with_dfinal=True)
    d = to_dev(inp)
    _, _, cs = ssd_forward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], D=d["D"], dt_bias=d["dt_bias"],
                           initial_states=d["initial_states"], chunk_size=128, keep_chunk_states=True)
    g = gpu_backward(w, inp, chunk_states=cs)
    o = oracle_backward(w, inp)
    T = w.seqlen
    errs = dict(dx=rel_l2(flat(g["dx"], T), o["dx"]), ddt=rel_l2(flat(g["ddt"], T), o["ddt_raw"]),
                dB=rel_l2(flat(g["dB"], T), o["dB"]), dC=rel_l2(flat(g["dC"], T), o["dC"]),
                dA=rel_l2(g["dA"].double().cpu().numpy(), o["dA"]), dD=rel_l2(g["dD"].double().cpu().numpy(), o["dD"]),
                dinit=rel_l2(g["dinitial_states"].double().cpu().numpy(), o["dinit"]))
    bad = {k: v for k, v in errs.items() if not v <= TOL["bf16"]}
    assert not bad, errs
