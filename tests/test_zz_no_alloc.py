"""ssd_fwd_noalloc: the forward for callers that cannot allocate device memory.

Runs through the C ABI and must give the same bits as ssd_fwd with a
caller-supplied workspace, on two calls in a row (the shared static scratch keeps
the previous call's contents; each call must re-initialise what it needs), and
report device-side errors through ssd_noalloc_query_status.  This file is
collected last on purpose.
"""
import numpy as np
import pytest
import torch

from state_space_model_scan_gb300 import inputs as I
from state_space_model_scan_gb300 import _lib
from helpers import to_dev

pytestmark = pytest.mark.gpu


def _args(w, inp):
    d = to_dev(inp)
    y = torch.full_like(d["x"], float("nan"))
    fin = torch.full((w.nseqs, w.nheads, w.headdim, w.dstate), float("nan"), device="cuda")
    prob = _lib.problem(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.chunk_size,
                        w.nseqs if inp["cu_seqlens"] is not None else 0)
    args = _lib.fwd_args(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], y, D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                         initial_states=d["initial_states"], final_states=fin, cu_seqlens=d["cu_seqlens"])
    return prob, args, y, fin, d


@pytest.mark.parametrize("w", [
    I.Workload("fused", 2, 1500, 8, 64, 2, 128, 128, "bf16", has_z=True, has_init=True),
    I.Workload("staged", 1, 300, 4, 32, 2, 64, 64, "f32", has_z=True, has_init=True),
    I.Workload("packed", 1, 600, 8, 64, 1, 128, 128, "bf16", has_init=True, seqlens=[100, 0, 373, 127]),
], ids=lambda w: w.name)
def test_noalloc_matches_workspace_forward_twice(w):
    inp = I.make_inputs(w)
    prob, args, y_ref, fin_ref, d_ref = _args(w, inp)   # d_ref: the device inputs stay alive
    ws = torch.empty(_lib.fwd_workspace_size(prob, args), dtype=torch.uint8, device="cuda")
    assert ws.numel() <= _lib.NOALLOC_SCRATCH_BYTES
    _lib.check(_lib.ssd_fwd(prob, args, ws), "ssd_fwd")
    torch.cuda.synchronize()
    for _ in range(2):
        prob2, args2, y, fin, d2 = _args(w, inp)
        _lib.check(_lib.ssd_fwd_noalloc(prob2, args2), "ssd_fwd_noalloc")
        torch.cuda.synchronize()
        assert _lib.noalloc_query_status() == 0
        # the same deterministic kernels on the same inputs: the same bits (a stale value
        # left in the shared scratch by the previous call would show here)
        assert torch.equal(y, y_ref)
        assert torch.equal(fin, fin_ref)


def test_noalloc_reports_device_errors_through_its_status_reader():
    """Bad cu_seqlens contents are found on the device; the noalloc caller has no
    workspace, so it reads them with ssd_noalloc_query_status; a good call after it
    clears the word again."""
    w = I.Workload("packed", 1, 600, 8, 64, 1, 128, 128, "bf16", has_init=True, seqlens=[100, 0, 373, 127])
    inp = I.make_inputs(w)
    bad = dict(inp)
    bad["cu_seqlens"] = torch.tensor([0, 100, 50, 473, 600], dtype=torch.int32)   # not non-decreasing
    prob, args, y, fin, d = _args(w, bad)
    assert _lib.ssd_fwd_noalloc(prob, args) == 0
    assert _lib.noalloc_query_status() == 1
    assert torch.isnan(y.float()).all() and torch.isnan(fin).all()   # no kernel wrote the outputs
    prob2, args2, y2, fin2, d2 = _args(w, inp)
    _lib.check(_lib.ssd_fwd_noalloc(prob2, args2), "ssd_fwd_noalloc")
    assert _lib.noalloc_query_status() == 0
    assert torch.isfinite(y2.float()).all()


def test_noalloc_rejects_problems_beyond_its_scratch():
    w = I.Workload("big", 4, 8192, 64, 64, 8, 128, 128, "bf16", has_z=False)
    # metadata only: the pointers are never dereferenced because the call is rejected first
    prob = _lib.problem(w.batch, w.seqlen, w.nheads, 64, 8, 128, 64, 0, "staged")
    x = torch.empty(1, dtype=torch.bfloat16, device="cuda")
    f = torch.empty(1, device="cuda")
    args = _lib.FwdArgs()
    for name, t, strides in (("x", x, [8192 * 64 * 64, 64 * 64, 64, 1]), ("y", x, [8192 * 64 * 64, 64 * 64, 64, 1]),
                             ("B", x, [8192 * 8 * 128, 8 * 128, 128, 1]), ("C", x, [8192 * 8 * 128, 8 * 128, 128, 1]),
                             ("dt", f, [8192 * 64, 64, 1]), ("A", f, [1])):
        tt = _lib.tensor(t)
        for i, s in enumerate(strides):
            tt.stride[i] = s
        setattr(args, name, tt)
    need = _lib.fwd_workspace_size(prob, args)
    assert need > _lib.NOALLOC_SCRATCH_BYTES
    assert _lib.ssd_fwd_noalloc(prob, args) == 4


def test_noalloc_forward_keeps_the_same_chunk_states():
    """The allocation-free forward writes the caller's chunk-state buffer like ssd_fwd does."""
    w = I.Workload("keep", 2, 900, 8, 64, 2, 128, 128, "bf16", has_z=True, has_init=True)
    inp = I.make_inputs(w)
    prob, args, y1, fin1, d1 = _args(w, inp)   # every tensor stays alive: args holds raw pointers
    n = _lib.chunk_states_size(prob, args)
    cs_ref = torch.zeros(n, dtype=torch.uint8, device="cuda")
    cs = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
    args.chunk_states = cs_ref.data_ptr()
    ws = torch.empty(_lib.fwd_workspace_size(prob, args), dtype=torch.uint8, device="cuda")
    _lib.check(_lib.ssd_fwd(prob, args, ws), "ssd_fwd")
    prob2, args2, y2, fin2, d2 = _args(w, inp)
    args2.chunk_states = cs.data_ptr()
    _lib.check(_lib.ssd_fwd_noalloc(prob2, args2), "ssd_fwd_noalloc")
    torch.cuda.synchronize()
    used = 2 * 8 * 8 * 16384   # batch rows x chunks per row x heads x tile bytes
    assert torch.equal(cs[:used], cs_ref[:used])
