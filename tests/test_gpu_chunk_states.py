"""Carried chunk states kept by the forward for the backward (tensor-core path, GPU).

The forward writes, per (chunk, head), the state entering the chunk; by the
recurrence that is the final state of the sequence's prefix that ends at the
chunk's first token, which the float64 sequential oracle gives directly.  The
backward that reads them must match the oracle's adjoint like the one that
recomputes them.
"""
import numpy as np
import pytest
import torch

from state_space_model_scan_gb300 import inputs as I
from state_space_model_scan_gb300 import _lib
from state_space_model_scan_gb300.api import ssd_forward, ssd_backward
from helpers import TOL, rel_l2, to_dev, oracle_backward, flat

pytestmark = pytest.mark.gpu

Q = 128   # chunk length of the tensor-core path
NAMES = [("dx", "dx"), ("ddt", "ddt_raw"), ("dA", "dA"), ("dB", "dB"), ("dC", "dC"), ("dD", "dD"), ("dz", "dz"),
         ("ddt_bias", "ddt_bias"), ("dinitial_states", "dinit")]


def decode_tiles(buf, n_tiles):
    """[tiles, P=64, N=128] float64 from the library's tiles: bf16 row n holds S[:, n]; its
    16-byte piece q (p = 8q .. 8q+7) sits at position q ^ (n % 8)."""
    t = buf[: n_tiles * 16384].view(torch.bfloat16).float().cpu().numpy().reshape(n_tiles, 128, 8, 8)
    n = np.arange(128)[:, None]
    q = np.arange(8)[None, :]
    g = t[:, n, q ^ (n & 7), :]   # [tiles, n, q, e]
    return g.reshape(n_tiles, 128, 64).transpose(0, 2, 1).astype(np.float64)


def oracle_chunk_states(w, inp):
    """{(tile index, head): state entering the tile}, from prefix runs of the oracle.  The tiles
    are the segments of the chunk grid (oracle.varlen_meta), listed sequence by sequence; the
    state entering a tile is the final state of its sequence's prefix that ends where the tile's
    rows of that sequence begin."""
    from oracle import sequential, varlen_meta
    o = I.to_oracle(inp, w)
    cu = [int(c) for c in o["cu"]]
    H, P, N = w.nheads, w.headdim, w.dstate
    if inp["cu_seqlens"] is not None:
        tiles = [(s, a) for (s, a, _) in varlen_meta.segments(cu, Q)[0]]
    else:
        tiles = [(b, cu[b] + c * Q) for b in range(w.batch) for c in range(-(-w.seqlen // Q))]
    out = {}
    for k, (s, a) in enumerate(tiles):
        t0 = cu[s]
        init = o["init"][s] if o["init"] is not None else np.zeros((H, P, N))
        if a == t0:
            st = init
        else:
            sl = slice(t0, a)
            _, fin = sequential.forward(o["x"][sl], o["dt_raw"][sl], o["A"], o["B"][sl], o["C"][sl], D=o["D"],
                                        z=None if o["z"] is None else o["z"][sl], dt_bias=o["dt_bias"],
                                        init=init[None], cu=np.array([0, a - t0]))
            st = fin[0]
        for h in range(H):
            out[(k, h)] = st[h]
    return out


def forward_keep(w, inp):
    d = to_dev(inp)
    y, fin, cs = ssd_forward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                             initial_states=d["initial_states"], cu_seqlens=d["cu_seqlens"], chunk_size=Q,
                             keep_chunk_states=True)
    torch.cuda.synchronize()
    return y, fin, cs


@pytest.mark.parametrize("case", [
    dict(B=2, L=384, lens=None),
    dict(B=1, L=0, lens=[200, 0, 300, 1, 129]),
])
def test_kept_chunk_states_are_the_carried_states(case):
    lens = case["lens"]
    L = sum(lens) if lens else case["L"]
    w = I.Workload("cs", case["B"], L, 4, 64, 2, 128, Q, "bf16", has_z=True, has_init=True, seqlens=lens)
    inp = I.make_inputs(w)
    _, _, cs = forward_keep(w, inp)
    ref = oracle_chunk_states(w, inp)
    nk = max(k for k, _ in ref) + 1
    got = decode_tiles(cs, nk * w.nheads).reshape(nk, w.nheads, 64, 128)
    a = np.stack([got[k, h] for (k, h) in ref])
    b = np.stack([ref[key] for key in ref])
    assert rel_l2(a, b) <= TOL["bf16"]
    # per tile too: no tile may be a stale or misplaced one
    for i, key in enumerate(ref):
        assert rel_l2(a[i], b[i]) <= 2e-2, key


@pytest.mark.parametrize("case", [
    dict(B=2, L=700, H=8, G=2, lens=None),
    dict(B=1, L=0, H=4, G=1, lens=[300, 0, 129, 1, 450]),
])
def test_backward_with_kept_states_matches_oracle(case):
    lens = case["lens"]
    L = sum(lens) if lens else case["L"]
    w = I.Workload("bk", case["B"], L, case["H"], 64, case["G"], 128, Q, "bf16", has_z=True, has_init=True,
                   seqlens=lens)
    inp = I.make_inputs(w, with_grad_inputs=True, with_dfinal=True)
    _, _, cs = forward_keep(w, inp)
    d = to_dev(inp)
    kw = dict(D=d["D"], z=d["z"], dt_bias=d["dt_bias"], initial_states=d["initial_states"],
              dfinal_states=d["dfinal_states"], cu_seqlens=d["cu_seqlens"], chunk_size=Q)
    g_kept = ssd_backward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], d["dy"], chunk_states=cs, **kw)
    g_rec = ssd_backward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], d["dy"], **kw)
    torch.cuda.synchronize()
    o = oracle_backward(w, inp)
    T = w.batch * w.seqlen
    for gn, on in NAMES:
        def host(t):
            a = flat(t, T) if t.dim() >= 3 and gn != "dinitial_states" else t.detach().double().cpu().numpy()
            return a.reshape(o[on].shape)
        a, r = host(g_kept[gn]), host(g_rec[gn])
        assert rel_l2(a, o[on]) <= TOL["bf16"], gn
        # the two paths differ only where a state rounds differently to bf16
        assert rel_l2(a, r) <= 5e-3, gn


def test_autograd_function_keeps_states():
    """SSDFunction keeps the states on the tensor-core path: same gradients as the explicit calls."""
    from state_space_model_scan_gb300.api import SSDFunction
    w = I.Workload("ag", 1, 500, 4, 64, 2, 128, Q, "bf16", has_z=True, has_init=True)
    inp = I.make_inputs(w, with_grad_inputs=True)
    d = to_dev(inp)
    x = d["x"].clone().requires_grad_(True)
    y, fin = SSDFunction.apply(x, d["dt_raw"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                               d["initial_states"], None, Q)
    y.backward(d["dy"])
    _, _, cs = forward_keep(w, inp)
    g = ssd_backward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], d["dy"], D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                     initial_states=d["initial_states"], chunk_size=Q, chunk_states=cs)
    torch.cuda.synchronize()
    assert torch.equal(x.grad, g["dx"])


def test_kept_states_rejected_off_the_tensor_core_path():
    w = I.Workload("f32", 1, 100, 2, 16, 1, 16, 64, "f32")
    d = to_dev(I.make_inputs(w))
    with pytest.raises(_lib.SSDError) as e:
        ssd_forward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], keep_chunk_states=True)
    assert e.value.code == 2
