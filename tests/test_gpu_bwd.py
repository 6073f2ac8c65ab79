"""Backward parity of the CUDA path against the oracle's adjoint (GPU).

The oracle's gradients are pinned on CPU by central differences and by torch
autograd of the quadratic form (tests/test_oracle_grad.py).
"""
import numpy as np
import pytest
import torch

from state_space_model_scan_gb300 import inputs as I
from helpers import TOL, rel_l2, gpu_backward, oracle_backward, flat

pytestmark = pytest.mark.gpu

NAMES = [("dx", "dx"), ("ddt", "ddt_raw"), ("dA", "dA"), ("dB", "dB"), ("dC", "dC"), ("dD", "dD"), ("dz", "dz"),
         ("ddt_bias", "ddt_bias"), ("dinitial_states", "dinit")]


def W(name="t", B=1, L=256, H=4, P=16, G=1, N=16, Q=None, dtype="f32", **kw):
    """A workload; the chunk length defaults to the one its path computes (128 for the
    tensor-core tile set, 64 for SIMT)."""
    if Q is None:
        Q = 128 if (dtype == "bf16" and P == 64 and N == 128) else 64
    return I.Workload(name, B, L, H, P, G, N, Q, dtype, **kw)


def for_algo(case, algo):
    """The SIMT path computes 64-token chunks: a staged run of a tensor-core case uses 64."""
    case = dict(case)
    if algo == "staged":
        case["Q"] = 64
    return case


def check_bwd(w, algo="auto", with_dfinal=True, tol=None):
    inp = I.make_inputs(w, with_grad_inputs=True, with_dfinal=with_dfinal)
    g = gpu_backward(w, inp, algo=algo)
    o = oracle_backward(w, inp)
    T = w.batch * w.seqlen
    tol = tol or TOL[w.dtype]
    errs = {}
    for gn, on in NAMES:
        if gn not in g:
            assert on not in o
            continue
        t = g[gn]
        a = flat(t, T) if t.dim() >= 3 and t.shape[0] == w.batch and gn not in ("dinitial_states",) else \
            t.detach().double().cpu().numpy()
        b = o[on]
        a = a.reshape(b.shape)
        assert np.isfinite(a).all(), gn
        errs[gn] = rel_l2(a, b)
    bad = {k: v for k, v in errs.items() if v > tol}
    assert not bad, (w, errs)
    return errs


@pytest.mark.parametrize("case", [
    dict(),
    dict(L=1), dict(L=70), dict(L=129, H=6, G=2, has_z=True, has_init=True),
    dict(B=2, L=100, H=6, G=3, P=32, N=32, has_z=True, has_init=True),
    dict(P=128, N=128, L=90, H=2, has_z=True),
    dict(has_D=False, has_dt_bias=False, L=77),
])
def test_bwd_fp32(case):
    check_bwd(W(**case))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", [
    dict(L=200, H=4, P=16, G=2, N=16, has_z=True, has_init=True),
    dict(B=2, L=45, H=3, P=32, G=3, N=64, has_z=True),
    dict(L=150, H=2, P=128, N=128, has_init=True),
])
def test_bwd_chunk32(case, dtype):
    """The SIMT backward at 32-token chunks (eight threads per chunk row)."""
    check_bwd(W(Q=32, dtype=dtype, **case), algo="staged")


def test_bwd_long_simt_chunks_refused():
    """The SIMT backward computes 32- and 64-token chunks only: 128 (fp32) and 256 are refused."""
    import pytest as _pt
    from state_space_model_scan_gb300 import _lib
    for Q in (128, 256):
        w = W(L=300, Q=Q)
        inp = I.make_inputs(w, with_grad_inputs=True)
        with _pt.raises(_lib.SSDError) as e:
            gpu_backward(w, inp, algo="staged")
        assert e.value.code == 2


@pytest.mark.parametrize("algo", ["staged", "fused"])
@pytest.mark.parametrize("case", [
    dict(L=600, H=8, P=64, G=2, N=128, Q=128, has_z=True, has_init=True),
    dict(L=1, H=2, P=64, G=1, N=128, Q=128, has_init=True),
    dict(L=127, H=6, P=64, G=2, N=128, Q=128, has_z=True),
    dict(B=2, L=300, H=3, P=64, G=3, N=128, Q=128, has_D=False, has_dt_bias=False),
    dict(L=1000, H=4, P=64, G=1, N=128, Q=128, has_z=True, has_init=True),
])
def test_bwd_bf16(case, algo):
    check_bwd(W(dtype="bf16", **for_algo(case, algo)), algo=algo)


@pytest.mark.parametrize("seg", [1, 3])
def test_bwd_fused_multi_unit(seg):
    w = W(B=2, L=1300, H=4, P=64, G=2, N=128, Q=128, dtype="bf16", has_z=True, has_init=True)
    inp = I.make_inputs(w, with_grad_inputs=True, with_dfinal=True)
    from helpers import gpu_backward as gb
    g = gb(w, inp, algo="fused", seg_chunks=seg)
    o = oracle_backward(w, inp)
    T = w.batch * w.seqlen
    for gn, on in NAMES:
        t = g[gn]
        a = flat(t, T) if t.dim() >= 3 and gn != "dinitial_states" else t.detach().double().cpu().numpy()
        assert rel_l2(a.reshape(o[on].shape), o[on]) <= TOL["bf16"], gn


@pytest.mark.parametrize("Q", [32, 64])
def test_bwd_varlen(Q):
    w = I.Workload("v", 1, 241, 4, 16, 2, 16, Q, "f32", has_z=True, has_init=True, seqlens=[40, 0, 130, 1, 70])
    check_bwd(w)


def test_bwd_varlen_fused():
    lens = [40, 0, 130, 1, 270, 128]
    w = I.Workload("v", 1, sum(lens), 4, 64, 2, 128, 128, "bf16", has_z=True, has_init=True, seqlens=lens)
    check_bwd(w, algo="fused")


@pytest.mark.parametrize("P,N", [(32, 32), (64, 128)])
def test_bwd_deterministic(P, N):
    w = W(L=700, H=4, P=P, G=2, N=N, dtype="bf16", has_z=True, has_init=True)
    inp = I.make_inputs(w, with_grad_inputs=True, with_dfinal=True)
    g1 = gpu_backward(w, inp)
    g2 = gpu_backward(w, inp)
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k


@pytest.mark.parametrize("H,G", [(24, 2), (16, 1)])
def test_bwd_heads_per_cta(H, G):
    """The gradient kernel's heads-per-CTA choice (whole group in one CTA, or subsets
    of it summed afterwards) changes only the summation order of dB and dC."""
    w = W(L=300, H=H, P=64, G=G, N=128, Q=128, dtype="bf16", has_z=True, has_init=True)
    inp = I.make_inputs(w, with_grad_inputs=True, with_dfinal=True)
    o = oracle_backward(w, inp)
    T = w.batch * w.seqlen
    hpg = H // G
    choices = [0] + [d for d in range(1, 33) if hpg % d == 0]
    ref = None
    for hs in choices:
        g = gpu_backward(w, inp, algo="fused", bwd_heads=hs)
        for gn, on in NAMES:
            t = g[gn]
            a = flat(t, T) if t.dim() >= 3 and gn != "dinitial_states" else t.detach().double().cpu().numpy()
            assert rel_l2(a.reshape(o[on].shape), o[on]) <= TOL["bf16"], (hs, gn)
        if ref is None:
            ref = g
        else:
            for k in g:
                if k not in ("dB", "dC"):
                    assert torch.equal(g[k], ref[k]), (hs, k)


def test_bwd_heads_invalid():
    from state_space_model_scan_gb300._lib import SSDError
    w = W(L=200, H=12, P=64, G=1, N=128, Q=128, dtype="bf16")
    inp = I.make_inputs(w, with_grad_inputs=True)
    for hs in (5, 33, -1):
        with pytest.raises(SSDError):
            gpu_backward(w, inp, algo="fused", bwd_heads=hs)


def test_bwd_rejects_five_chunk_units():
    """The backward's state recompute keeps each chunk of a unit in its own TMEM slice, four at
    most: five-chunk units are refused (the forward accepts them)."""
    from state_space_model_scan_gb300._lib import SSDError
    w = W(L=700, H=4, P=64, G=2, N=128, Q=128, dtype="bf16")
    inp = I.make_inputs(w, with_grad_inputs=True)
    with pytest.raises(SSDError):
        gpu_backward(w, inp, algo="fused", seg_chunks=5)


@pytest.mark.parametrize("lens", [None, [1000, 3000, 1120]])
def test_bwd_tail_split(lens):
    """More (chunk, group) pairs than SMs: the gradient kernel's last partial wave is split into
    items of half a group whose dB/dC shares are summed afterwards; packed sequences also leave
    work items past the real chunk count, which are skipped."""
    if lens is None:
        w = W(L=128 * 40, H=32, P=64, G=4, N=128, Q=128, dtype="bf16", has_z=True, has_init=True)
    else:
        w = I.Workload("v", 1, sum(lens), 32, 64, 4, 128, 128, "bf16", has_z=True, has_init=True, seqlens=lens)
    check_bwd(w, algo="fused")


def test_bwd_row_store_alignment_paths_agree():
    """dx / dz rows go out as 256-bit stores when base and strides are 32-byte aligned, as
    128-bit stores otherwise (16-byte aligned views): both give the same bits."""
    from state_space_model_scan_gb300 import _lib
    from helpers import to_dev
    w = W(L=700, H=8, P=64, G=2, N=128, Q=128, dtype="bf16", has_z=True, has_init=True)
    inp = I.make_inputs(w, with_grad_inputs=True, with_dfinal=True)
    d = to_dev(inp)
    H = w.nheads

    def run(offset):
        n = d["x"].numel()
        bx = torch.zeros(n + 16, dtype=torch.bfloat16, device="cuda")
        bz = torch.zeros(n + 16, dtype=torch.bfloat16, device="cuda")
        dx = bx[offset:offset + n].view(d["x"].shape)
        dz = bz[offset:offset + n].view(d["x"].shape)
        g = dict(ddt=torch.empty_like(d["dt_raw"]), dA=torch.empty(H, device="cuda"), dB=torch.empty_like(d["B"]),
                 dC=torch.empty_like(d["C"]), dD=torch.empty(H, device="cuda"), ddt_bias=torch.empty(H, device="cuda"),
                 dinit=torch.empty_like(d["initial_states"]))
        prob = _lib.problem(w.batch, w.seqlen, H, 64, w.ngroups, 128, 128)
        fa = _lib.fwd_args(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], None, D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                           initial_states=d["initial_states"])
        ba = _lib.bwd_args(fa, d["dy"], dx, g["ddt"], g["dA"], g["dB"], g["dC"], dD=g["dD"], dz=dz,
                           ddt_bias=g["ddt_bias"], dinitial_states=g["dinit"], dfinal_states=d["dfinal_states"])
        ws = torch.empty(_lib.bwd_workspace_size(prob, ba), dtype=torch.uint8, device="cuda")
        _lib.check(_lib.ssd_bwd(prob, ba, ws), "ssd_bwd")
        torch.cuda.synchronize()
        return dx.clone(), dz.clone(), g

    dx0, dz0, g0 = run(0)      # 32-byte aligned base
    dx1, dz1, g1 = run(8)      # 16 bytes off
    assert dx0.data_ptr() % 32 == 0
    assert torch.equal(dx0, dx1) and torch.equal(dz0, dz1)
    for k in g0:
        assert torch.equal(g0[k], g1[k]), k
