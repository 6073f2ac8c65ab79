"""Causal depthwise conv1d (+ SiLU) over the packed xBC channels on the GPU, forward and
backward, against the float64 oracle: dtypes, kernel widths, tile edges, packed sequences
shorter than the kernel, strided inputs, the full Nemotron-Nano xBC size, and conv -> split
(views) -> scan as in a Mamba-2 block."""
import numpy as np
import pytest
import torch

from oracle import conv1d as oc
from state_space_model_scan_gb300 import inputs as I
from state_space_model_scan_gb300.api import conv1d_forward, conv1d_backward, split_xbc, ssd_forward
from helpers import TOL, rel_l2, oracle_forward

pytestmark = pytest.mark.gpu


def make(B, L, Cn, K, dtype, bias=True, seed=0):
    g = torch.Generator().manual_seed(seed)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    u = torch.randn(B, L, Cn, generator=g, dtype=torch.float64).to(td)
    w = (0.5 * torch.randn(Cn, K, generator=g, dtype=torch.float64)).to(torch.float32)
    b = (0.1 * torch.randn(Cn, generator=g, dtype=torch.float64)).to(torch.float32) if bias else None
    dout = torch.randn(B, L, Cn, generator=g, dtype=torch.float64).to(td)
    return u, w, b, dout


def h(t):
    return None if t is None else t.double().cpu().numpy()


def check(u, w, b, dout, dtype, silu=True, cu=None):
    ud, wd, dd = u.cuda(), w.cuda(), dout.cuda()
    bd = b.cuda() if b is not None else None
    cud = torch.tensor(cu, dtype=torch.int32, device="cuda") if cu is not None else None
    out = conv1d_forward(ud, wd, bd, cu_seqlens=cud, silu=silu)
    du, dw, db = conv1d_backward(ud, wd, dd, bd, cu_seqlens=cud, silu=silu)
    torch.cuda.synchronize()
    tol = TOL[dtype]
    dw_ref = np.zeros(w.shape)
    db_ref = np.zeros(w.shape[0])
    for bb in range(u.shape[0]):
        oo, _ = oc.forward(h(u[bb]), h(w), h(b), cu=cu, silu=silu)
        odu, odw, odb = oc.backward(h(u[bb]), h(w), h(dout[bb]), h(b), cu=cu, silu=silu)
        assert rel_l2(h(out[bb]), oo) <= tol
        assert rel_l2(h(du[bb]), odu) <= tol
        dw_ref += odw
        db_ref += odb
    assert rel_l2(h(dw), dw_ref) <= tol
    if b is not None:
        assert rel_l2(h(db), db_ref) <= tol
    return out, du, dw, db


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("K", [1, 2, 4, 8])
@pytest.mark.parametrize("B,L,Cn", [(1, 1, 8), (2, 63, 64), (1, 65, 2048 + 8), (3, 200, 24)])
def test_conv_matches_oracle(dtype, K, B, L, Cn):
    check(*make(B, L, Cn, K, dtype), dtype)


@pytest.mark.parametrize("silu,bias", [(False, True), (True, False)])
def test_conv_activation_and_bias_options(silu, bias):
    check(*make(2, 130, 32, 4, "f32", bias=bias), "f32", silu=silu)


@pytest.mark.parametrize("lens", [[3, 0, 1, 2, 200, 5, 64, 63, 1], [64, 64, 128], [1] * 20])
def test_conv_packed_sequences_never_mix(lens):
    """Sequences shorter than the kernel, empty ones, boundaries on and off the 64-token tiles."""
    cu = [0] + list(np.cumsum(lens))
    u, w, b, dout = make(1, cu[-1], 48, 4, "f32")
    check(u, w, b, dout, "f32", cu=cu)


def test_conv_strided_token_rows():
    """The packed xBC as a view into a wider buffer (token stride > channels)."""
    g = torch.Generator().manual_seed(3)
    wide = torch.randn(2, 90, 96, generator=g).to(torch.bfloat16).cuda()
    u = wide[..., 8:72]
    assert u.stride(1) == 96
    w = (0.5 * torch.randn(64, 4, generator=g)).cuda()
    out = conv1d_forward(u, w)
    torch.cuda.synchronize()
    for bb in range(2):
        oo, _ = oc.forward(h(u[bb]), h(w))
        assert rel_l2(h(out[bb]), oo) <= TOL["bf16"]


def test_conv_full_nemotron_xbc():
    """8192 tokens x (64 x 64 + 2 x 8 x 128) channels, kernel 4, bf16, forward and backward."""
    u, w, b, dout = make(1, 8192, 6144, 4, "bf16", seed=7)
    check(u, w, b, dout, "bf16")


def test_conv_split_scan_as_in_a_mamba2_block():
    """conv1d + SiLU over the packed xBC, x/B/C as views of its output, then the scan; against
    the same composition of the float64 oracles."""
    H, P, G, N, L = 8, 64, 2, 128, 400
    Cn = H * P + 2 * G * N
    u, w, b, _ = make(1, L, Cn, 4, "bf16", seed=11)
    wl = I.Workload("blk", 1, L, H, P, G, N, 128, "bf16", has_z=True, has_init=False)
    inp = I.make_inputs(wl)
    xbc = conv1d_forward(u.cuda(), w.cuda(), b.cuda())
    x, Bm, Cm = split_xbc(xbc, H, P, G, N)
    assert not x.is_contiguous()
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y, fin = ssd_forward(x, d["dt_raw"], d["A"], Bm, Cm, D=d["D"], z=d["z"], dt_bias=d["dt_bias"], chunk_size=128)
    torch.cuda.synchronize()
    # the oracle's composition, from the same rounded conv output the scan consumed
    oo, _ = oc.forward(h(u[0]), h(w), h(b))
    assert rel_l2(h(xbc[0]), oo) <= TOL["bf16"]
    ref = dict(inp)
    ref["x"], ref["B"], ref["C"] = (t.cpu() for t in split_xbc(xbc, H, P, G, N))
    yo, fo = oracle_forward(wl, ref)
    assert rel_l2(y.double().cpu().numpy().reshape(L, H, P), yo) <= TOL["bf16"]
