"""Gated normalisation over feature groups on the GPU (forward and backward) against the
float64 oracle: RMS and LayerNorm, the gate before or after the norm, dtypes, with and
without the gate, group sizes (register, staged and two-pass kernels), strided rows, the
full Nemotron-Nano width, determinism, and the composition scan -> gated norm of a Mamba-2
block."""
import numpy as np
import pytest
import torch

from oracle import gated_norm as gn
from state_space_model_scan_gb300 import inputs as I
from state_space_model_scan_gb300.api import gated_norm_forward, gated_norm_backward, ssd_forward
from helpers import TOL, rel_l2, to_dev, oracle_forward, flat

pytestmark = pytest.mark.gpu


def tensors(rows, width, dtype, gate, seed=0, row_pad=0):
    g = torch.Generator().manual_seed(seed)
    base = torch.randn(rows, width + row_pad, generator=g, dtype=torch.float64)
    y = base[:, :width]
    z = torch.randn(rows, width, generator=g, dtype=torch.float64) if gate else None
    w = (1.0 + 0.3 * torch.randn(width, generator=g, dtype=torch.float64)).to(torch.float32)
    dout = torch.randn(rows, width, generator=g, dtype=torch.float64)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    cast = lambda t: None if t is None else t.to(td)
    return cast(base)[:, :width] if row_pad else cast(y), cast(z), w, cast(dout)


def host(t):
    return None if t is None else t.double().cpu().numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("gate", [True, False])
@pytest.mark.parametrize("rows,width,group", [(1, 64, 64), (37, 256, 64), (100, 512, 8), (64, 1536, 512),
                                              (33, 6144, 6144)])
def test_gated_norm_matches_oracle(dtype, gate, rows, width, group):
    y, z, w, dout = tensors(rows, width, dtype, gate)
    yd, zd, wd, dd = (None if t is None else t.cuda() for t in (y, z, w, dout))
    out, rstd = gated_norm_forward(yd, wd, group, z=zd)
    dy, dz, dw = gated_norm_backward(yd, wd, rstd, dd, group, z=zd)
    torch.cuda.synchronize()
    oo, orstd = gn.forward(host(y), host(w), group, z=host(z))
    ody, odz, odw = gn.backward(host(y), host(w), host(dout), group, z=host(z))
    tol = TOL[dtype]
    assert rel_l2(host(out), oo) <= tol
    assert rel_l2(host(rstd), orstd) <= tol
    assert rel_l2(host(dy), ody) <= tol
    assert rel_l2(host(dw), odw) <= tol
    if gate:
        assert rel_l2(host(dz), odz) <= tol


@pytest.mark.parametrize("mode", [dict(layer_norm=True), dict(gate_after=True),
                                  dict(layer_norm=True, gate_after=True)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("gate", [True, False])
@pytest.mark.parametrize("rows,width,group", [(37, 256, 64), (64, 1536, 512), (33, 6144, 6144)])
def test_gated_norm_modes_match_oracle(mode, dtype, gate, rows, width, group):
    """LayerNorm and/or the gate after the norm, through every kernel size class; the inputs
    carry a per-row offset so the LayerNorm mean matters."""
    y, z, w, dout = tensors(rows, width, dtype, gate, seed=9)
    y = (y.double() + torch.linspace(-2.0, 3.0, rows, dtype=torch.float64)[:, None]).to(y.dtype)
    yd, zd, wd, dd = (None if t is None else t.cuda() for t in (y, z, w, dout))
    out, rstd = gated_norm_forward(yd, wd, group, z=zd, **mode)
    dy, dz, dw = gated_norm_backward(yd, wd, rstd, dd, group, z=zd, **mode)
    torch.cuda.synchronize()
    oo, orstd = gn.forward(host(y), host(w), group, z=host(z), **mode)
    ody, odz, odw = gn.backward(host(y), host(w), host(dout), group, z=host(z), **mode)
    tol = TOL[dtype]
    assert rel_l2(host(out), oo) <= tol
    assert rel_l2(host(rstd), orstd) <= tol
    assert rel_l2(host(dy), ody) <= tol
    assert rel_l2(host(dw), odw) <= tol
    if gate:
        assert rel_l2(host(dz), odz) <= tol


def test_gated_norm_strided_rows_and_determinism():
    """Rows at a padded stride (a view into a wider buffer); two runs give the same bits."""
    y, z, w, dout = tensors(300, 512, "bf16", True, row_pad=64)
    yd = y.cuda() if y.is_contiguous() else torch.empty_strided(y.shape, (576, 1), dtype=y.dtype, device="cuda")
    yd.copy_(y)
    assert yd.stride(0) == 576
    zd, wd, dd = z.cuda(), w.cuda(), dout.cuda()
    r1 = gated_norm_forward(yd, wd, 128, z=zd)
    r2 = gated_norm_forward(yd, wd, 128, z=zd)
    b1 = gated_norm_backward(yd, wd, r1[1], dd, 128, z=zd)
    b2 = gated_norm_backward(yd, wd, r1[1], dd, 128, z=zd)
    torch.cuda.synchronize()
    assert torch.equal(r1[0], r2[0]) and torch.equal(r1[1], r2[1])
    for a, b in zip(b1, b2):
        assert torch.equal(a, b)
    oo, _ = gn.forward(host(y), host(w), 128, z=host(z))
    assert rel_l2(host(r1[0]), oo) <= TOL["bf16"]


def test_gated_norm_full_nemotron_width():
    """8192 tokens x (64 heads x 64), groups of 512 (the heads of one B/C group), bf16."""
    y, z, w, dout = tensors(8192, 4096, "bf16", True, seed=5)
    yd, zd, wd, dd = y.cuda(), z.cuda(), w.cuda(), dout.cuda()
    out, rstd = gated_norm_forward(yd, wd, 512, z=zd)
    dy, dz, dw = gated_norm_backward(yd, wd, rstd, dd, 512, z=zd)
    torch.cuda.synchronize()
    rows = np.arange(0, 8192, 61)
    oo, _ = gn.forward(host(y)[rows], host(w), 512, z=host(z)[rows])
    ody, odz, _ = gn.backward(host(y)[rows], host(w), host(dout)[rows], 512, z=host(z)[rows])
    assert rel_l2(host(out)[rows], oo) <= TOL["bf16"]
    assert rel_l2(host(dy)[rows], ody) <= TOL["bf16"]
    assert rel_l2(host(dz)[rows], odz) <= TOL["bf16"]
    # dw sums every row: check it against the oracle over all rows
    _, _, odw = gn.backward(host(y), host(w), host(dout), 512, z=host(z))
    assert rel_l2(host(dw), odw) <= TOL["bf16"]


def test_scan_then_gated_norm_as_in_a_mamba2_block():
    """ssd_fwd without the gate, then the gated normalisation over each B/C group's heads,
    against the same composition of the float64 oracles."""
    w_ = I.Workload("blk", 1, 700, 8, 64, 2, 128, 128, "bf16", has_z=True, has_init=True)
    inp = I.make_inputs(w_)
    d = to_dev(inp)
    y, _ = ssd_forward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], D=d["D"], dt_bias=d["dt_bias"],
                       initial_states=d["initial_states"], chunk_size=128)
    weight = torch.linspace(0.5, 1.5, 8 * 64, device="cuda")
    out, _ = gated_norm_forward(y.reshape(1, 700, 512), weight, 4 * 64, z=d["z"].reshape(1, 700, 512))
    torch.cuda.synchronize()
    nz = dict(inp)
    nz["z"] = None
    yo, _ = oracle_forward(w_, nz)
    oo, _ = gn.forward(yo.reshape(700, 512), weight.double().cpu().numpy(), 256,
                       z=inp["z"].double().numpy().reshape(700, 512))
    assert rel_l2(out.double().cpu().numpy().reshape(700, 512), oo) <= TOL["bf16"]
