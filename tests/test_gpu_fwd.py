"""Forward parity of the CUDA path against the float64 oracle (GPU).

Tolerances (rel-L2 per output tensor): 1e-4 for fp32 inputs, 1e-2 for bf16
inputs with fp32 state and accumulation.
"""
import dataclasses

import numpy as np
import pytest
import torch

from state_space_model_scan_gb300 import inputs as I
from state_space_model_scan_gb300 import _lib
from helpers import TOL, rel_l2, gpu_forward, oracle_forward, flat, to_dev

pytestmark = pytest.mark.gpu

ALGOS = ["staged"]
BF16_ALGOS = ["staged", "fused"]


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


def check_fwd(w, algo="auto", heads=None, tol=None, **kw):
    inp = I.make_inputs(w)
    y, fin = gpu_forward(w, inp, algo=algo, **kw)
    yo, fo = oracle_forward(w, inp, heads=heads)
    T = w.batch * w.seqlen
    yg = flat(y, T)
    fg = fin.detach().double().cpu().numpy()
    if heads is not None:
        yg, yo = yg[:, heads], yo[:, heads]
        fg, fo = fg[:, heads], fo[:, heads]
    tol = tol or TOL[w.dtype]
    ey, ef = rel_l2(yg, yo), rel_l2(fg, fo)
    assert np.isfinite(yg).all() and np.isfinite(fg).all()
    assert ey <= tol and ef <= tol, (w, ey, ef)
    return ey, ef


@pytest.mark.parametrize("algo", ["staged", "auto"])
def test_tiny_fp32_workload(algo):
    """batch 1, L=256, 4 heads x 16, 1 group, N=16, chunk 64, fp32, no z, zero init."""
    check_fwd(I.named("tiny_f32"), algo=algo)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("case", [
    dict(L=1), dict(L=63), dict(L=65), dict(L=200), dict(L=300),
    dict(B=3, L=130, H=6, G=2),                    # 3 heads per group, ragged tail
    dict(H=6, G=3, P=32, N=64, has_z=True),
    dict(P=128, N=128, L=150, H=2),                # largest compiled tile
    dict(P=16, N=16, L=97),                        # smallest
    dict(has_D=False, has_dt_bias=False, has_z=True, has_init=True, L=180),
])
def test_fp32_cases(algo, case):
    check_fwd(W(**case), algo=algo)


@pytest.mark.parametrize("algo", BF16_ALGOS)
@pytest.mark.parametrize("case", [
    dict(L=1000, H=8, P=64, G=2, N=128, Q=128, has_z=True, has_init=True),
    dict(B=2, L=333, H=4, P=64, G=1, N=128, Q=128, has_z=False),
    dict(L=1, H=2, P=64, G=1, N=128, Q=128, has_init=True),
    dict(L=127, H=6, P=64, G=2, N=128, Q=128, has_z=True),
    dict(B=3, L=129, H=3, P=64, G=3, N=128, Q=128, has_D=False, has_dt_bias=False),
])
def test_bf16_cases(algo, case):
    check_fwd(W(dtype="bf16", **for_algo(case, algo)), algo=algo)


@pytest.mark.parametrize("Q", [32, 128, 256])
@pytest.mark.parametrize("case", [
    dict(L=300, H=4, P=16, G=2, N=16, has_z=True, has_init=True),   # ragged tail, several chunks
    dict(B=2, L=97, H=3, P=32, G=1, N=64),                          # shorter than a 128/256 chunk
    dict(L=513, H=2, P=64, G=1, N=128, has_init=True),              # the tensor-core shape, on SIMT
])
def test_simt_chunk_lengths(Q, case):
    """The SIMT forward at chunk lengths 32, 128 and 256 (the same exact function; only the
    chunking, and so the rounding order, differs), fp32 and bf16 inputs."""
    check_fwd(W(Q=Q, **case), algo="staged")
    check_fwd(W(Q=Q, dtype="bf16", **case), algo="staged")


@pytest.mark.parametrize("Q", [16, 512])
def test_chunk_lengths_no_path_computes_are_refused(Q):
    """No silent re-chunking: a chunk length that no path computes is refused."""
    for dtype, P, N in (("f32", 16, 16), ("bf16", 64, 128)):
        w = W(L=300, P=P, N=N, Q=Q, dtype=dtype)
        inp = I.make_inputs(w)
        with pytest.raises(_lib.SSDError) as e:
            gpu_forward(w, inp)
        assert e.value.code == 2


@pytest.mark.parametrize("seg", [1, 2, 3, 4, 5])
def test_fused_units_and_lookback(seg):
    """Several work units per sequence: every unit's carry-in comes from the
    predecessors' published aggregates / end states."""
    w = W(B=2, L=1900, H=8, P=64, G=4, N=128, Q=128, dtype="bf16", has_z=True, has_init=True)
    check_fwd(w, algo="fused", seg_chunks=seg)


def test_fused_matches_staged_closely():
    w = W(L=700, H=4, P=64, G=1, N=128, Q=128, dtype="bf16", has_z=True, has_init=True)
    inp = I.make_inputs(w)
    y1, f1 = gpu_forward(w, inp, algo="fused")
    y2, f2 = gpu_forward(dataclasses.replace(w, chunk_size=64), inp, algo="staged")
    assert rel_l2(y1.double().cpu(), y2.double().cpu()) < 1e-2
    assert rel_l2(f1.double().cpu(), f2.double().cpu()) < 1e-2


def test_fused_rejects_unsupported_shapes():
    w = W(L=64, H=2, P=32, N=128, Q=128, dtype="bf16")
    inp = I.make_inputs(w)
    with pytest.raises(_lib.SSDError) as e:
        gpu_forward(w, inp, algo="fused")
    assert e.value.code == 2
    w = W(L=64, H=2, P=64, N=128, Q=128, dtype="f32")
    inp = I.make_inputs(w)
    with pytest.raises(_lib.SSDError) as e:
        gpu_forward(w, inp, algo="fused")
    assert e.value.code == 2


def test_stage_intermediates_match_chunked_oracle():
    """dt, cs and carry-in states left in the workspace by the staged path equal the
    chunkwise float64 decomposition at the same internal chunk length."""
    from oracle import chunked64
    w = W(L=150, H=3, P=16, G=1, N=16, has_init=True, has_z=True)
    inp = I.make_inputs(w)
    d = to_dev(inp)
    y = torch.empty_like(d["x"])
    fin = torch.empty(1, 3, 16, 16, device="cuda")
    prob = _lib.problem(1, w.seqlen, 3, 16, 1, 16, 64, 0, "staged")
    args = _lib.fwd_args(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], y, D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                         initial_states=d["initial_states"], final_states=fin)
    n = _lib.fwd_workspace_size(prob, args)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    _lib.check(_lib.ssd_fwd(prob, args, ws), "ssd_fwd")
    torch.cuda.synchronize()
    lay = _lib.debug_layout(prob, args)
    Q = lay.qi
    nch = -(-w.seqlen // Q)
    raw = ws.cpu().numpy()
    counts = raw[lay.meta_counts:lay.meta_counts + 16].view(np.int32)
    assert counts[0] == nch and counts[3] == 0
    dtg = raw[lay.dt:lay.dt + 4 * nch * 3 * Q].view(np.float32).reshape(nch, 3, Q)
    csg = raw[lay.cs:lay.cs + 4 * nch * 3 * Q].view(np.float32).reshape(nch, 3, Q)
    stg = raw[lay.states:lay.states + 4 * nch * 3 * 256].view(np.float32).reshape(nch, 3, 16, 16)
    o = I.to_oracle(inp, w)
    v = o["dt_raw"] + o["dt_bias"][None, :]
    dt = np.where(v > 0, v + np.log1p(np.exp(-np.abs(v))), np.log1p(np.exp(np.minimum(v, 0))))
    for h in range(3):
        _, _, inter = chunked64.forward_one(o["x"][:, h], dt[:, h], o["A"][h], o["B"][:, 0], o["C"][:, 0], Q,
                                            o["init"][0, h])
        assert rel_l2(dtg[:, h], inter["dt"]) < 1e-6
        assert rel_l2(csg[:, h], inter["cs"]) < 1e-5
        assert rel_l2(stg[:, h], inter["carry_in"]) < 1e-5


@pytest.mark.parametrize("P,N,dtype,tol", [(32, 32, "f32", 1e-5), (64, 128, "bf16", 1e-2)])
def test_split_sequence_invariance_gpu(P, N, dtype, tol):
    """run(L1) -> final -> run(L2, init=final) equals run(L1+L2), also for splits that
    are not chunk-aligned."""
    w = W(L=300, H=4, P=P, G=2, N=N, has_init=True, has_z=True, dtype=dtype)
    inp = I.make_inputs(w)
    y, fin = gpu_forward(w, inp)
    for L1 in (64, 101, 128):
        a = dict(inp)
        b = dict(inp)
        for k in ("x", "dt_raw", "B", "C", "z"):
            a[k] = inp[k][:, :L1].contiguous()
            b[k] = inp[k][:, L1:].contiguous()
        y1, f1 = gpu_forward(dataclasses.replace(w, seqlen=L1), a)
        b["initial_states"] = f1.cpu()
        y2, f2 = gpu_forward(dataclasses.replace(w, seqlen=300 - L1), b)
        ycat = torch.cat([y1, y2], 1)
        assert rel_l2(ycat.double().cpu(), y.double().cpu()) < tol
        assert rel_l2(f2.double().cpu(), fin.double().cpu()) < tol


@pytest.mark.parametrize("P,N,dtype", [(32, 32, "f32"), (64, 128, "bf16")])
def test_strided_views_of_packed_buffer(P, N, dtype):
    """x, B and C as strided views into one packed [B, L, H*P + 2*G*N] buffer."""
    Bsz, L, H, G = 2, 300, 4, 2
    w = W(B=Bsz, L=L, H=H, P=P, G=G, N=N, has_z=True, dtype=dtype)
    inp = I.make_inputs(w)
    packed = torch.cat([inp["x"].reshape(Bsz, L, H * P), inp["B"].reshape(Bsz, L, G * N),
                        inp["C"].reshape(Bsz, L, G * N)], -1).cuda()
    xs = packed[..., :H * P].view(Bsz, L, H, P)
    Bs = packed[..., H * P:H * P + G * N].view(Bsz, L, G, N)
    Cs = packed[..., H * P + G * N:].view(Bsz, L, G, N)
    assert not xs.is_contiguous()
    d = to_dev(inp)
    from state_space_model_scan_gb300.api import ssd_forward
    y1, f1 = ssd_forward(xs, d["dt_raw"], d["A"], Bs, Cs, D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                         chunk_size=w.chunk_size)
    y2, f2 = ssd_forward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                         chunk_size=w.chunk_size)
    assert torch.equal(y1, y2) and torch.equal(f1, f2)


@pytest.mark.parametrize("P,N", [(32, 64), (64, 128)])
def test_deterministic_and_every_output_written(P, N):
    w = W(L=1257, H=4, P=P, G=2, N=N, dtype="bf16", has_z=True, has_init=True)
    inp = I.make_inputs(w)
    d = to_dev(inp)
    from state_space_model_scan_gb300.api import ssd_forward
    outs = []
    for _ in range(2):
        y = torch.full_like(d["x"], float("nan"))
        f = torch.full((1, 4, P, N), float("nan"), device="cuda")
        ssd_forward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                    initial_states=d["initial_states"], chunk_size=w.chunk_size, y=y, final_states=f, seg_chunks=1)
        torch.cuda.synchronize()
        assert torch.isfinite(y.float()).all() and torch.isfinite(f).all()
        outs.append((y, f))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_zero_length_batch():
    w = W(L=0, H=2, P=16, N=16, has_init=True)
    inp = I.make_inputs(w)
    y, fin = gpu_forward(w, inp)
    assert y.numel() == 0
    assert torch.equal(fin.cpu(), inp["initial_states"])
