"""Packed variable-length sequences (cu_seqlens) on the GPU: the packed-sequence
metadata bit-exact against the oracle's definition, the library's chunk tiles and
work units against their restatement, parity with the oracle on chunk grids whose
boundaries do not meet sequence starts (chunks spanning two and three sequences,
sequences shorter than a chunk), packed vs separate runs, empty sequences, and bad
cu_seqlens contents reported through the device status word."""
import numpy as np
import pytest
import torch

from state_space_model_scan_gb300 import inputs as I
from state_space_model_scan_gb300 import _lib
from oracle import varlen_meta
from helpers import TOL, rel_l2, gpu_forward, oracle_forward, flat, to_dev
import unit_schedule

pytestmark = pytest.mark.gpu


def VW(lens, H=4, P=16, G=2, N=16, dtype="f32", Q=None, **kw):
    if Q is None:
        Q = 128 if (dtype == "bf16" and P == 64 and N == 128) else 64
    return I.Workload("v", 1, sum(lens), H, P, G, N, Q, dtype, has_init=True, seqlens=list(lens), **kw)


def cu_of(lens):
    return [0] + list(np.cumsum(lens).astype(int))


GOLDEN_CU = [([1, 1, 4], 4), ([0, 2, 0, 7, 0], 8), ([4, 4, 2], 4), ([3, 0, 7], 4), ([2, 9, 1], 4), ([2, 1], 1)]


@pytest.mark.parametrize("lens,Q", GOLDEN_CU + [
    ([5, 0, 300, 64, 1, 128, 0, 77], 64), ([5, 0, 300, 64, 1, 128, 0, 77], 128),
    ([40, 0, 130, 1, 270, 128], 128), ([0], 16), ([0, 0, 1], 2), ([1000], 256),
    (I.varlen_lengths(16, 512, 8192, 0), 128), (I.varlen_lengths(16, 512, 8192, 0), 256),
])
def test_varlen_metadata_bit_exact(lens, Q):
    """ssd_varlen_metadata: seq_idx, chunk_begin and the segments, bitwise equal to the
    definition-level builder."""
    cu = cu_of(lens)
    L = cu[-1]
    code, seq_idx, begin, segs, status = _lib.varlen_metadata(torch.tensor(cu, dtype=torch.int32, device="cuda"),
                                                              L, Q)
    torch.cuda.synchronize()
    assert code == 0 and int(status.item()) == 0
    ref_segs, ref_begin = varlen_meta.segments(cu, Q)
    assert begin.cpu().tolist() == ref_begin
    n = ref_begin[-1]
    assert [tuple(r) for r in segs[:n].cpu().tolist()] == ref_segs
    assert (segs[n:] == -1).all()            # nothing written past the segments
    if L > 0:
        assert seq_idx.cpu().tolist() == varlen_meta.seq_idx(cu)


@pytest.mark.parametrize("bad", [[0, 10, 5, 20], [1, 10, 20], [0, 10, 19]])
def test_varlen_metadata_rejects_bad_cu(bad):
    code, seq_idx, begin, segs, status = _lib.varlen_metadata(torch.tensor(bad, dtype=torch.int32, device="cuda"),
                                                              20, 4)
    torch.cuda.synchronize()
    assert code == 0 and int(status.item()) == 1
    assert (begin == -1).all() and (segs == -1).all() and (seq_idx == -1).all()


def run_meta(w, inp, algo, seg=0):
    d = to_dev(inp)
    y = torch.empty_like(d["x"])
    S = w.nseqs
    fin = torch.empty(S, w.nheads, w.headdim, w.dstate, device="cuda")
    prob = _lib.problem(1, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.chunk_size, S, algo, seg)
    args = _lib.fwd_args(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], y, D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                         initial_states=d["initial_states"], final_states=fin, cu_seqlens=d["cu_seqlens"])
    ws = torch.empty(_lib.fwd_workspace_size(prob, args), dtype=torch.uint8, device="cuda")
    _lib.check(_lib.ssd_fwd(prob, args, ws), "ssd_fwd")
    torch.cuda.synchronize()
    lay = _lib.debug_layout(prob, args)
    raw = ws.cpu().numpy()
    counts = raw[lay.meta_counts:lay.meta_counts + 16].view(np.int32)
    return raw, lay, counts, d


@pytest.mark.parametrize("algo", ["staged", "fused"])
def test_chunk_tiles_are_the_segments(algo):
    """The forward's chunk tiles (one per segment of a physical chunk) equal the oracle's
    segments renumbered as (seq, row, chunk start t0, end - t0, first - t0)."""
    lens = [5, 0, 300, 64, 1, 128, 0, 77, 2, 3]
    w = VW(lens, P=64, N=128, dtype="bf16", Q=64 if algo == "staged" else 128)
    raw, lay, counts, _ = run_meta(w, I.make_inputs(w), algo)
    Q = lay.qi
    segs, _ = varlen_meta.segments(cu_of(lens), Q)
    ref = [(s, 0, (a // Q) * Q, e - (a // Q) * Q, a - (a // Q) * Q) for (s, a, e) in segs]
    assert counts[0] == len(ref) and counts[3] == 0
    assert unit_schedule.decode_chunks(raw[lay.chunk_info:], counts[0]) == ref


def test_fused_unit_list_matches_the_scheduler_restatement():
    """Scheduler self-consistency: the device-built work-unit list equals the Python
    restatement of the same scheduling rules (tests/unit_schedule.py)."""
    lens = [5, 0, 300, 640, 1, 1280, 0, 77]
    w = VW(lens, P=64, N=128, dtype="bf16")
    raw, lay, counts, _ = run_meta(w, I.make_inputs(w), "fused", seg=2)
    ref = unit_schedule.build(cu=cu_of(lens), Q=128, R=2, KB=4)
    assert lay.units >= 0 and counts[1] == len(ref["units"]) and counts[3] == 0
    assert unit_schedule.decode_units(raw[lay.units:], counts[1]) == ref["units"]


@pytest.mark.parametrize("dtype,P,N,algo", [("f32", 16, 16, "staged"), ("bf16", 16, 16, "staged"),
                                             ("bf16", 64, 128, "fused"), ("bf16", 64, 128, "staged")])
def test_varlen_matches_oracle(dtype, P, N, algo):
    """Sequences starting inside chunks, a chunk holding three sequences (lens 130, 1, 70 at
    Q = 128 or 64), empty and 1-token sequences."""
    w = VW([40, 0, 130, 1, 70, 64, 129, 300], dtype=dtype, P=P, N=N, has_z=True,
           Q=64 if algo == "staged" else None)
    inp = I.make_inputs(w)
    y, fin = gpu_forward(w, inp, algo=algo, seg_chunks=1 if algo == "fused" else 0)
    yo, fo = oracle_forward(w, inp)
    assert rel_l2(flat(y, w.seqlen), yo) <= TOL[dtype]
    assert rel_l2(fin.double().cpu().numpy(), fo) <= TOL[dtype]


@pytest.mark.parametrize("Q", [32, 256])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_varlen_simt_chunk_lengths(Q, dtype):
    """Packed sequences at chunk lengths 32 and 256 (SIMT path): at 256 the first chunk holds
    six sequences (40, 0, 130, 1, 70 tokens and the head of the 64-token one), at 32 most
    sequences span several chunks."""
    w = VW([40, 0, 130, 1, 70, 64, 129, 300], dtype=dtype, has_z=True, Q=Q)
    inp = I.make_inputs(w)
    y, fin = gpu_forward(w, inp, algo="staged")
    yo, fo = oracle_forward(w, inp)
    assert rel_l2(flat(y, w.seqlen), yo) <= TOL[dtype]
    assert rel_l2(fin.double().cpu().numpy(), fo) <= TOL[dtype]


@pytest.mark.parametrize("seg", [1, 2, 5])
def test_varlen_fused_units_across_shared_chunks(seg):
    """Many short and long sequences on the tensor-core path with several units per
    sequence: every tile's rows of the other sequences are masked, every sequence's carry
    starts from its own initial state, mid-chunk."""
    lens = [3, 200, 1, 1, 2, 700, 0, 129, 127, 128, 500, 5]
    w = VW(lens, H=8, P=64, G=2, N=128, dtype="bf16", has_z=True)
    inp = I.make_inputs(w)
    y, fin = gpu_forward(w, inp, algo="fused", seg_chunks=seg)
    yo, fo = oracle_forward(w, inp)
    for s in range(len(lens)):
        c = cu_of(lens)
        if lens[s]:
            assert rel_l2(flat(y, w.seqlen)[c[s]:c[s + 1]], yo[c[s]:c[s + 1]]) <= TOL["bf16"], s
        assert rel_l2(fin[s].double().cpu().numpy(), fo[s]) <= TOL["bf16"], s


@pytest.mark.parametrize("P,N", [(16, 16), (64, 128)])
def test_packed_equals_separate_runs(P, N):
    """Packed on the global chunk grid vs each sequence alone (its own grid): the same
    function, so equal within the tolerance (the chunk boundaries, hence the rounding
    order, differ)."""
    lens = [50, 130, 7, 260]
    w = VW(lens, dtype="bf16", P=P, N=N)
    inp = I.make_inputs(w)
    y, fin = gpu_forward(w, inp)
    cu = inp["cu_seqlens"].tolist()
    for s in range(len(lens)):
        a = dict(inp)
        for k in ("x", "dt_raw", "B", "C", "z"):
            a[k] = inp[k][:, cu[s]:cu[s + 1]].contiguous()
        a["initial_states"] = inp["initial_states"][s:s + 1]
        a["cu_seqlens"] = None
        ws = I.Workload("s", 1, lens[s], w.nheads, w.headdim, w.ngroups, w.dstate, w.chunk_size, "bf16",
                        has_init=True)
        ys, fs = gpu_forward(ws, a)
        assert rel_l2(ys.double().cpu(), y[:, cu[s]:cu[s + 1]].double().cpu()) <= 1e-2
        assert rel_l2(fs[0].double().cpu(), fin[s].double().cpu()) <= 1e-2


@pytest.mark.parametrize("P,N", [(16, 16), (64, 128)])
def test_empty_sequences_return_initial_state(P, N):
    w = VW([0, 10, 0], P=P, N=N, dtype="bf16")
    inp = I.make_inputs(w)
    y, fin = gpu_forward(w, inp)
    assert torch.equal(fin[0].cpu(), inp["initial_states"][0])
    assert torch.equal(fin[2].cpu(), inp["initial_states"][2])


@pytest.mark.parametrize("bad", [[0, 10, 5, 20], [1, 10, 20], [0, 10, 19]])
def test_bad_cu_seqlens_reported_on_device(bad):
    """Contents of cu_seqlens live on the device: the metadata kernel validates them,
    writes SSD_ERR_INVALID_ARGUMENT to the workspace status word and no other
    kernel touches the outputs."""
    L = 20
    w = I.Workload("bad", 1, L, 2, 16, 1, 16, 64, "f32", has_init=True, seqlens=[L])
    inp = I.make_inputs(w)
    d = to_dev(inp)
    S = len(bad) - 1
    cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
    y = torch.full_like(d["x"], 7.0)
    fin = torch.full((S, 2, 16, 16), 7.0, device="cuda")
    init = torch.zeros(S, 2, 16, 16, device="cuda")
    prob = _lib.problem(1, L, 2, 16, 1, 16, 64, S, "staged")
    args = _lib.fwd_args(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], y, D=d["D"], dt_bias=d["dt_bias"],
                         initial_states=init, final_states=fin, cu_seqlens=cu)
    ws = torch.empty(_lib.fwd_workspace_size(prob, args), dtype=torch.uint8, device="cuda")
    assert _lib.ssd_fwd(prob, args, ws) == 0
    assert _lib.query_status(ws) == 1
    assert (y == 7.0).all() and (fin == 7.0).all()


@pytest.mark.parametrize("B,L,seg,algo", [(3, 1000, 2, "fused"), (2, 8192, 0, "fused"), (1, 129, 1, "fused"),
                                          (3, 700, 0, "staged"), (2, 1, 0, "staged")])
def test_fixed_batch_metadata_bit_exact(B, L, seg, algo):
    """Without cu_seqlens the lists have a closed form (one thread per entry): every batch
    row is its own sequence with its own chunk grid; tiles and units as restated."""
    fused = algo == "fused"
    P, N, Q = (64, 128, 128) if fused else (16, 16, 64)
    w = I.Workload("fb", B, L, 4, P, 2, N, Q, "bf16")
    inp = I.make_inputs(w)
    d = to_dev(inp)
    y = torch.empty_like(d["x"])
    prob = _lib.problem(B, L, 4, P, 2, N, Q, 0, algo, seg)
    args = _lib.fwd_args(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], y, D=d["D"], dt_bias=d["dt_bias"])
    ws = torch.empty(_lib.fwd_workspace_size(prob, args), dtype=torch.uint8, device="cuda")
    _lib.check(_lib.ssd_fwd(prob, args, ws), "ssd_fwd")
    torch.cuda.synchronize()
    lay = _lib.debug_layout(prob, args)
    raw = ws.cpu().numpy()
    counts = raw[lay.meta_counts:lay.meta_counts + 16].view(np.int32)
    if fused:
        got = unit_schedule.decode_units(raw[lay.units:], counts[1])
        n = -(-L // 128)
        if prob.seg_chunks:   # units of seg_chunks tiles
            ref = unit_schedule.build(batch=B, seqlen=L, Q=128, R=int(prob.seg_chunks), KB=4)
        else:   # the library's own choice: U units per row (the unit count tells U), n/U tiles each
            U = max(1, int(counts[1]) // B)
            ref = unit_schedule.build(batch=B, seqlen=L, Q=128, R=-(-n // U), KB=4, num=U, den=max(n, 1))
            if n >= 4:   # units of 4 or 5 tiles
                assert {u[4] for u in got} <= {4, 5}
        assert counts[1] == len(ref["units"]) and counts[3] == 0
        assert got == ref["units"]
    else:
        ref = unit_schedule.build(batch=B, seqlen=L, Q=lay.qi)
    assert counts[0] == len(ref["chunks"]) and counts[3] == 0
    assert unit_schedule.decode_chunks(raw[lay.chunk_info:], counts[0]) == ref["chunks"]
