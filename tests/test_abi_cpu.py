"""The C ABI on the CPU: the library loads, exports every declared symbol, and
host-side validation returns the documented status codes (no GPU needed: every
call here fails validation before anything is enqueued)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssd.h")


@pytest.fixture(scope="module")
def lib():
    from state_space_model_scan_gb300 import build, _lib
    build.build()
    return _lib


def declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_[a-z_0-9]+)\s*\(", txt)))


def test_library_exports_every_declared_symbol(lib):
    L = lib.load()
    names = declared_functions()
    assert set(names) == set(lib.EXPORTS), names
    for n in names:
        assert hasattr(L, n), n


def test_abi_version_and_status_strings(lib):
    assert lib.abi_version() == 5
    for code, name in lib.STATUS_NAMES.items():
        assert lib.status_string(code) == name
    assert lib.status_string(99) == "SSD_ERR_UNKNOWN"


def _fake(dtype, strides, ptr=0x100000):
    t = lib_mod().Tensor()
    t.ptr = ptr
    t.dtype = dtype
    for i, s in enumerate(strides):
        t.stride[i] = s
    return t


def lib_mod():
    from state_space_model_scan_gb300 import _lib
    return _lib


def good_case(Bsz=2, L=100, H=4, P=16, G=2, N=16, bf16=True):
    m = lib_mod()
    dt_ = m.SSD_BF16 if bf16 else m.SSD_F32
    xs = [L * H * P, H * P, P, 1]
    bs = [L * G * N, G * N, N, 1]
    a = m.FwdArgs()
    a.x = _fake(dt_, xs)
    a.y = _fake(dt_, xs)
    a.z = _fake(dt_, xs)
    a.B = _fake(dt_, bs)
    a.C = _fake(dt_, bs)
    a.dt = _fake(m.SSD_F32, [L * H, H, 1])
    a.A = _fake(m.SSD_F32, [1])
    a.D = _fake(m.SSD_F32, [1])
    a.dt_bias = _fake(m.SSD_F32, [1])
    a.final_states = _fake(m.SSD_F32, [H * P * N, P * N, N, 1])
    p = m.problem(Bsz, L, H, P, G, N, 64)
    return p, a


def ws_size(p, a):
    m = lib_mod()
    n = ctypes.c_size_t(0)
    rc = m.load().ssd_fwd_workspace_size(ctypes.byref(p), ctypes.byref(a), ctypes.byref(n))
    return rc, n.value


def test_valid_problem_has_workspace(lib):
    p, a = good_case()
    rc, n = ws_size(p, a)
    assert rc == 0 and n > 0


@pytest.mark.parametrize("mutate,code", [
    (lambda p, a: setattr(p, "ngroups", 3), 1),                  # H % G != 0
    (lambda p, a: setattr(p, "headdim", 48), 2),                 # P outside the compiled set
    (lambda p, a: setattr(p, "dstate", 256), 2),                 # N outside the compiled set
    (lambda p, a: setattr(p, "chunk_size", 100), 2),             # not a power of two
    (lambda p, a: setattr(p, "chunk_size", 0), 1),
    (lambda p, a: setattr(p, "batch", 0), 1),
    (lambda p, a: setattr(a.x, "ptr", None), 1),                 # missing required input
    (lambda p, a: setattr(a.y, "ptr", None), 1),                 # missing required output
    (lambda p, a: setattr(a.B, "dtype", 0), 1),                  # dtype mix
    (lambda p, a: setattr(a.dt, "dtype", 1), 1),                 # dt must be f32
    (lambda p, a: a.x.stride.__setitem__(3, 2), 1),              # innermost stride must be 1
    (lambda p, a: a.final_states.stride.__setitem__(0, 7), 1),   # states must be contiguous
    (lambda p, a: setattr(p, "nseqs", 5), 1),                    # nseqs without cu_seqlens must match batch
    (lambda p, a: setattr(a, "cu_seqlens", 0x2000), 1),          # cu_seqlens needs batch 1
    (lambda p, a: setattr(p, "algo", 7), 1),
])
def test_validation_codes(lib, mutate, code):
    p, a = good_case()
    mutate(p, a)
    rc, _ = ws_size(p, a)
    assert rc == code
    # the call itself fails the same way before touching the device
    m = lib_mod()
    rc2 = m.load().ssd_fwd(ctypes.byref(p), ctypes.byref(a), ctypes.c_void_p(0x100000), ctypes.c_size_t(1 << 40),
                           None)
    assert rc2 == code


@pytest.mark.parametrize("P,N,bf16,Q,algo,aligned,code,qi", [
    (16, 16, True, 64, "auto", True, 0, 64),        # SIMT computes 32-, 64-, 128- and 256-token chunks
    (16, 16, True, 32, "auto", True, 0, 32),
    (16, 16, True, 128, "auto", True, 0, 128),
    (16, 16, False, 256, "auto", True, 0, 256),
    (16, 16, True, 16, "auto", True, 2, None),      # ... and nothing shorter
    (64, 128, True, 128, "auto", True, 0, 128),     # tensor-core tile set: 128-token chunks
    (64, 128, True, 64, "auto", True, 0, 64),       # same shape at 64: the SIMT path, honoured
    (64, 128, True, 256, "auto", True, 0, 256),     # ... and at 256: SIMT, never re-chunked
    (64, 128, True, 128, "fused", True, 0, 128),
    (64, 128, True, 64, "fused", True, 2, None),    # the tensor-core path computes 128 only
    (64, 128, True, 256, "split", True, 2, None),
    (64, 128, True, 128, "staged", True, 0, 128),   # an explicit SIMT run at 128
    (64, 128, True, 128, "auto", False, 3, None),   # tensor-core chunk length, strides break the TMA rule
    (64, 128, False, 128, "auto", True, 0, 128),    # fp32 inputs run SIMT (here at 128)
    (64, 64, True, 128, "auto", True, 0, 128),      # dstate 64: the tensor-core tiles' zero-extended half
    (64, 64, True, 128, "split", True, 0, 128),
    (64, 32, True, 128, "auto", True, 0, 128),      # dstate 32: the zero-extended tensor-core tiles too
    (64, 32, True, 64, "auto", True, 0, 64),
])
def test_chunk_size_is_honoured(lib, P, N, bf16, Q, algo, aligned, code, qi):
    """Each chunk_size outcome of the forward: the path that computes exactly that chunk
    length, or SSD_ERR_UNSUPPORTED / SSD_ERR_MISALIGNED; the debug layout reports the chunk used."""
    m = lib_mod()
    p, a = good_case(P=P, N=N, bf16=bf16)
    p.chunk_size = Q
    p.algo = m.ALGO[algo]
    if not aligned:
        a.x.stride[2] = P + 4
        a.x.stride[1] = 4 * (P + 4)
    rc, _ = ws_size(p, a)
    assert rc == code
    if code == 0:
        lay = m.DebugLayout()
        assert m.load().ssd_fwd_debug_layout(ctypes.byref(p), ctypes.byref(a), ctypes.byref(lay)) == 0
        assert lay.qi == qi


@pytest.mark.parametrize("P,N,bf16,Q,code", [
    (16, 16, True, 32, 0),      # the SIMT backward: 32- and 64-token chunks
    (16, 16, False, 64, 0),
    (16, 16, True, 128, 2),     # its per-chunk tiles at 128 or 256 exceed shared memory
    (16, 16, True, 256, 2),
    (64, 128, True, 128, 0),    # the tensor-core backward: 128
    (64, 128, False, 128, 2),   # fp32 inputs at 128: no backward computes it
])
def test_bwd_chunk_size_is_honoured(lib, P, N, bf16, Q, code):
    """Each chunk_size outcome of the backward (never re-chunked)."""
    m = lib_mod()
    p, a = good_case(P=P, N=N, bf16=bf16)
    p.chunk_size = Q
    b = _tc_bwd_args(p, a)
    n = ctypes.c_size_t(0)
    assert m.load().ssd_bwd_workspace_size(ctypes.byref(p), ctypes.byref(b), ctypes.byref(n)) == code


def test_varlen_metadata_validates_on_host(lib):
    """Argument checks of ssd_varlen_metadata happen before any launch."""
    m = lib_mod().load()
    d = ctypes.c_void_p(0x100000)
    assert m.ssd_varlen_metadata(None, 2, 10, 4, d, d, d, d, None) == 1
    assert m.ssd_varlen_metadata(d, 2, 10, 4, d, None, d, d, None) == 1
    assert m.ssd_varlen_metadata(d, 2, 10, 4, d, d, None, d, None) == 1
    assert m.ssd_varlen_metadata(d, 2, 10, 4, d, d, d, None, None) == 1
    assert m.ssd_varlen_metadata(d, 0, 10, 4, d, d, d, d, None) == 1
    assert m.ssd_varlen_metadata(d, 2, -1, 4, d, d, d, d, None) == 1
    assert m.ssd_varlen_metadata(d, 2, 10, 0, d, d, d, d, None) == 1
    assert m.ssd_varlen_metadata(d, 2, 10, 1 << 17, d, d, d, d, None) == 2
    assert m.ssd_varlen_metadata(d, (1 << 24) + 1, 10, 4, d, d, d, d, None) == 2


def test_workspace_checks(lib):
    m = lib_mod()
    p, a = good_case()
    rc, n = ws_size(p, a)
    assert m.load().ssd_fwd(ctypes.byref(p), ctypes.byref(a), ctypes.c_void_p(0x100000), ctypes.c_size_t(n - 1),
                            None) == 4
    assert m.load().ssd_fwd(ctypes.byref(p), ctypes.byref(a), None, ctypes.c_size_t(n), None) == 4
    assert m.load().ssd_fwd(ctypes.byref(p), ctypes.byref(a), ctypes.c_void_p(0x100010), ctypes.c_size_t(n),
                            None) == 3


def test_bwd_requires_matching_gradients(lib):
    m = lib_mod()
    p, a = good_case()
    b = m.BwdArgs()
    b.fwd = a
    xs = [a.x.stride[i] for i in range(4)]
    for f in ("dy", "dx", "dz"):
        setattr(b, f, _fake(a.x.dtype, xs))
    for f in ("dB", "dC"):
        setattr(b, f, _fake(a.x.dtype, [a.B.stride[i] for i in range(4)]))
    b.ddt = _fake(m.SSD_F32, [a.dt.stride[i] for i in range(3)])
    for f in ("dA", "dD", "ddt_bias"):
        setattr(b, f, _fake(m.SSD_F32, [1]))
    n = ctypes.c_size_t(0)
    assert m.load().ssd_bwd_workspace_size(ctypes.byref(p), ctypes.byref(b), ctypes.byref(n)) == 0
    b.dz = m.Tensor()      # z given but dz missing
    assert m.load().ssd_bwd_workspace_size(ctypes.byref(p), ctypes.byref(b), ctypes.byref(n)) == 1


def test_unit_schedule_restatement():
    """The Python restatement of the library's tile and unit lists (a scheduler
    self-consistency check, built on the oracle's segments) on two hand-worked cases."""
    import unit_schedule as meta
    m = meta.build(cu=[0, 5, 5, 300], Q=64, R=2, KB=8)
    # tiles: (seq, row, t0 of the physical chunk, end - t0, first - t0)
    assert m["chunks"] == [(0, 0, 0, 5, 0), (2, 0, 0, 64, 5), (2, 0, 64, 64, 0), (2, 0, 128, 64, 0),
                           (2, 0, 192, 64, 0), (2, 0, 256, 44, 0)]
    assert [u[:5] for u in m["units"]] == [(0, 0, 0, 5, 1), (2, 0, 0, 128, 2), (2, 0, 128, 128, 2),
                                           (2, 0, 256, 44, 1)]
    assert [u[5] for u in m["units"]] == [-1, -1, 1, 2]
    assert [u[6] for u in m["units"]] == [0, 0, 1, 2]
    assert [u[7] for u in m["units"]] == [1, 0, 0, 1]
    assert [u[8] for u in m["units"]] == [0, 5, 0, 0]
    # blocks of two units; sequence 1 starts inside physical chunk 4 and has 6 tiles
    m = meta.build(cu=[0, 300, 600], Q=64, R=1, KB=2)
    assert [(u[0], u[6]) for u in m["units"]] == [(0, 0), (0, 1), (1, 0), (1, 1), (0, 2), (0, 3), (1, 2), (1, 3),
                                                  (0, 4), (1, 4), (1, 5)]
    assert [u[5] for u in m["units"]] == [-1, 0, -1, 2, 1, 4, 3, 6, 5, 7, 9]
    assert [(u[2], u[3], u[8]) for u in m["units"] if u[0] == 1][:2] == [(256, 64, 44), (320, 64, 0)]


def test_unit_schedule_balanced_units():
    """Units of one sequence differ by at most one tile, the larger ones first, and
    cover its tiles exactly; a units-per-tile ratio above 1/R raises the count."""
    import unit_schedule as meta
    m = meta.build(batch=2, seqlen=64 * 9, Q=64, R=4, KB=4)
    assert [u[4] for u in m["units"] if u[0] == 0] == [3, 3, 3]
    m = meta.build(batch=1, seqlen=128 * 64 - 5, Q=128, R=4, KB=4, num=19, den=64)
    sizes = [u[4] for u in m["units"]]
    assert sizes == [4] * 7 + [3] * 12
    pos = 0
    for u in sorted(m["units"], key=lambda r: r[6]):
        assert u[2] == pos and u[3] == min(u[4] * 128, 128 * 64 - 5 - pos)
        pos += u[3]
    assert pos == 128 * 64 - 5
    # the library's choice at 64 chunks and 64 heads on 152 SMs: 14 units of 5 or 4 tiles
    m = meta.build(batch=1, seqlen=128 * 64, Q=128, R=5, KB=4, num=14, den=64)
    assert [u[4] for u in sorted(m["units"], key=lambda r: r[6])] == [5] * 8 + [4] * 6
    # never fewer units than ceil(n/R), never more than n
    assert len(meta.build(batch=1, seqlen=640, Q=64, R=4, num=1, den=100)["units"]) == 3
    assert len(meta.build(batch=1, seqlen=640, Q=64, R=4, num=5, den=1)["units"]) == 10


def test_selftest_bounded_wait_validates_on_host(lib):
    """Argument checks happen before any launch (no GPU needed)."""
    import ctypes
    m = lib.load()
    assert m.ssd_selftest_bounded_wait(None, ctypes.c_size_t(4096), 10, None) == 1


def _tc_case(Bsz=2, L=1000, H=8, G=2, cu=None):
    """A problem on the tensor-core path (bf16, headdim 64, dstate 128), fake 16-byte-aligned pointers."""
    m = lib_mod()
    p, a = good_case(Bsz=Bsz, L=L, H=H, P=64, G=G, N=128)
    p.chunk_size = 128
    if cu is not None:
        p.batch = 1
        p.nseqs = cu
        a.cu_seqlens = 0x300000
        for t in ("x", "y", "z", "B", "C", "dt"):
            getattr(a, t).stride[0] = 0
        a.final_states = m.Tensor()
    return p, a


def _chunk_states_size(p, a):
    m = lib_mod()
    n = ctypes.c_size_t(0)
    rc = m.load().ssd_chunk_states_size(ctypes.byref(p), ctypes.byref(a), ctypes.byref(n))
    return rc, n.value


def test_chunk_states_size(lib):
    """One bf16 64 x 128 tile per (chunk of 128 tokens, head), for the largest chunk count."""
    p, a = _tc_case(Bsz=2, L=1000, H=8)
    assert _chunk_states_size(p, a) == (0, 2 * 8 * 8 * 64 * 128 * 2)
    p, a = _tc_case(L=1000, H=8, cu=5)   # packed: ceil(L / 128) + nseqs chunks at most
    assert _chunk_states_size(p, a) == (0, (8 + 5) * 8 * 64 * 128 * 2)
    p, a = good_case()                   # SIMT path: no chunk-state buffer
    assert _chunk_states_size(p, a)[0] == 2


def test_chunk_states_argument_checks(lib):
    m = lib_mod()
    p, a = good_case()
    a.chunk_states = 0x400000            # SIMT path does not take kept states
    assert ws_size(p, a)[0] == 2
    p, a = _tc_case()
    a.chunk_states = 0x400008            # not 16-byte aligned
    assert ws_size(p, a)[0] == 3
    a.chunk_states = 0x400000
    assert ws_size(p, a)[0] == 0


def test_bwd_workspace_drops_states_when_kept(lib):
    """Given the forward's chunk states, the backward reserves no workspace copy of them."""
    m = lib_mod()
    p, a = _tc_case(Bsz=1, L=4096, H=8)
    b = m.BwdArgs()
    xs = [a.x.stride[i] for i in range(4)]
    for f in ("dy", "dx", "dz"):
        setattr(b, f, _fake(a.x.dtype, xs))
    for f in ("dB", "dC"):
        setattr(b, f, _fake(a.x.dtype, [a.B.stride[i] for i in range(4)]))
    b.ddt = _fake(m.SSD_F32, [a.dt.stride[i] for i in range(3)])
    for f in ("dA", "dD", "ddt_bias"):
        setattr(b, f, _fake(m.SSD_F32, [1]))
    n0, n1 = ctypes.c_size_t(0), ctypes.c_size_t(0)
    b.fwd = a
    assert m.load().ssd_bwd_workspace_size(ctypes.byref(p), ctypes.byref(b), ctypes.byref(n0)) == 0
    a.chunk_states = 0x400000
    b.fwd = a
    assert m.load().ssd_bwd_workspace_size(ctypes.byref(p), ctypes.byref(b), ctypes.byref(n1)) == 0
    assert n0.value - n1.value >= 32 * 8 * 64 * 128 * 2


def _tc_bwd_args(p, a):
    m = lib_mod()
    b = m.BwdArgs()
    b.fwd = a
    xs = [a.x.stride[i] for i in range(4)]
    for f in ("dy", "dx", "dz"):
        setattr(b, f, _fake(a.x.dtype, xs))
    for f in ("dB", "dC"):
        setattr(b, f, _fake(a.x.dtype, [a.B.stride[i] for i in range(4)]))
    b.ddt = _fake(m.SSD_F32, [a.dt.stride[i] for i in range(3)])
    for f in ("dA", "dD", "ddt_bias"):
        setattr(b, f, _fake(m.SSD_F32, [1]))
    return b


@pytest.mark.parametrize("field,value,code", [
    ("bwd_heads", 0, 0), ("bwd_heads", 2, 0), ("bwd_heads", 12, 0),   # 12 heads per group
    ("bwd_heads", 5, 1),                                                # not a divisor of 12
    ("bwd_heads", 33, 1), ("bwd_heads", -1, 1),
    ("seg_chunks", 4, 0), ("seg_chunks", 5, 2),                         # the backward's recompute: 4 at most
    ("seg_chunks", 9, 1),
    ("reserved0", 1, 1),
])
def test_bwd_planner_validation(lib, field, value, code):
    """The tensor-core backward's planning choices are checked on the host (no GPU)."""
    m = lib_mod()
    p, a = _tc_case(Bsz=1, L=1000, H=12, G=1)
    p.algo = 2   # fused
    setattr(p, field, value)
    b = _tc_bwd_args(p, a)
    n = ctypes.c_size_t(0)
    assert m.load().ssd_bwd_workspace_size(ctypes.byref(p), ctypes.byref(b), ctypes.byref(n)) == code


def test_fwd_accepts_five_chunk_units(lib):
    p, a = _tc_case(Bsz=1, L=1000, H=12, G=1)
    p.algo = 2
    p.seg_chunks = 5
    assert ws_size(p, a)[0] == 0
    p.seg_chunks = 6
    assert ws_size(p, a)[0] == 2


@pytest.mark.parametrize("field,value,code", [
    ("width", 0, 1), ("group_size", 0, 1), ("group_size", 7, 1),     # 7 does not divide 4096
    ("group_size", 12, 2),                                           # not a multiple of 8 (divides 4092? no: width 48 below)
    ("group_size", 8192, 2), ("eps", -1.0, 1), ("dtype", 5, 1), ("rows", -1, 1),
    ("flags", 1, 0), ("flags", 2, 0), ("flags", 3, 0),               # LayerNorm, gate after, both
    ("flags", 4, 1), ("flags", -1, 1),                               # no other flag
])
def test_gated_norm_validation(lib, field, value, code):
    """Host-side checks of the gated normalisation entry points (nothing reaches the device)."""
    m = lib_mod()
    p = m.NormProblem(16, 48 if field == "group_size" and value == 12 else 4096, 512, 1e-5, m.SSD_BF16, 0)
    if field == "group_size" and value == 8192:
        p.width = 8192
    setattr(p, field, value)
    n = ctypes.c_size_t(0)
    assert m.load().ssd_gated_norm_bwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == code
    if code != 0:   # (a valid problem would go on to launch)
        d = ctypes.c_void_p(0x100000)
        assert m.load().ssd_gated_norm_fwd(ctypes.byref(p), d, 4096, None, 0, d, d, 4096, d, None) == code


def test_gated_norm_pointer_checks(lib):
    m = lib_mod()
    p = m.NormProblem(16, 4096, 512, 1e-5, m.SSD_BF16, 0)
    d = ctypes.c_void_p(0x100000)
    f = m.load().ssd_gated_norm_fwd
    assert f(ctypes.byref(p), None, 4096, None, 0, d, d, 4096, d, None) == 1               # y required
    assert f(ctypes.byref(p), ctypes.c_void_p(0x100008), 4096, None, 0, d, d, 4096, d, None) == 3   # 16-byte rule
    assert f(ctypes.byref(p), d, 4100, None, 0, d, d, 4096, d, None) == 3                  # stride % 8
    assert f(ctypes.byref(p), d, 100, None, 0, d, d, 4096, d, None) == 1                   # stride < width
    n = ctypes.c_size_t(0)
    assert m.load().ssd_gated_norm_bwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0 and n.value > 0
    b = m.load().ssd_gated_norm_bwd
    assert b(ctypes.byref(p), d, 4096, None, 0, d, d, d, 4096, d, 4096, None, 0, d, d, ctypes.c_size_t(n.value - 4),
             None) == 4                                                                    # workspace too small


@pytest.mark.parametrize("field,value,code", [
    ("batch", 0, 1), ("seqlen", -1, 1), ("channels", 0, 1), ("width", 0, 1), ("reserved", 1, 1),
    ("dtype", 7, 1), ("activation", 2, 1), ("nseqs", 3, 1),       # nseqs without cu_seqlens
    ("width", 9, 2), ("channels", 20, 2),                          # width 1..8, channels % 8
])
def test_conv1d_validation(lib, field, value, code):
    """Host-side checks of the conv1d entry points (nothing reaches the device)."""
    m = lib_mod()
    p = m.ConvProblem(2, 64, 64, 4, 0, m.SSD_BF16, 1, 0, 0)
    setattr(p, field, value)
    n = ctypes.c_size_t(0)
    assert m.load().ssd_conv1d_bwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == code
    d = ctypes.c_void_p(0x100000)
    assert m.load().ssd_conv1d_fwd(ctypes.byref(p), d, 64 * 64, 64, d, None, None, d, 64 * 64, 64, None) == code


def test_conv1d_pointer_and_layout_checks(lib):
    m = lib_mod()
    p = m.ConvProblem(2, 64, 64, 4, 0, m.SSD_BF16, 1, 0, 0)
    d = ctypes.c_void_p(0x100000)
    f = m.load().ssd_conv1d_fwd
    assert f(ctypes.byref(p), None, 4096, 64, d, None, None, d, 4096, 64, None) == 1        # u required
    assert f(ctypes.byref(p), d, 4096, 64, None, None, None, d, 4096, 64, None) == 1        # weight required
    assert f(ctypes.byref(p), ctypes.c_void_p(0x100008), 4096, 64, d, None, None, d, 4096, 64, None) == 3
    assert f(ctypes.byref(p), d, 4096, 60, d, None, None, d, 4096, 64, None) == 1           # token stride < channels
    assert f(ctypes.byref(p), d, 4096, 72 + 4, d, None, None, d, 4096, 64, None) == 1       # rows overlap
    assert f(ctypes.byref(p), d, 64 * 76, 76, d, None, None, d, 4096, 64, None) == 3        # stride % 8
    # packed sequences: batch 1 and nseqs >= 1
    p2 = m.ConvProblem(2, 64, 64, 4, 2, m.SSD_BF16, 1, 0, 0)
    assert f(ctypes.byref(p2), d, 4096, 64, d, None, d, d, 4096, 64, None) == 1
    p2.batch, p2.nseqs = 1, 0
    assert f(ctypes.byref(p2), d, 4096, 64, d, None, d, d, 4096, 64, None) == 1
    # empty sequence: nothing to check or launch
    p3 = m.ConvProblem(1, 0, 64, 4, 0, m.SSD_F32, 0, 0, 0)
    assert f(ctypes.byref(p3), None, 0, 0, d, None, None, None, 0, 0, None) == 0
    n = ctypes.c_size_t(0)
    assert m.load().ssd_conv1d_bwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    assert n.value == 2 * 1 * 64 * 5 * 4                     # 2 rows x 1 tile of 64 tokens x channels x (width+1) f32
    b = m.load().ssd_conv1d_bwd
    args = lambda ws, nb, dw=d, db=None, bias=None: (ctypes.byref(p), d, 4096, 64, d, bias, None, d, 4096, 64,
                                                     d, 4096, 64, dw, db, ws, ctypes.c_size_t(nb), None)
    assert b(*args(d, n.value - 4)) == 4                     # workspace too small
    assert b(*args(None, n.value)) == 4
    assert b(*args(ctypes.c_void_p(0x100004), n.value)) == 3
    assert b(*args(d, n.value, dw=None)) == 1                # dweight required
    assert b(*args(d, n.value, bias=d)) == 1                 # bias given, dbias missing


@pytest.mark.parametrize("field,value,code", [
    ("batch", 0, 1), ("seqlen", -1, 1), ("nheads", 0, 1), ("chunk_size", 0, 1),
    ("headdim", 32, 2), ("dstate", 128, 2), ("chunk_size", 128, 2),   # compiled set: 64 / 64 / 64
])
def test_complex_validation(lib, field, value, code):
    """Host-side checks of the complex-A scan entry point (nothing reaches the device)."""
    m = lib_mod()
    p = m.ComplexProblem(2, 128, 4, 64, 64, 64)
    setattr(p, field, value)
    d = ctypes.c_void_p(0x100000)
    ws = ctypes.c_size_t(256)
    f = m.load().ssd_complex_fwd
    assert f(ctypes.byref(p), d, d, d, d, d, None, d, None, None, d, ws, None) == code


def test_complex_pointer_checks(lib):
    m = lib_mod()
    p = m.ComplexProblem(2, 128, 4, 64, 64, 64)
    n = ctypes.c_size_t(0)
    assert m.load().ssd_complex_fwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0 and n.value == 256
    d, odd = ctypes.c_void_p(0x100000), ctypes.c_void_p(0x100008)
    f = m.load().ssd_complex_fwd
    ws = ctypes.c_size_t(n.value)
    assert f(ctypes.byref(p), None, d, d, d, d, None, d, None, None, d, ws, None) == 1      # x required
    assert f(ctypes.byref(p), d, d, None, d, d, None, d, None, None, d, ws, None) == 1      # A required
    assert f(ctypes.byref(p), d, d, d, d, d, None, None, None, None, d, ws, None) == 1      # y_real required
    assert f(ctypes.byref(p), d, d, d, d, d, None, d, None, None, d, ctypes.c_size_t(8), None) == 4
    assert f(ctypes.byref(p), d, d, d, d, d, None, d, None, None, None, ws, None) == 4
    assert f(ctypes.byref(p), odd, d, d, d, d, None, d, None, None, d, ws, None) == 3      # 16-byte rule
    assert f(ctypes.byref(p), d, d, d, d, d, odd, d, None, None, d, ws, None) == 3
    # no tokens and no final state asked for: nothing to do
    p0 = m.ComplexProblem(2, 0, 4, 64, 64, 64)
    assert f(ctypes.byref(p0), None, None, d, None, None, None, None, None, None, d, ws, None) == 0
