"""ctypes binding of libssd.so (include/ssd.h).

Argument marshalling only: every step of the scan runs in the library's CUDA
kernels.  Torch is used to own device memory and to supply the current stream;
nothing here computes any part of the scan.  If libssd.so is missing the calls
raise -- there is no fallback.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssd.so")

SSD_OK = 0
STATUS_NAMES = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARGUMENT", 2: "SSD_ERR_UNSUPPORTED", 3: "SSD_ERR_MISALIGNED",
                4: "SSD_ERR_WORKSPACE_TOO_SMALL", 5: "SSD_ERR_CUDA", 6: "SSD_ERR_DEVICE_TIMEOUT"}
SSD_F32, SSD_BF16 = 0, 1
ALGO = {"auto": 0, "staged": 1, "fused": 2, "split": 3}

# Every symbol include/ssd.h declares.
EXPORTS = ["ssd_fwd_workspace_size", "ssd_fwd", "ssd_bwd_workspace_size", "ssd_bwd", "ssd_query_status",
           "ssd_status_string", "ssd_abi_version", "ssd_fwd_debug_layout", "ssd_fwd_noalloc",
           "ssd_selftest_bounded_wait", "ssd_chunk_states_size", "ssd_noalloc_query_status", "ssd_varlen_metadata",
           "ssd_gated_norm_fwd", "ssd_gated_norm_bwd_workspace_size", "ssd_gated_norm_bwd",
           "ssd_conv1d_fwd", "ssd_conv1d_bwd_workspace_size", "ssd_conv1d_bwd",
           "ssd_complex_fwd_workspace_size", "ssd_complex_fwd"]
NOALLOC_SCRATCH_BYTES = 64 << 20


class SSDError(RuntimeError):
    def __init__(self, code, where):
        self.code = int(code)
        super().__init__("%s: %s" % (where, STATUS_NAMES.get(int(code), str(code))))


class Tensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("stride", ctypes.c_int64 * 4)]


class Problem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("ngroups", ctypes.c_int64), ("dstate", ctypes.c_int64),
                ("chunk_size", ctypes.c_int64), ("nseqs", ctypes.c_int64), ("algo", ctypes.c_int32),
                ("seg_chunks", ctypes.c_int32), ("bwd_heads", ctypes.c_int32), ("reserved0", ctypes.c_int32)]


_FWD_FIELDS = ["x", "dt", "A", "B", "C", "D", "z", "dt_bias", "initial_states", "y", "final_states"]


class FwdArgs(ctypes.Structure):
    _fields_ = [(n, Tensor) for n in _FWD_FIELDS] + [("cu_seqlens", ctypes.c_void_p), ("chunk_states", ctypes.c_void_p)]


_BWD_FIELDS = ["dy", "dfinal_states", "dx", "ddt", "dA", "dB", "dC", "dD", "dz", "ddt_bias", "dinitial_states"]


class BwdArgs(ctypes.Structure):
    _fields_ = [("fwd", FwdArgs)] + [(n, Tensor) for n in _BWD_FIELDS]


class NormProblem(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("width", ctypes.c_int64), ("group_size", ctypes.c_int64),
                ("eps", ctypes.c_float), ("dtype", ctypes.c_int32), ("flags", ctypes.c_int32)]


class ConvProblem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("channels", ctypes.c_int64),
                ("width", ctypes.c_int64), ("nseqs", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("activation", ctypes.c_int32), ("reserved", ctypes.c_int32), ("pad", ctypes.c_int32)]


class ComplexProblem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("dstate", ctypes.c_int64), ("chunk_size", ctypes.c_int64)]


class DebugLayout(ctypes.Structure):
    _fields_ = [("meta_counts", ctypes.c_int64), ("chunk_info", ctypes.c_int64), ("dt", ctypes.c_int64),
                ("cs", ctypes.c_int64), ("states", ctypes.c_int64), ("units", ctypes.c_int64),
                ("qi", ctypes.c_int64)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libssd.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libssd.so not found at %s: build it with state_space_model_scan_gb300.build.build()" % path)
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    lib.ssd_fwd_workspace_size.argtypes = [P(Problem), P(FwdArgs), P(ctypes.c_size_t)]
    lib.ssd_fwd.argtypes = [P(Problem), P(FwdArgs), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.ssd_bwd_workspace_size.argtypes = [P(Problem), P(BwdArgs), P(ctypes.c_size_t)]
    lib.ssd_bwd.argtypes = [P(Problem), P(BwdArgs), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.ssd_query_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.ssd_status_string.argtypes = [ctypes.c_int]
    lib.ssd_status_string.restype = ctypes.c_char_p
    lib.ssd_abi_version.restype = ctypes.c_int32
    lib.ssd_fwd_debug_layout.argtypes = [P(Problem), P(FwdArgs), P(DebugLayout)]
    lib.ssd_fwd_noalloc.argtypes = [P(Problem), P(FwdArgs), ctypes.c_void_p]
    lib.ssd_selftest_bounded_wait.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_void_p]
    lib.ssd_chunk_states_size.argtypes = [P(Problem), P(FwdArgs), P(ctypes.c_size_t)]
    lib.ssd_noalloc_query_status.argtypes = [ctypes.c_void_p]
    lib.ssd_varlen_metadata.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p]
    V, I64 = ctypes.c_void_p, ctypes.c_int64
    lib.ssd_gated_norm_fwd.argtypes = [P(NormProblem), V, I64, V, I64, V, V, I64, V, V]
    lib.ssd_gated_norm_bwd_workspace_size.argtypes = [P(NormProblem), P(ctypes.c_size_t)]
    lib.ssd_gated_norm_bwd.argtypes = [P(NormProblem), V, I64, V, I64, V, V, V, I64, V, I64, V, I64, V, V,
                                       ctypes.c_size_t, V]
    lib.ssd_conv1d_fwd.argtypes = [P(ConvProblem), V, I64, I64, V, V, V, V, I64, I64, V]
    lib.ssd_conv1d_bwd_workspace_size.argtypes = [P(ConvProblem), P(ctypes.c_size_t)]
    lib.ssd_conv1d_bwd.argtypes = [P(ConvProblem), V, I64, I64, V, V, V, V, I64, I64, V, I64, I64, V, V, V,
                                   ctypes.c_size_t, V]
    lib.ssd_complex_fwd_workspace_size.argtypes = [P(ComplexProblem), P(ctypes.c_size_t)]
    lib.ssd_complex_fwd.argtypes = [P(ComplexProblem), V, V, V, V, V, V, V, V, V, V, ctypes.c_size_t, V]
    for f in ("ssd_fwd_workspace_size", "ssd_fwd", "ssd_bwd_workspace_size", "ssd_bwd", "ssd_query_status",
              "ssd_fwd_debug_layout", "ssd_fwd_noalloc", "ssd_selftest_bounded_wait", "ssd_chunk_states_size",
              "ssd_noalloc_query_status", "ssd_varlen_metadata", "ssd_gated_norm_fwd",
              "ssd_gated_norm_bwd_workspace_size", "ssd_gated_norm_bwd", "ssd_conv1d_fwd",
              "ssd_conv1d_bwd_workspace_size", "ssd_conv1d_bwd", "ssd_complex_fwd_workspace_size",
              "ssd_complex_fwd"):
        getattr(lib, f).restype = ctypes.c_int
    _lib = lib
    return lib


def tensor(t, rank=None):
    """An ssd_tensor for a torch tensor (or an absent one for None)."""
    out = Tensor()
    if t is None:
        return out
    if t.dtype == torch.bfloat16:
        out.dtype = SSD_BF16
    elif t.dtype == torch.float32:
        out.dtype = SSD_F32
    else:
        out.dtype = -1
    out.ptr = t.data_ptr()
    st = list(t.stride())
    for i, s in enumerate(st[:4]):
        out.stride[i] = s
    return out


def problem(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size, nseqs=0, algo="auto", seg_chunks=0,
            bwd_heads=0):
    return Problem(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size, nseqs, ALGO[algo], seg_chunks,
                   bwd_heads, 0)


def fwd_args(x, dt, A, B, C, y, D=None, z=None, dt_bias=None, initial_states=None, final_states=None,
             cu_seqlens=None, chunk_states=None):
    """chunk_states: a device buffer (any dtype) of chunk_states_size bytes, or None."""
    a = FwdArgs()
    for name, t in dict(x=x, dt=dt, A=A, B=B, C=C, D=D, z=z, dt_bias=dt_bias, initial_states=initial_states,
                        y=y, final_states=final_states).items():
        setattr(a, name, tensor(t))
    a.cu_seqlens = None if cu_seqlens is None else cu_seqlens.data_ptr()
    a.chunk_states = None if chunk_states is None else chunk_states.data_ptr()
    return a


def bwd_args(fwd, dy, dx, ddt, dA, dB, dC, dD=None, dz=None, ddt_bias=None, dinitial_states=None,
             dfinal_states=None):
    b = BwdArgs()
    b.fwd = fwd
    for name, t in dict(dy=dy, dfinal_states=dfinal_states, dx=dx, ddt=ddt, dA=dA, dB=dB, dC=dC, dD=dD, dz=dz,
                        ddt_bias=ddt_bias, dinitial_states=dinitial_states).items():
        setattr(b, name, tensor(t))
    return b


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def check(code, where):
    if code != SSD_OK:
        raise SSDError(code, where)


def fwd_workspace_size(prob, args):
    n = ctypes.c_size_t(0)
    check(load().ssd_fwd_workspace_size(ctypes.byref(prob), ctypes.byref(args), ctypes.byref(n)),
          "ssd_fwd_workspace_size")
    return int(n.value)


def chunk_states_size(prob, args):
    """Bytes of the chunk-state buffer the forward can keep for the backward (tensor-core path)."""
    n = ctypes.c_size_t(0)
    check(load().ssd_chunk_states_size(ctypes.byref(prob), ctypes.byref(args), ctypes.byref(n)),
          "ssd_chunk_states_size")
    return int(n.value)


def bwd_workspace_size(prob, args):
    n = ctypes.c_size_t(0)
    check(load().ssd_bwd_workspace_size(ctypes.byref(prob), ctypes.byref(args), ctypes.byref(n)),
          "ssd_bwd_workspace_size")
    return int(n.value)


def ssd_fwd(prob, args, workspace, stream=None):
    """Raw call: returns the status code (no raise)."""
    return load().ssd_fwd(ctypes.byref(prob), ctypes.byref(args), ctypes.c_void_p(workspace.data_ptr()),
                          ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream_handle(stream))


def ssd_bwd(prob, args, workspace, stream=None):
    return load().ssd_bwd(ctypes.byref(prob), ctypes.byref(args), ctypes.c_void_p(workspace.data_ptr()),
                          ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream_handle(stream))


def ssd_fwd_noalloc(prob, args, stream=None):
    """Raw call of the forward that uses the library's static scratch (no workspace)."""
    return load().ssd_fwd_noalloc(ctypes.byref(prob), ctypes.byref(args), _stream_handle(stream))


def noalloc_query_status(stream=None):
    """Status word the last ssd_fwd_noalloc call left on the current device (synchronises)."""
    return int(load().ssd_noalloc_query_status(_stream_handle(stream)))


def varlen_metadata(cu_seqlens, seqlen, chunk_size, stream=None, with_seq_idx=True):
    """Packed-sequence metadata on the chunk grid (ssd_varlen_metadata): returns the raw
    status code and, on SSD_OK, device tensors seq_idx [seqlen] (or None), chunk_begin
    [n_chunks + 1], segments [n_chunks + nseqs, 3] (the first chunk_begin[-1] rows are
    valid) and the device status word [1]."""
    dev = cu_seqlens.device
    S = cu_seqlens.numel() - 1
    nch = -(-int(seqlen) // int(chunk_size))
    seq_idx = torch.full((max(int(seqlen), 1),), -1, dtype=torch.int32, device=dev) if with_seq_idx else None
    begin = torch.full((nch + 1,), -1, dtype=torch.int32, device=dev)
    segs = torch.full((nch + S, 3), -1, dtype=torch.int32, device=dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    code = int(load().ssd_varlen_metadata(ctypes.c_void_p(cu_seqlens.data_ptr()), S, int(seqlen), int(chunk_size),
                                          None if seq_idx is None else ctypes.c_void_p(seq_idx.data_ptr()),
                                          ctypes.c_void_p(begin.data_ptr()), ctypes.c_void_p(segs.data_ptr()),
                                          ctypes.c_void_p(status.data_ptr()), _stream_handle(stream)))
    return code, seq_idx, begin, segs, status


def selftest_bounded_wait(workspace, wait_ms, stream=None):
    """Enqueue the bounded-wait self-test (see include/ssd.h); read the result with query_status."""
    return int(load().ssd_selftest_bounded_wait(ctypes.c_void_p(workspace.data_ptr()),
                                                ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                                                ctypes.c_int32(wait_ms), _stream_handle(stream)))


def query_status(workspace, stream=None):
    return int(load().ssd_query_status(ctypes.c_void_p(workspace.data_ptr()), _stream_handle(stream)))


def debug_layout(prob, args):
    out = DebugLayout()
    check(load().ssd_fwd_debug_layout(ctypes.byref(prob), ctypes.byref(args), ctypes.byref(out)),
          "ssd_fwd_debug_layout")
    return out


def status_string(code):
    return load().ssd_status_string(int(code)).decode()


def abi_version():
    return int(load().ssd_abi_version())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _rowstride(t):
    return 0 if t is None else int(t.stride(-2)) if t.dim() >= 2 else int(t.shape[-1])


SSD_NORM_LAYER, SSD_NORM_GATE_AFTER = 1, 2


def norm_problem(rows, width, group_size, eps, dtype, layer_norm=False, gate_after=False):
    flags = (SSD_NORM_LAYER if layer_norm else 0) | (SSD_NORM_GATE_AFTER if gate_after else 0)
    return NormProblem(rows, width, group_size, eps, SSD_BF16 if dtype == torch.bfloat16 else SSD_F32, flags)


def gated_norm_fwd(prob, y, z, weight, out, rstd, stream=None):
    """Raw call on 2-D [rows, width] views (row stride = stride(0)); returns the status code."""
    return int(load().ssd_gated_norm_fwd(ctypes.byref(prob), _ptr(y), _rowstride(y), _ptr(z), _rowstride(z),
                                         _ptr(weight), _ptr(out), _rowstride(out), _ptr(rstd),
                                         _stream_handle(stream)))


def gated_norm_bwd_workspace_size(prob):
    n = ctypes.c_size_t(0)
    check(load().ssd_gated_norm_bwd_workspace_size(ctypes.byref(prob), ctypes.byref(n)),
          "ssd_gated_norm_bwd_workspace_size")
    return int(n.value)


def gated_norm_bwd(prob, y, z, weight, rstd, dout, dy, dz, dweight, workspace, stream=None):
    return int(load().ssd_gated_norm_bwd(ctypes.byref(prob), _ptr(y), _rowstride(y), _ptr(z), _rowstride(z),
                                         _ptr(weight), _ptr(rstd), _ptr(dout), _rowstride(dout), _ptr(dy),
                                         _rowstride(dy), _ptr(dz), _rowstride(dz), _ptr(dweight),
                                         _ptr(workspace),
                                         ctypes.c_size_t(0 if workspace is None else workspace.numel() *
                                                         workspace.element_size()),
                                         _stream_handle(stream)))


def conv_problem(batch, seqlen, channels, width, nseqs, dtype, silu):
    return ConvProblem(batch, seqlen, channels, width, nseqs, SSD_BF16 if dtype == torch.bfloat16 else SSD_F32,
                       1 if silu else 0, 0, 0)


def _bl(t):
    """(batch stride, token stride) of a [batch, seqlen, channels] tensor."""
    return (0, 0) if t is None else (int(t.stride(0)), int(t.stride(1)))


def conv1d_fwd(prob, u, weight, bias, cu_seqlens, out, stream=None):
    """Raw call on [batch, seqlen, channels] tensors; returns the status code."""
    return int(load().ssd_conv1d_fwd(ctypes.byref(prob), _ptr(u), *_bl(u), _ptr(weight), _ptr(bias),
                                     _ptr(cu_seqlens), _ptr(out), *_bl(out), _stream_handle(stream)))


def conv1d_bwd_workspace_size(prob):
    n = ctypes.c_size_t(0)
    check(load().ssd_conv1d_bwd_workspace_size(ctypes.byref(prob), ctypes.byref(n)), "ssd_conv1d_bwd_workspace_size")
    return int(n.value)


def conv1d_bwd(prob, u, weight, bias, cu_seqlens, dout, du, dweight, dbias, workspace, stream=None):
    return int(load().ssd_conv1d_bwd(ctypes.byref(prob), _ptr(u), *_bl(u), _ptr(weight), _ptr(bias),
                                     _ptr(cu_seqlens), _ptr(dout), *_bl(dout), _ptr(du), *_bl(du), _ptr(dweight),
                                     _ptr(dbias), _ptr(workspace),
                                     ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                                     _stream_handle(stream)))


def complex_fwd_workspace_size(prob):
    n = ctypes.c_size_t(0)
    check(load().ssd_complex_fwd_workspace_size(ctypes.byref(prob), ctypes.byref(n)), "ssd_complex_fwd_workspace_size")
    return int(n.value)


def complex_fwd(prob, x, dt, A, B, C, init, y_re, y_im, final, workspace, stream=None):
    """Raw call (complex tensors are complex64, contiguous); returns the status code."""
    return int(load().ssd_complex_fwd(ctypes.byref(prob), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(init),
                                      _ptr(y_re), _ptr(y_im), _ptr(final), _ptr(workspace),
                                      ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                                      _stream_handle(stream)))
