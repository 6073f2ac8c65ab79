"""Torch-facing wrappers around the C ABI.

They allocate outputs and workspace with torch, marshal pointers/strides/stream
into the ABI structs and raise on a non-OK status.  All arithmetic runs in
libssd.so.
"""
import torch

from . import _lib


class Workspace:
    """A reusable device workspace: grows to the largest size requested."""

    def __init__(self, device=None):
        self.device = device
        self.buf = None

    def get(self, nbytes):
        nbytes = max(int(nbytes), 256)
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device or "cuda")
        return self.buf


def _nseqs(x, cu_seqlens):
    return (cu_seqlens.numel() - 1) if cu_seqlens is not None else x.shape[0]


def ssd_forward(x, dt, A, B, C, D=None, z=None, dt_bias=None, initial_states=None, cu_seqlens=None,
                chunk_size=128, return_final_states=True, algo="auto", seg_chunks=0, workspace=None,
                y=None, final_states=None, stream=None, keep_chunk_states=False, chunk_states=None,
                state_dtype=None):
    """y, final_states = SSD scan (see include/ssd.h for the definition and layouts).

    x, z: [B, L, H, P]; dt: [B, L, H] fp32; A, D, dt_bias: [H] fp32; B, C: [B, L, G, N];
    initial_states: [S, H, P, N] fp32 or bf16; cu_seqlens: int32 [S+1] (batch 1).
    state_dtype: storage dtype of the returned final states (default: that of initial_states,
    else fp32); the scan itself carries its state in fp32 either way.
    keep_chunk_states: also return the carried chunk states (a uint8 device buffer, tensor-core
    path only; raises SSDError(SSD_ERR_UNSUPPORTED) otherwise) for ssd_backward(chunk_states=...),
    which then skips their recompute.  chunk_states: a caller-owned buffer to fill instead.
    """
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    S = _nseqs(x, cu_seqlens)
    if y is None:
        y = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    if final_states is None and return_final_states:
        sdt = state_dtype or (initial_states.dtype if initial_states is not None else torch.float32)
        final_states = torch.empty(S, H, P, N, dtype=sdt, device=x.device)
    prob = _lib.problem(Bsz, L, H, P, G, N, chunk_size, S if cu_seqlens is not None else 0, algo, seg_chunks)
    args = _lib.fwd_args(x, dt, A, B, C, y, D=D, z=z, dt_bias=dt_bias, initial_states=initial_states,
                         final_states=final_states, cu_seqlens=cu_seqlens)
    if keep_chunk_states or chunk_states is not None:
        need = _lib.chunk_states_size(prob, args)
        if chunk_states is None:
            chunk_states = torch.empty(need, dtype=torch.uint8, device=x.device)
        if chunk_states.numel() * chunk_states.element_size() < need:
            raise ValueError("chunk_states holds %d bytes, %d needed" % (chunk_states.numel() * chunk_states.element_size(), need))
        args.chunk_states = chunk_states.data_ptr()
    nbytes = _lib.fwd_workspace_size(prob, args)
    ws = workspace.get(nbytes) if workspace is not None else torch.empty(max(nbytes, 256), dtype=torch.uint8,
                                                                          device=x.device)
    _lib.check(_lib.ssd_fwd(prob, args, ws, stream), "ssd_fwd")
    if keep_chunk_states:
        return y, final_states, chunk_states
    return y, final_states


def ssd_backward(x, dt, A, B, C, dy, D=None, z=None, dt_bias=None, initial_states=None, dfinal_states=None,
                 cu_seqlens=None, chunk_size=128, algo="auto", seg_chunks=0, bwd_heads=0, workspace=None,
                 stream=None, chunk_states=None):
    """Gradients of sum(dy*y) + sum(dfinal_states*final_states).  Returns a dict with
    dx, ddt, dA, dB, dC and, when the matching input is given, dD, dz, ddt_bias, dinitial_states.
    bwd_heads: heads per CTA of the tensor-core gradient kernel (0 = library choice).
    chunk_states: the buffer ssd_forward(keep_chunk_states=True) returned for the same inputs."""
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    S = _nseqs(x, cu_seqlens)
    dev = x.device
    g = dict(dx=torch.empty(x.shape, dtype=x.dtype, device=dev),
             ddt=torch.empty(dt.shape, dtype=torch.float32, device=dev),
             dA=torch.empty(H, dtype=torch.float32, device=dev),
             dB=torch.empty(B.shape, dtype=B.dtype, device=dev),
             dC=torch.empty(C.shape, dtype=C.dtype, device=dev))
    if D is not None:
        g["dD"] = torch.empty(H, dtype=torch.float32, device=dev)
    if z is not None:
        g["dz"] = torch.empty(z.shape, dtype=z.dtype, device=dev)
    if dt_bias is not None:
        g["ddt_bias"] = torch.empty(H, dtype=torch.float32, device=dev)
    if initial_states is not None:   # in the initial states' storage dtype
        g["dinitial_states"] = torch.empty(S, H, P, N, dtype=initial_states.dtype, device=dev)
    prob = _lib.problem(Bsz, L, H, P, G, N, chunk_size, S if cu_seqlens is not None else 0, algo, seg_chunks,
                        bwd_heads)
    fa = _lib.fwd_args(x, dt, A, B, C, None, D=D, z=z, dt_bias=dt_bias, initial_states=initial_states,
                       cu_seqlens=cu_seqlens, chunk_states=chunk_states)
    ba = _lib.bwd_args(fa, dy, g["dx"], g["ddt"], g["dA"], g["dB"], g["dC"], dD=g.get("dD"), dz=g.get("dz"),
                       ddt_bias=g.get("ddt_bias"), dinitial_states=g.get("dinitial_states"),
                       dfinal_states=dfinal_states)
    nbytes = _lib.bwd_workspace_size(prob, ba)
    ws = workspace.get(nbytes) if workspace is not None else torch.empty(max(nbytes, 256), dtype=torch.uint8,
                                                                          device=dev)
    _lib.check(_lib.ssd_bwd(prob, ba, ws, stream), "ssd_bwd")
    return g


def _rows(t, width):
    """[..., width] (features contiguous, rows at a common stride) as a 2-D [rows, width] view."""
    return t.reshape(-1, width)


def gated_norm_forward(y, weight, group_size, z=None, eps=1e-5, layer_norm=False, gate_after=False, stream=None):
    """out, rstd = the gated normalisation of y over groups of `group_size` features (see
    include/ssd.h, ssd_gated_norm_fwd): RMS (default) or LayerNorm (layer_norm=True, no bias)
    of u = y silu(z), times weight; with gate_after=True, of u = y, times weight and silu(z).
    y, z: [..., width]."""
    width = y.shape[-1]
    y2 = _rows(y, width)
    z2 = _rows(z, width) if z is not None else None
    out = torch.empty_like(y2)
    rstd = torch.empty(y2.shape[0], width // group_size, dtype=torch.float32, device=y.device)
    prob = _lib.norm_problem(y2.shape[0], width, group_size, eps, y.dtype, layer_norm, gate_after)
    _lib.check(_lib.gated_norm_fwd(prob, y2, z2, weight, out, rstd, stream), "ssd_gated_norm_fwd")
    return out.reshape(y.shape), rstd


def gated_norm_backward(y, weight, rstd, dout, group_size, z=None, eps=1e-5, layer_norm=False, gate_after=False,
                        stream=None):
    """dy, dz (None without z), dweight: gradients of sum(dout * out) (same options as the forward)."""
    width = y.shape[-1]
    y2, d2 = _rows(y, width), _rows(dout, width)
    z2 = _rows(z, width) if z is not None else None
    dy = torch.empty_like(y2)
    dz = torch.empty_like(z2) if z is not None else None
    dw = torch.empty(width, dtype=torch.float32, device=y.device)
    prob = _lib.norm_problem(y2.shape[0], width, group_size, eps, y.dtype, layer_norm, gate_after)
    ws = torch.empty(max(_lib.gated_norm_bwd_workspace_size(prob), 16), dtype=torch.uint8, device=y.device)
    _lib.check(_lib.gated_norm_bwd(prob, y2, z2, weight, rstd, d2, dy, dz, dw, ws, stream), "ssd_gated_norm_bwd")
    return dy.reshape(y.shape), (dz.reshape(z.shape) if dz is not None else None), dw


def conv1d_forward(xbc, weight, bias=None, cu_seqlens=None, silu=True, stream=None):
    """Causal depthwise conv1d (+ SiLU) over the sequence axis of xbc [batch, seqlen, channels]
    (see include/ssd.h, ssd_conv1d_fwd); packed sequences (cu_seqlens, batch 1) never mix."""
    Bsz, L, Cn = xbc.shape
    out = torch.empty(Bsz, L, Cn, dtype=xbc.dtype, device=xbc.device)
    prob = _lib.conv_problem(Bsz, L, Cn, weight.shape[1], 0 if cu_seqlens is None else cu_seqlens.numel() - 1,
                             xbc.dtype, silu)
    _lib.check(_lib.conv1d_fwd(prob, xbc, weight, bias, cu_seqlens, out, stream), "ssd_conv1d_fwd")
    return out


def conv1d_backward(xbc, weight, dout, bias=None, cu_seqlens=None, silu=True, stream=None):
    """dxbc, dweight, dbias (None without bias): gradients of sum(dout * conv1d_forward(...))."""
    Bsz, L, Cn = xbc.shape
    du = torch.empty(Bsz, L, Cn, dtype=xbc.dtype, device=xbc.device)
    dw = torch.empty_like(weight)
    db = torch.empty_like(bias) if bias is not None else None
    prob = _lib.conv_problem(Bsz, L, Cn, weight.shape[1], 0 if cu_seqlens is None else cu_seqlens.numel() - 1,
                             xbc.dtype, silu)
    ws = torch.empty(max(_lib.conv1d_bwd_workspace_size(prob), 16), dtype=torch.uint8, device=xbc.device)
    _lib.check(_lib.conv1d_bwd(prob, xbc, weight, bias, cu_seqlens, dout, du, dw, db, ws, stream), "ssd_conv1d_bwd")
    return du, dw, db


def split_xbc(xbc, nheads, headdim, ngroups, dstate):
    """x [B, L, H, P], B and C [B, L, G, N] as views of the packed xbc [B, L, H P + 2 G N] (no copy);
    the scan takes them as they are (strided tensors)."""
    Bsz, L, Cn = xbc.shape
    hp, gn = nheads * headdim, ngroups * dstate
    assert Cn == hp + 2 * gn
    x = xbc[..., :hp].unflatten(-1, (nheads, headdim))
    Bm = xbc[..., hp:hp + gn].unflatten(-1, (ngroups, dstate))
    Cm = xbc[..., hp + gn:].unflatten(-1, (ngroups, dstate))
    return x, Bm, Cm


class SSDFunction(torch.autograd.Function):
    """Autograd wrapper: forward and backward both run in libssd.so.  On the tensor-core
    path the forward keeps its carried chunk states for the backward."""

    @staticmethod
    def forward(ctx, x, dt, A, B, C, D, z, dt_bias, initial_states, cu_seqlens, chunk_size):
        kw = dict(D=D, z=z, dt_bias=dt_bias, initial_states=initial_states, cu_seqlens=cu_seqlens,
                  chunk_size=chunk_size)
        try:
            y, fin, cs = ssd_forward(x, dt, A, B, C, keep_chunk_states=True, **kw)
        except _lib.SSDError as e:   # the SIMT path recomputes its states
            if e.code != 2:
                raise
            y, fin = ssd_forward(x, dt, A, B, C, **kw)
            cs = None
        ctx.save_for_backward(x, dt, A, B, C, D, z, dt_bias, initial_states, cu_seqlens)
        ctx.chunk_states = cs
        ctx.chunk_size = chunk_size
        return y, fin

    @staticmethod
    def backward(ctx, dy, dfin):
        x, dt, A, B, C, D, z, dt_bias, init, cu = ctx.saved_tensors
        g = ssd_backward(x, dt, A, B, C, dy.contiguous(), D=D, z=z, dt_bias=dt_bias, initial_states=init,
                         dfinal_states=None if dfin is None else dfin.contiguous(), cu_seqlens=cu,
                         chunk_size=ctx.chunk_size, chunk_states=ctx.chunk_states)
        return (g["dx"], g["ddt"], g["dA"], g["dB"], g["dC"], g.get("dD"), g.get("dz"), g.get("ddt_bias"),
                g.get("dinitial_states"), None, None)


def complex_ssd_forward(x, A, B, C, dt, initial_states=None, chunk_size=64, return_imag=False,
                        return_final=False, stream=None):
    """Complex-A SSD scan (Mamba-3-Lite): h_t = exp(softplus(dt_t) A) h_{t-1} + x_t (outer) B_t,
    y_t = sum_n C_t[n] h_t[:, n].  x [batch, seqlen, nheads, headdim], B/C [batch, seqlen, nheads,
    dstate] and A [nheads] complex64; dt [batch, seqlen, nheads] float32; initial_states
    [batch, nheads, headdim, dstate] complex64.  Returns Re y (float32), then Im y and the final
    state when asked for."""
    Bt, T, H, Dh = x.shape
    N = B.shape[-1]
    dev = x.device
    for t in (x, B, C, A) + ((initial_states,) if initial_states is not None else ()):
        if t.dtype != torch.complex64 or not t.is_contiguous():
            raise ValueError("complex tensors must be contiguous complex64")
    if dt.dtype != torch.float32 or not dt.is_contiguous():
        raise ValueError("dt must be contiguous float32")
    prob = _lib.ComplexProblem(Bt, T, H, Dh, N, chunk_size)
    y_re = torch.empty(Bt, T, H, Dh, dtype=torch.float32, device=dev)
    y_im = torch.empty_like(y_re) if return_imag else None
    final = torch.empty(Bt, H, Dh, N, dtype=torch.complex64, device=dev) if return_final else None
    ws = torch.empty(_lib.complex_fwd_workspace_size(prob), dtype=torch.uint8, device=dev)
    _lib.check(_lib.complex_fwd(prob, x, dt, A, B, C, initial_states, y_re, y_im, final, ws, stream),
               "ssd_complex_fwd")
    out = (y_re,)
    if return_imag:
        out += (y_im,)
    if return_final:
        out += (final,)
    return out[0] if len(out) == 1 else out
