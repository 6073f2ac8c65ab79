"""Seeded synthetic inputs for the SSD scan.

This module only draws random numbers and casts them; it holds none of the scan's
arithmetic, so both the CUDA path's tests and the float64 oracle consume the
same rounded values from it.

Value distributions (the shapes and distributions of the Nemotron-Nano-shaped
and long-sequence workloads the source pages benchmark):

* A        = -exp(U[ln 1, ln 16])                          -> A in [-16, -1]
* dt_bias  = softplus^-1(u), u = exp(U[ln 1e-3, ln 1e-1])  -> softplus(dt_bias) in [1e-3, 1e-1]
* D ~ N(0, 1);  dt_raw ~ 0.5 N(0, 1);  x, B, C, z ~ N(0, 1)
* initial_states ~ 0.1 N(0, 1);  dy ~ N(0, 1);  dfinal ~ 0.1 N(0, 1)

The second parameter of N(., .) is the standard deviation.  Every tensor has its
own generator seeded from (seed, tensor index), so switching one feature off does
not change the other tensors.  Values are drawn in float64 on the CPU and rounded
once (round-to-nearest-even) to the storage dtype.
"""
from dataclasses import dataclass, field, replace
import math
from typing import List, Optional

import torch

_ORDER = ["A", "dt_bias", "D", "dt_raw", "x", "B", "C", "z", "initial_states", "dy", "dfinal_states", "seqlens"]


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    ngroups: int
    dstate: int
    chunk_size: int
    dtype: str = "bf16"          # storage dtype of x, z, B, C, y and their gradients
    has_z: bool = True
    has_D: bool = True
    has_dt_bias: bool = True
    has_init: bool = False
    seqlens: Optional[List[int]] = field(default=None, hash=False)  # packed varlen (batch == 1)
    seed: int = 0

    @property
    def nseqs(self) -> int:
        return len(self.seqlens) if self.seqlens is not None else self.batch

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen


def varlen_lengths(nseq: int, lo: int, hi: int, seed: int) -> List[int]:
    """`nseq` lengths drawn i.i.d. uniform on the integers [lo, hi]."""
    g = torch.Generator().manual_seed(seed * 1000 + _ORDER.index("seqlens"))
    return [int(v) for v in torch.randint(lo, hi + 1, (nseq,), generator=g)]


def named(name: str, L: Optional[int] = None) -> Workload:
    """The workloads used by the tests and the benchmark, by name."""
    if name == "tiny_f32":       # batch 1, L=256, 4 heads x 16, 1 group, N=16, chunk 64, fp32, no z
        return Workload(name, 1, 256, 4, 16, 1, 16, 64, "f32", has_z=False, has_D=True)
    if name == "nemotron_nano":  # batch 1, L=8192, 64 heads x 64, 8 groups, N=128, chunk 128, bf16, z + D
        return Workload(name, 1, 8192, 64, 64, 8, 128, 128, "bf16", has_z=True, has_D=True)
    if name == "long_seq":       # batch 1, 128 heads x 64, 1 group, N=128, chunk 128, init, no z
        return Workload(name + "_L%d" % (L or 8192), 1, L or 8192, 128, 64, 1, 128, 128, "bf16",
                        has_z=False, has_D=True, has_init=True)
    if name == "varlen":         # 16 packed sequences, lengths U{512..8192}, 80 heads x 64, 1 group
        # The continuous-batching workload is quoted with 256-token chunks; the tensor-core
        # tile set computes 128-token chunks (the scan's result does not depend on the chunk
        # length), so it is timed at 128, on a chunk grid over the packed axis; the SIMT path
        # computes it at 256 as well (a parity case).
        lens = varlen_lengths(16, 512, 8192, 0)
        return Workload(name, 1, sum(lens), 80, 64, 1, 128, 128, "bf16", has_z=False, has_D=True,
                        has_init=True, seqlens=lens)
    raise KeyError(name)


def _gen(seed: int, key: str) -> torch.Generator:
    return torch.Generator().manual_seed(seed * 1000 + _ORDER.index(key))


def _cast(t64: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return t64.to(torch.bfloat16)
    if dtype == "f32":
        return t64.to(torch.float32)
    if dtype == "f64":
        return t64
    raise ValueError(dtype)


def make_inputs(w: Workload, with_grad_inputs: bool = False, with_dfinal: bool = False) -> dict:
    """CPU tensors for workload `w`.

    x, z: [B, L, H, P]; B, C: [B, L, G, N] in `w.dtype`; dt_raw [B, L, H] fp32;
    A, D, dt_bias [H] fp32; initial_states [S, H, P, N] fp32 (S = nseqs);
    cu_seqlens int32 [S+1] for packed workloads; dy like x; dfinal_states like
    the states.  Optional tensors are None when the feature is off.
    """
    Bsz, L, H, P, G, N = w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate
    d = torch.float64
    out = {}
    u = torch.rand(H, generator=_gen(w.seed, "A"), dtype=d)
    out["A"] = (-torch.exp(u * math.log(16.0))).to(torch.float32)
    u = torch.rand(H, generator=_gen(w.seed, "dt_bias"), dtype=d)
    dtv = torch.exp(math.log(1e-3) + u * (math.log(1e-1) - math.log(1e-3)))
    out["dt_bias"] = (dtv + torch.log(-torch.expm1(-dtv))).to(torch.float32) if w.has_dt_bias else None
    out["D"] = torch.randn(H, generator=_gen(w.seed, "D"), dtype=d).to(torch.float32) if w.has_D else None
    out["dt_raw"] = (0.5 * torch.randn(Bsz, L, H, generator=_gen(w.seed, "dt_raw"), dtype=d)).to(torch.float32)
    out["x"] = _cast(torch.randn(Bsz, L, H, P, generator=_gen(w.seed, "x"), dtype=d), w.dtype)
    out["B"] = _cast(torch.randn(Bsz, L, G, N, generator=_gen(w.seed, "B"), dtype=d), w.dtype)
    out["C"] = _cast(torch.randn(Bsz, L, G, N, generator=_gen(w.seed, "C"), dtype=d), w.dtype)
    out["z"] = _cast(torch.randn(Bsz, L, H, P, generator=_gen(w.seed, "z"), dtype=d), w.dtype) if w.has_z else None
    S = w.nseqs
    out["initial_states"] = ((0.1 * torch.randn(S, H, P, N, generator=_gen(w.seed, "initial_states"), dtype=d))
                             .to(torch.float32) if w.has_init else None)
    if w.seqlens is not None:
        assert Bsz == 1
        cu = [0]
        for n in w.seqlens:
            cu.append(cu[-1] + int(n))
        assert cu[-1] == L
        out["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32)
    else:
        out["cu_seqlens"] = None
    if with_grad_inputs:
        out["dy"] = _cast(torch.randn(Bsz, L, H, P, generator=_gen(w.seed, "dy"), dtype=d), w.dtype)
        out["dfinal_states"] = ((0.1 * torch.randn(S, H, P, N, generator=_gen(w.seed, "dfinal_states"), dtype=d))
                                .to(torch.float32) if with_dfinal else None)
    return out


def to_oracle(inp: dict, w: Workload) -> dict:
    """The same values as float64 NumPy arrays on a flat token axis, with the
    token offsets of each sequence (``cu``), for the oracle's calling convention."""
    import numpy as np

    def f(t, shape=None):
        if t is None:
            return None
        a = t.to(torch.float64).numpy()
        return a.reshape(shape) if shape is not None else a

    Bsz, L, H, P, G, N = w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate
    T = Bsz * L
    if inp.get("cu_seqlens") is not None:
        cu = inp["cu_seqlens"].to(torch.int64).numpy()
    else:
        cu = np.arange(Bsz + 1, dtype=np.int64) * L
    o = dict(x=f(inp["x"], (T, H, P)), dt_raw=f(inp["dt_raw"], (T, H)), A=f(inp["A"]),
             B=f(inp["B"], (T, G, N)), C=f(inp["C"], (T, G, N)), D=f(inp["D"]),
             z=f(inp["z"], (T, H, P)) if inp["z"] is not None else None,
             dt_bias=f(inp["dt_bias"]), init=f(inp["initial_states"]), cu=cu)
    if "dy" in inp:
        o["dy"] = f(inp["dy"], (T, H, P))
        o["dfinal"] = f(inp["dfinal_states"])
    return o


def complex_inputs(batch: int, seqlen: int, nheads: int, headdim: int = 64, dstate: int = 64, seed: int = 0,
                   with_init: bool = True) -> dict:
    """CPU tensors for the complex-A scan (the Mamba-3-Lite variant).

    * Re A = -exp(U[ln 0.1, ln 1]), Im A = U[-pi, pi]      (A [H] complex64)
    * dt ~ N(0, 1) before softplus                          (dt [B, L, H] float32)
    * x, B, C: complex normal, real and imaginary parts N(0, 1/2) each (unit variance)
    * initial_states: 0.1 x complex normal                   ([B, H, headdim, dstate])
    Each tensor draws from its own generator; values drawn in float64, rounded once.
    """
    d = torch.float64
    g = lambda k: torch.Generator().manual_seed(seed * 1000 + 500 + k)

    def cn(k, *shape):
        gen = g(k)
        re = torch.randn(*shape, generator=gen, dtype=d)
        im = torch.randn(*shape, generator=gen, dtype=d)
        return (torch.complex(re, im) / math.sqrt(2.0)).to(torch.complex64)

    u = torch.rand(nheads, generator=g(0), dtype=d)
    ph = torch.rand(nheads, generator=g(1), dtype=d)
    A = torch.complex(-torch.exp(math.log(0.1) + u * (0.0 - math.log(0.1))), (2 * ph - 1) * math.pi)
    out = dict(A=A.to(torch.complex64),
               dt=torch.randn(batch, seqlen, nheads, generator=g(2), dtype=d).to(torch.float32),
               x=cn(3, batch, seqlen, nheads, headdim),
               B=cn(4, batch, seqlen, nheads, dstate),
               C=cn(5, batch, seqlen, nheads, dstate))
    out["initial_states"] = (0.1 * cn(6, batch, nheads, headdim, dstate).to(torch.complex128)).to(
        torch.complex64) if with_init else None
    return out
