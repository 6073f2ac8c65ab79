"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the float64 oracle on the same rounded inputs, compare."""
import numpy as np
import torch

from state_space_model_scan_gb300 import inputs as inp_mod
from state_space_model_scan_gb300.api import ssd_forward, ssd_backward

TOL = {"f32": 1e-4, "bf16": 1e-2}


def rel_l2(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def to_dev(inp, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def gpu_forward(w, inp, algo="auto", seg_chunks=0, **kw):
    d = to_dev(inp)
    y, fin = ssd_forward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                         initial_states=d["initial_states"], cu_seqlens=d["cu_seqlens"], chunk_size=w.chunk_size,
                         algo=algo, seg_chunks=seg_chunks, **kw)
    torch.cuda.synchronize()
    return y, fin


def gpu_backward(w, inp, algo="auto", **kw):
    d = to_dev(inp)
    g = ssd_backward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], d["dy"], D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                     initial_states=d["initial_states"], dfinal_states=d.get("dfinal_states"),
                     cu_seqlens=d["cu_seqlens"], chunk_size=w.chunk_size, algo=algo, **kw)
    torch.cuda.synchronize()
    return g


def flat(t, T):
    """[B, L, ...] -> [B*L, ...] float64 numpy."""
    a = t.detach().to(torch.float64).cpu().numpy()
    return a.reshape((T,) + a.shape[2:])


def oracle_forward(w, inp, heads=None):
    from oracle import sequential
    o = inp_mod.to_oracle(inp, w)
    return sequential.forward(o["x"], o["dt_raw"], o["A"], o["B"], o["C"], D=o["D"], z=o["z"], dt_bias=o["dt_bias"],
                              init=o["init"], cu=o["cu"], heads=heads)


def oracle_backward(w, inp, heads=None):
    from oracle import sequential
    o = inp_mod.to_oracle(inp, w)
    return sequential.backward(o["x"], o["dt_raw"], o["A"], o["B"], o["C"], o["dy"], D=o["D"], z=o["z"],
                               dt_bias=o["dt_bias"], init=o["init"], dfinal=o.get("dfinal"), cu=o["cu"],
                               heads=heads)
