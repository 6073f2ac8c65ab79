"""Benchmark of the SSD scan hot path on GB300.

One step, each call replayed from a CUDA graph with the L2 flushed (256 MB write)
before it:
  * the Nemotron-Nano-shaped workload (batch 1, L=8192, 64 heads x 64, 8 groups,
    dstate 128, chunk 128, z gate and D skip, bf16 x/B/C/z, fp32 dt/A/D/states):
    inference forward (metadata + fused tensor-core forward), then a training step =
    forward that also keeps the carried chunk states + backward that reads them;
  * the other forward workloads, one forward each: the long-sequence sweep (128 heads
    x 64, 1 group, dstate 128, initial states, L = 1k .. 32k) and the packed varlen
    workload (16 sequences of U{512..8192} tokens, 80 heads x 64, own initial states);
  * the kernels around the scan, forward and backward at the Nemotron-Nano widths (8192
    tokens, bf16): the gated RMS normalisation of y over 8 groups of 512 features and the
    causal conv1d (width 4, SiLU) over the packed xBC (6144 channels); and the complex-A
    scan of the Mamba-3-Lite variant at its 434M configuration (8 x 2048 tokens, 16 heads,
    headdim = dstate = chunk = 64).
`value` is the inference forward's tokens/s at the Nemotron-Nano shape (median over
the steps of its CUDA-event time); `ms_per_step` is the training step's median device
time (forward + backward); `sweep` holds the other workloads' median forward times,
tokens/s and HBM roofline fractions, `extras` the same for the kernels around the
scan; `e2e` is forward tokens/s with every step's inputs copied from pinned host memory and its y copied back inside the timed region, two
independent steps in flight (copy-in, compute and copy-out streams).  Clocks and
throttle reasons are sampled through NVML every millisecond during the timed steps.
Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the float64 CPU oracle (the reference arm of this build)
on a bounded sample of the same workload on the host cores.  With N > 1 (under
torchrun) every rank runs an independent replica (the scan does not shard:
replicas only) and rank 0 reports the aggregate over ranks.
"""
import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ssd_fwd_tokens_per_s"
WORKLOAD = "nemotron_nano"
L2_FLUSH_BYTES = 256 << 20


def workload_desc(w):
    return ("Mamba-2 SSD fwd+bwd, batch %d, L=%d, %d heads x %d, %d groups, dstate %d, chunk %d, z gate + D skip, "
            "bf16 x/B/C/z, fp32 dt/A/D/states" % (w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate,
                                                  w.chunk_size))


def algorithmic_bytes(w, fwd=True, state_bytes=4):
    """Compulsory HBM bytes of one forward (or backward) of workload w (states stored in
    `state_bytes` per element)."""
    b_x = 2 if w.dtype == "bf16" else 4
    T = w.batch * w.seqlen
    per_tok_heads = w.nheads * w.headdim * b_x
    bc = 2 * w.ngroups * w.dstate * b_x
    st = w.nseqs * w.nheads * w.headdim * w.dstate * state_bytes
    if fwd:
        n = T * ((3 if w.has_z else 2) * per_tok_heads + bc + 4 * w.nheads) + st   # x, z, y, B, C, dt, final
        if w.has_init:
            n += st
        return n
    # backward: read x, z, B, C, dt, dy; write dx, dz, dB, dC, ddt
    nz = 2 if w.has_z else 0
    return T * ((4 + nz) * per_tok_heads + 2 * bc + 2 * 4 * w.nheads)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), "measured"
    return 6800.0, "fallback"


def profile_traffic(kernel_src):
    """Per-launch DRAM bytes of the fused forward from the committed ncu summary,
    or None when the kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "fused_fwd_nemotron_nano.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", txt)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m or not t:
        return None
    cur = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()
    return float(t.group(1)) if m.group(1) == cur else None


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


class NvmlSampler:
    """Clock, power and throttle-reason samples of one GPU through NVML (ctypes), every
    `interval` seconds on a background thread; None from start() when NVML is absent."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid, interval=0.001):
        import ctypes
        self.ct = ctypes
        self.interval = interval
        self.samples = []
        self.stop = threading.Event()
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        key = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        if lib.nvmlDeviceGetHandleByUUID(key.encode(), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for " + key)
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))   # NVML_CLOCK_SM
        self.max_mhz = float(mx.value)

    def _run(self):
        ct, lib = self.ct, self.lib
        clk, pw, rs = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        while not self.stop.is_set():
            a = lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk))
            b = lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw))
            c = self.reasons_fn(self.h, ct.byref(rs))
            if a == 0 and c == 0:
                self.samples.append((float(clk.value), pw.value / 1000.0 if b == 0 else None, int(rs.value)))
            time.sleep(self.interval)

    def __enter__(self):
        self.t = threading.Thread(target=self._run, daemon=True)
        self.t.start()
        return self

    def __exit__(self, *a):
        self.stop.set()
        self.t.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"], "source": "nvml"}
        sm = sorted(v[0] for v in self.samples)
        pw = sorted(v[1] for v in self.samples if v[1] is not None)
        reasons = set()
        for _, _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(sm), "sm_mhz_min": sm[0], "power_w_median": pw[len(pw) // 2] if pw else None,
                "source": "nvml, 1 ms"}


def clock_sampler(dev_index):
    """NVML sampler of the CUDA device (by UUID), else the nvidia-smi one."""
    import torch
    try:
        return NvmlSampler(str(torch.cuda.get_device_properties(dev_index).uuid))
    except (OSError, AttributeError, TypeError):
        return ClockSampler(dev_index)


def median(v):
    v = sorted(v)
    n = len(v)
    return v[n // 2] if n % 2 else 0.5 * (v[n // 2 - 1] + v[n // 2])


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(vals, device="cpu"):
    """Each value's maximum over the ranks of the default process group (unchanged without
    one).  The bench reports whole-job throughput as the units of all ranks over the slowest
    rank's time."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return [float(v) for v in vals]
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


_ORACLE_INPUTS = {}


def _cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part", "hardware")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_oracle_sample(w, seconds_budget=20.0):
    """Time the float64 oracle forward on a bounded sample of the workload:
    all tokens of a few heads (heads are independent), scaled to tokens/s of the
    full workload.  Uses every host core (OpenMP over heads)."""
    import numpy as np
    from state_space_model_scan_gb300 import inputs as I
    from oracle import sequential
    if w.name not in _ORACLE_INPUTS:
        _ORACLE_INPUTS[w.name] = I.to_oracle(I.make_inputs(w), w)
    o = _ORACLE_INPUTS[w.name]
    cores = os.cpu_count() or 1
    # all heads when that stays within the bound, else as many as there are cores
    nheads = w.nheads if w.nheads <= 4 * cores else max(1, min(w.nheads, cores))
    heads = list(range(nheads))
    what = "the full workload" if nheads == w.nheads else "all tokens of %d of %d heads, scaled by heads" % (
        nheads, w.nheads)
    # the oracle on one host thread: all tokens of a few heads, scaled by heads
    n1 = min(4, w.nheads)
    t1 = time.perf_counter()
    sequential.forward(o["x"], o["dt_raw"], o["A"], o["B"], o["C"], D=o["D"], z=o["z"], dt_bias=o["dt_bias"],
                       init=o["init"], cu=o["cu"], heads=list(range(n1)), threads=1)
    dt1 = time.perf_counter() - t1
    # and on every host core
    t0 = time.perf_counter()
    sequential.forward(o["x"], o["dt_raw"], o["A"], o["B"], o["C"], D=o["D"], z=o["z"], dt_bias=o["dt_bias"],
                       init=o["init"], cu=o["cu"], heads=heads, threads=cores)
    dt = time.perf_counter() - t0
    threads = sequential.num_threads()
    tok_per_s = (w.batch * w.seqlen) * (nheads / w.nheads) / dt
    return {"value": tok_per_s, "unit": "tokens/s", "cores": min(cores, nheads), "kind": "oracle",
            "sample": "float64 sequential oracle forward over %s (%d tokens, %.2f s)" % (what, w.batch * w.seqlen, dt),
            "threads": threads,
            "value_1thread": (w.batch * w.seqlen) * (n1 / w.nheads) / dt1,
            "sample_1thread": "one host thread, all tokens of %d of %d heads, scaled by heads (%.2f s)" % (
                n1, w.nheads, dt1),
            "cpu": _cpu_model()}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from state_space_model_scan_gb300 import inputs as I
    w = I.named(WORKLOAD)
    vals = []
    for i in range(args.warmup + args.steps):
        r = cpu_oracle_sample(w)
        if i >= args.warmup:
            vals.append(r)
    v = sum(r["value"] for r in vals) / len(vals)
    toks = w.batch * w.seqlen
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * toks / v, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(w) + " (forward only on the oracle)", "global_batch": w.batch,
                       "seq_len": w.seqlen},
            "cpu_baseline": dict(vals[-1], value=v),
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def sweep_bytes(w, state_bytes=4):
    """Algorithmic HBM bytes of one forward of workload w (inputs read once, y and the
    states written once, initial states read once)."""
    return algorithmic_bytes(w, fwd=True, state_bytes=state_bytes)


def build_extras(dev, s, w):
    """Graph-captured calls of the other kernels, each with its algorithmic bytes per launch."""
    import torch
    from state_space_model_scan_gb300 import inputs as I
    from state_space_model_scan_gb300 import _lib
    out = []
    g = torch.Generator().manual_seed(7)
    T = w.batch * w.seqlen
    width, gsize = w.nheads * w.headdim, w.headdim * w.nheads // w.ngroups
    bf = torch.bfloat16

    def capture(name, fn, nbytes, launches, tokens, keep):
        with torch.cuda.stream(s):
            _lib.check(fn(s), name)
        s.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            _lib.check(fn(torch.cuda.current_stream()), name)
        out.append(dict(name=name, graph=gr, bytes=nbytes, launches=launches, tokens=tokens, keep=keep))

    # gated RMS normalisation over the scan output: rows = tokens, width = H*P, groups of H*P/G
    y = torch.randn(T, width, generator=g).to(bf).to(dev)
    z = torch.randn(T, width, generator=g).to(bf).to(dev)
    nw = (1.0 + 0.1 * torch.randn(width, generator=g)).to(dev)
    nout, dout = torch.empty_like(y), torch.randn(T, width, generator=g).to(bf).to(dev)
    rstd = torch.empty(T, width // gsize, dtype=torch.float32, device=dev)
    ndy, ndz, ndw = torch.empty_like(y), torch.empty_like(z), torch.empty(width, device=dev)
    nprob = _lib.norm_problem(T, width, gsize, 1e-5, bf)
    nws = torch.empty(max(_lib.gated_norm_bwd_workspace_size(nprob), 16), dtype=torch.uint8, device=dev)
    el = T * width * 2
    capture("gated_norm_fwd", lambda st: _lib.gated_norm_fwd(nprob, y, z, nw, nout, rstd, st),
            3 * el + rstd.numel() * 4 + width * 4, 1, T, (y, z, nw, nout, rstd))
    capture("gated_norm_bwd", lambda st: _lib.gated_norm_bwd(nprob, y, z, nw, rstd, dout, ndy, ndz, ndw, nws, st),
            5 * el + rstd.numel() * 4 + 2 * width * 4, 2, T, (dout, ndy, ndz, ndw, nws))
    # causal depthwise conv1d + SiLU over the packed xBC: channels H*P + 2*G*N, width 4
    Cn = width + 2 * w.ngroups * w.dstate
    u = torch.randn(1, T, Cn, generator=g).to(bf).to(dev)
    cw = (0.5 * torch.randn(Cn, 4, generator=g)).to(dev)
    cb = (0.1 * torch.randn(Cn, generator=g)).to(dev)
    cout, cdo = torch.empty_like(u), torch.randn(1, T, Cn, generator=g).to(bf).to(dev)
    cdu, cdw, cdb = torch.empty_like(u), torch.empty_like(cw), torch.empty_like(cb)
    cprob = _lib.conv_problem(1, T, Cn, 4, 0, bf, True)
    cws = torch.empty(_lib.conv1d_bwd_workspace_size(cprob), dtype=torch.uint8, device=dev)
    ue = T * Cn * 2
    capture("conv1d_fwd", lambda st: _lib.conv1d_fwd(cprob, u, cw, cb, None, cout, st), 2 * ue, 1, T,
            (u, cw, cb, cout))
    capture("conv1d_bwd", lambda st: _lib.conv1d_bwd(cprob, u, cw, cb, None, cdo, cdu, cdw, cdb, cws, st),
            3 * ue, 2, T, (cdo, cdu, cdw, cdb, cws))
    # complex-A scan, 8 x 2048 tokens, 16 heads, headdim = dstate = chunk = 64
    ci = {k: (v.to(dev) if v is not None else None) for k, v in I.complex_inputs(8, 2048, 16, seed=434).items()}
    xp = _lib.ComplexProblem(8, 2048, 16, 64, 64, 64)
    yr = torch.empty(8, 2048, 16, 64, dtype=torch.float32, device=dev)
    cfin = torch.empty(8, 16, 64, 64, dtype=torch.complex64, device=dev)
    xws = torch.empty(_lib.complex_fwd_workspace_size(xp), dtype=torch.uint8, device=dev)
    cbytes = 3 * ci["x"].numel() * 8 + ci["dt"].numel() * 4 + yr.numel() * 4 + 2 * cfin.numel() * 8
    capture("complex_fwd_434m", lambda st: _lib.complex_fwd(xp, ci["x"], ci["dt"], ci["A"], ci["B"], ci["C"],
                                                            ci["initial_states"], yr, None, cfin, xws, st),
            cbytes, 1, 8 * 2048, (ci, yr, cfin, xws))
    return out


def run_gpu(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device() if world == 1 else local)
    from state_space_model_scan_gb300 import inputs as I
    from state_space_model_scan_gb300 import _lib
    w = I.named(WORKLOAD)
    inp = I.make_inputs(w, with_grad_inputs=True)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    Bsz, L, H, P, G, N = w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate
    y = torch.empty_like(d["x"])
    fin = torch.empty(Bsz, H, P, N, dtype=torch.float32, device=dev)
    prob = _lib.problem(Bsz, L, H, P, G, N, w.chunk_size)
    fargs = _lib.fwd_args(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], y, D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                          final_states=fin)
    g = dict(dx=torch.empty_like(d["x"]), ddt=torch.empty_like(d["dt_raw"]),
             dA=torch.empty(H, device=dev), dB=torch.empty_like(d["B"]), dC=torch.empty_like(d["C"]),
             dD=torch.empty(H, device=dev), dz=torch.empty_like(d["z"]), ddt_bias=torch.empty(H, device=dev))
    # the training step's forward keeps the carried chunk states; its backward reads them
    cstates = torch.empty(_lib.chunk_states_size(prob, fargs), dtype=torch.uint8, device=dev)
    fargs_t = _lib.fwd_args(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], y, D=d["D"], z=d["z"],
                            dt_bias=d["dt_bias"], final_states=fin, chunk_states=cstates)
    bfa = _lib.fwd_args(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], None, D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                        chunk_states=cstates)
    bargs = _lib.bwd_args(bfa, d["dy"], g["dx"], g["ddt"], g["dA"], g["dB"], g["dC"], dD=g["dD"], dz=g["dz"],
                          ddt_bias=g["ddt_bias"])
    wsf = torch.empty(_lib.fwd_workspace_size(prob, fargs), dtype=torch.uint8, device=dev)
    wsb = torch.empty(_lib.bwd_workspace_size(prob, bargs), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    s = torch.cuda.Stream(device=dev)
    # warm the calls once outside capture (module load, attributes)
    with torch.cuda.stream(s):
        _lib.check(_lib.ssd_fwd(prob, fargs, wsf, s), "ssd_fwd")
        _lib.check(_lib.ssd_fwd(prob, fargs_t, wsf, s), "ssd_fwd")
        _lib.check(_lib.ssd_bwd(prob, bargs, wsb, s), "ssd_bwd")
    s.synchronize()
    gf, gft, gb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(gf, stream=s):
        _lib.check(_lib.ssd_fwd(prob, fargs, wsf, torch.cuda.current_stream()), "ssd_fwd")
    with torch.cuda.graph(gft, stream=s):
        _lib.check(_lib.ssd_fwd(prob, fargs_t, wsf, torch.cuda.current_stream()), "ssd_fwd")
    with torch.cuda.graph(gb, stream=s):
        _lib.check(_lib.ssd_bwd(prob, bargs, wsb, torch.cuda.current_stream()), "ssd_bwd")
    # kernels per call: forward = metadata + fused forward; backward (chunk states kept by the
    # forward) = metadata, dstates, reverse state scan, gradient kernel, the finishing sums
    # (tail pairs' dB/dC, per-head dA/dD/ddt_bias) (the ncu launch list in profiles/ shows the same set)
    launches_fwd, launches_bwd = 2, 5

    # the other forward workloads: the long-sequence sweep and the packed varlen batch
    sweep = []
    if not args.no_sweep:
        import dataclasses
        variants = ([(I.named("long_seq", L=n), torch.float32) for n in (1024, 2048, 4096, 8192, 16384, 32768)] +
                    [(I.named("varlen"), torch.float32),
                     # the variants: dstate 64 on the tensor-core path, and bf16 state storage
                     (dataclasses.replace(w, name="nemotron_nano_dstate64", dstate=64), torch.float32),
                     (dataclasses.replace(I.named("long_seq", L=8192), name="long_seq_L8192_bf16_states"),
                      torch.bfloat16)])
        for sw, sdt in variants:
            si = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in I.make_inputs(sw).items()}
            if si["initial_states"] is not None:
                si["initial_states"] = si["initial_states"].to(sdt)
            S = sw.nseqs
            sy = torch.empty_like(si["x"])
            sfin = torch.empty(S, sw.nheads, sw.headdim, sw.dstate, dtype=sdt, device=dev)
            sprob = _lib.problem(sw.batch, sw.seqlen, sw.nheads, sw.headdim, sw.ngroups, sw.dstate, sw.chunk_size,
                                 S if si["cu_seqlens"] is not None else 0)
            sargs = _lib.fwd_args(si["x"], si["dt_raw"], si["A"], si["B"], si["C"], sy, D=si["D"], z=si["z"],
                                  dt_bias=si["dt_bias"], initial_states=si["initial_states"], final_states=sfin,
                                  cu_seqlens=si["cu_seqlens"])
            sws = torch.empty(_lib.fwd_workspace_size(sprob, sargs), dtype=torch.uint8, device=dev)
            with torch.cuda.stream(s):
                _lib.check(_lib.ssd_fwd(sprob, sargs, sws, s), "ssd_fwd")
            s.synchronize()
            sg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(sg, stream=s):
                _lib.check(_lib.ssd_fwd(sprob, sargs, sws, torch.cuda.current_stream()), "ssd_fwd")
            # metadata + forward (+ the empty-sequence final states of a packed batch, + the state
            # conversions of bf16 or dstate-64 states)
            conv = (1 if sdt == torch.bfloat16 or sw.dstate != 128 else 0) * (1 + (si["initial_states"] is not None))
            sweep.append(dict(w=sw, graph=sg, keep=(si, sy, sfin, sws, sargs), state_bytes=2 if sdt == torch.bfloat16 else 4,
                              launches=(3 if si["cu_seqlens"] is not None else 2) + conv))

    # the steps next to the scan: the gated RMS normalisation after it and the conv1d over the
    # packed xBC before it (Nemotron-Nano widths, 8192 tokens, bf16), and the complex-A scan of
    # the Mamba-3-Lite variant (its 434M configuration); forward and backward where both exist
    extras = []
    if not args.no_sweep:
        extras = build_extras(dev, s, w)

    def step(ev=None, sev=None):
        with torch.cuda.stream(s):
            flush.fill_(float(rank + 1))
            if ev is not None:
                ev[0].record(s)
            gf.replay()                    # inference forward
            if ev is not None:
                ev[1].record(s)
            flush.fill_(float(rank + 2))
            if ev is not None:
                ev[2].record(s)
            gft.replay()                   # training step: forward keeping the chunk states ...
            if ev is not None:
                ev[3].record(s)
            gb.replay()                    # ... and the backward
            if ev is not None:
                ev[4].record(s)
            for j, c in enumerate(sweep + extras):  # the other workloads
                flush.fill_(float(rank + 3 + j))
                if sev is not None:
                    sev[j][0].record(s)
                c["graph"].replay()
                if sev is not None:
                    sev[j][1].record(s)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    sevs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in sweep + extras]
            for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    with clock_sampler(dev.index if dev.index is not None else 0) as clk:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            step(evs[i], sevs[i])
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    fwd_ms = median([e[0].elapsed_time(e[1]) for e in evs])
    fwdt_ms = median([e[2].elapsed_time(e[3]) for e in evs])
    bwd_ms = median([e[3].elapsed_time(e[4]) for e in evs])
    step_ms = median([e[2].elapsed_time(e[4]) for e in evs])
    sweep_ms = [median([sevs[i][j][0].elapsed_time(sevs[i][j][1]) for i in range(args.steps)])
                for j in range(len(sweep) + len(extras))]
    red = max_over_ranks([fwd_ms, fwdt_ms, bwd_ms, step_ms] + sweep_ms, device=dev)
    fwd_ms, fwdt_ms, bwd_ms, step_ms, sweep_ms = red[0], red[1], red[2], red[3], red[4:]
    extra_ms = sweep_ms[len(sweep):]
    sweep_ms = sweep_ms[:len(sweep)]
    toks = w.batch * w.seqlen
    value = world * toks / (fwd_ms * 1e-3)

    # End to end through the C ABI with host buffers: every step copies its own inputs from
    # pinned host memory, runs ssd_fwd and copies its y back.  Steps are independent, so two are
    # in flight (two buffer sets; copy-in, compute and copy-out streams; the host link is
    # full duplex): step i+1's inputs travel while step i computes and step i-1's y returns.
    # (Splitting the inputs over two copy streams was measured no faster: the host-to-device
    # copies run at the link's rate, about 185 GB/s.)
    names = ("x", "dt_raw", "B", "C", "z")
    nset = 2
    dsets = [d] + [{k: torch.empty_like(d[k]) for k in names} for _ in range(nset - 1)]
    ysets = [y] + [torch.empty_like(y) for _ in range(nset - 1)]
    hosts = [{k: d[k].cpu().pin_memory() for k in names} for _ in range(nset)]
    yhosts = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(nset)]
    fsets = [_lib.fwd_args(ds["x"], ds["dt_raw"], d["A"], ds["B"], ds["C"], ys, D=d["D"], z=ds["z"],
                           dt_bias=d["dt_bias"], final_states=fin) for ds, ys in zip(dsets, ysets)]
    h2d = sum(t.numel() * t.element_size() for t in hosts[0].values())
    d2h = yhosts[0].numel() * yhosts[0].element_size()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(nset)]
    ev_c = [torch.cuda.Event() for _ in range(nset)]
    ev_out = [torch.cuda.Event() for _ in range(nset)]
    used = [False] * nset

    def e2e_step(i):
        k = i % nset
        with torch.cuda.stream(s_in):
            if used[k]:
                s_in.wait_event(ev_c[k])   # the set's previous step has read its inputs
            for n in names:
                dsets[k][n].copy_(hosts[k][n], non_blocking=True)
            ev_in[k].record(s_in)
        with torch.cuda.stream(s):
            s.wait_event(ev_in[k])
            if used[k]:
                s.wait_event(ev_out[k])    # and its y has been copied out
            _lib.check(_lib.ssd_fwd(prob, fsets[k], wsf, s), "ssd_fwd")
            ev_c[k].record(s)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_c[k])
            yhosts[k].copy_(ysets[k], non_blocking=True)
            ev_out[k].record(s_out)
        used[k] = True

    for i in range(max(1, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(args.steps):
        e2e_step(i)
    s_out.wait_event(ev_c[(args.steps - 1) % nset])
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / args.steps], device=dev)[0]
    e2e_val = world * toks / (e2e_ms * 1e-3)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peak, peak_kind = measured_peaks()
    alg = algorithmic_bytes(w, fwd=True)
    achieved = alg / (fwd_ms * 1e-3) / 1e9
    traffic = profile_traffic(os.path.join(ROOT, "state_space_model_scan_gb300", "csrc", "fused_fwd.cu"))
    sweep_out = []
    for c, ms in zip(sweep, sweep_ms):
        sw = c["w"]
        b = sweep_bytes(sw, c["state_bytes"])
        sweep_out.append({"workload": sw.name, "seqlen": sw.seqlen, "nseqs": sw.nseqs, "nheads": sw.nheads,
                          "dstate": sw.dstate, "state_dtype": "bf16" if c["state_bytes"] == 2 else "f32",
                          "chunk_size": sw.chunk_size, "fwd_ms": ms, "tokens_per_s": sw.batch * sw.seqlen / (ms * 1e-3),
                          "algorithmic_bytes": b, "achieved_gbs": b / (ms * 1e-3) / 1e9,
                          "roofline_frac": b / (ms * 1e-3) / 1e9 / peak})
    extras_out = []
    for c, ms in zip(extras, extra_ms):
        gbs = c["bytes"] / (ms * 1e-3) / 1e9
        extras_out.append({"workload": c["name"], "ms": ms, "tokens_per_s": c["tokens"] / (ms * 1e-3),
                           "algorithmic_bytes": c["bytes"], "achieved_gbs": gbs, "roofline_frac": gbs / peak,
                           "launches": c["launches"]})
    n_launch_step = (2 * launches_fwd + launches_bwd + sum(c["launches"] for c in sweep) +
                     sum(c["launches"] for c in extras))
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(w), "global_batch": w.batch * world, "seq_len": w.seqlen,
                   "chunk_size": w.chunk_size, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed before every timed call (256 MB write)",
                   "timing": "CUDA graph replay, CUDA events, median over the steps"},
        "fwd_ms": fwd_ms, "fwd_bwd_ms": step_ms, "fwd_train_ms": fwdt_ms, "bwd_ms": bwd_ms,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "ssd_fwd (metadata + fused tensor-core forward)",
                     "algorithmic_bytes_per_launch": alg, "peak_source": peak_kind},
        "bwd_roofline": {"bound": "hbm", "achieved": algorithmic_bytes(w, fwd=False) / (bwd_ms * 1e-3) / 1e9,
                         "peak": peak, "unit": "GB/s",
                         "frac": algorithmic_bytes(w, fwd=False) / (bwd_ms * 1e-3) / 1e9 / peak,
                         "algorithmic_bytes_per_launch": algorithmic_bytes(w, fwd=False)},
        "sweep": sweep_out,
        "extras": extras_out,
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        # library kernels in the two timed regions: the step loop and the end-to-end loop
        "gpu_launches": args.steps * n_launch_step + args.steps * launches_fwd,
        "clocks": clk.summary(),
        "wall_s": wall,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(w)
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def run_fwd_only(args):
    """Forward only, plain calls (no graph, no backward): the command the ncu captures run."""
    import torch
    from state_space_model_scan_gb300 import inputs as I
    from state_space_model_scan_gb300.api import ssd_forward, Workspace
    w = I.named(WORKLOAD)
    inp = I.make_inputs(w)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    ws = Workspace()
    y = torch.empty_like(d["x"])
    fin = torch.empty(w.batch, w.nheads, w.headdim, w.dstate, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for i in range(args.warmup + args.steps):
        e0.record()
        ssd_forward(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"], dt_bias=d["dt_bias"],
                    chunk_size=w.chunk_size, workspace=ws, y=y, final_states=fin, seg_chunks=args.seg_chunks)
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1))
    print(json.dumps({"mode": "fwd", "workload": WORKLOAD, "fwd_ms": times,
                      "tokens_per_s": w.batch * w.seqlen / (sum(times) / len(times) * 1e-3)}))


def run_extras_only(args):
    """The kernels around the scan only (graph replays, L2 flushed before each): the command the
    ncu captures of those kernels run."""
    import torch
    from state_space_model_scan_gb300 import inputs as I
    dev = torch.device("cuda", torch.cuda.current_device())
    s = torch.cuda.Stream(device=dev)
    extras = build_extras(dev, s, I.named(WORKLOAD))
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    times = {c["name"]: [] for c in extras}
    for i in range(args.warmup + args.steps):
        for c in extras:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                flush.fill_(float(i))
                e0.record(s)
                c["graph"].replay()
                e1.record(s)
            s.synchronize()
            if i >= args.warmup:
                times[c["name"]].append(e0.elapsed_time(e1))
    print(json.dumps({"mode": "extras", "ms": {k: median(v) for k, v in times.items()}}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mode", default="bench", choices=["bench", "fwd", "extras"])
    ap.add_argument("--no-sweep", action="store_true", help="time the Nemotron-Nano workload only")
    ap.add_argument("--seg-chunks", type=int, default=0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.mode == "fwd":
        run_fwd_only(args)
    elif args.mode == "extras":
        run_extras_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
