"""Benchmark: chunk-level Gated DeltaNet fwd+bwd tokens/s on one GB300.

Workload: B=1, H=16, d_k=d_v=128, T=262144 bf16 (fp32 state), split into 8
chunks of 32768 run in order through gdn_chunk_fwd (state chained forward),
then in reverse through gdn_chunk_bwd (state gradient chained backward),
do ~ N(0,1)*0.02, dS_out = 0 at the sequence end. One step = that whole
forward + backward pass. Inputs are synthetic (seeded) and larger than L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun) every rank runs its own independent sequence (weak
scaling; heads and sequences share nothing, so there is no collective) and
`value` is the total tokens of all ranks per second. Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "GDN chunk fwd+bwd tokens/s at H=16,d=128,256K on 1 GB300; % of roofline"
UNIT = "tokens/s"
WORKLOAD_INDEX = 2


def measured_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu capture
    (profiles/kernel_dram_traffic.json), or None if the kernel's source has
    changed since the counters were taken."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "kernel_dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
        def sha(rel):
            with open(os.path.join(ROOT, rel), "rb") as f:
                return hashlib.sha256(f.read()).hexdigest()
        common = "chunked_linear_recurrence_gated_gb300/csrc/gdn_common.cuh"
        if sha(rec["source"]) != rec["source_sha256"] or sha(common) != rec["common_sha256"]:
            return None
        return rec["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------- algorithmic model
def alg_bytes_per_token_head(dk, dv, esz=2):
    """Bytes the method must move per token-head: fwd reads q,k,v (+g,beta) and
    writes o; bwd reads q,k,v,g,beta,do and writes dq,dk,dv,dg,dbeta."""
    fwd = esz * (2 * dk + dv) + 2 * esz + esz * dv
    bwd = esz * (2 * dk + dv + dv) + 2 * esz + esz * (2 * dk + dv) + 2 * esz
    return fwd, bwd


def alg_flops_per_token_head(dk, dv, C=64):
    fwd = 2 * C * (3 * dk + 2 * dv) + 6 * dk * dv + C * C / 3
    bwd = 18 * C * dk + 10 * C * dv + 16 * dk * dv + 4 * C * C + C * C / 3
    return fwd, bwd


# Per-kernel algorithmic work per 64-token block-head (C = 64), used for the
# dominant kernel's roofline: bytes the kernel must move in this design
# (inputs, outputs and workspace intermediates it reads or writes), and the
# contraction flops it must do.
def kernel_model(name, dk, dv, esz=2, C=64):
    f4 = 4
    if name == "simt_pre":
        by = C * (dk + dv) * esz + 2 * C * esz + C * (dk + dv) * f4 + C * f4
        fl = 2 * C * C * dk + C ** 3 / 3 + 2 * C * C * dk + 2 * C * C * dv
    elif name == "simt_st":
        by = C * (dk + dv) * f4 + C * dk * esz + C * f4 + dk * dv * f4 + C * dv * f4
        fl = 4 * C * dk * dv
    elif name == "simt_out":
        by = 2 * C * dk * esz + C * f4 + dk * dv * f4 + C * dv * f4 + C * dv * esz
        fl = 2 * C * dk * dv + 2 * C * C * dk + 2 * C * C * dv
    elif name == "simt_st_bwd":
        by = 2 * C * dk * esz + C * dk * f4 + C * dv * esz + C * f4 + dk * dv * f4 + C * dv * f4
        fl = 2 * C * C * dk + 2 * C * C * dv + 6 * C * dk * dv
    elif name == "simt_grad":
        by = (C * (2 * dk + 2 * dv) * esz + 2 * C * esz + 2 * dk * dv * f4 + 2 * C * dv * f4
              + C * C * f4 + C * f4 + C * (2 * dk + dv) * esz + 2 * C * esz)
        fl = 6 * C * dk * dv + 10 * C * C * dk + 6 * C * C * dv + 4 * C ** 3
    elif name == "tc_pre":
        by = C * (2 * dk + dv) * esz + 2 * C * esz + C * (dk + dv) * esz + C * C * esz + C * f4
        fl = 4 * C * C * dk + C ** 3 / 3 + 2 * C * C * dk + 2 * C * C * dv
    elif name == "tc_chain_fwd":
        by = C * (3 * dk + dv) * esz + C * C * esz + C * f4 + C * dv * esz
        fl = 6 * C * dk * dv + 2 * C * C * dv
    elif name == "tc_chain_fwd_keep":  # forward chain that also keeps H_b, V^new
        by = (C * (3 * dk + dv) * esz + C * C * esz + C * f4 + C * dv * esz
              + dk * dv * esz + C * dv * esz)
        fl = 6 * C * dk * dv + 2 * C * C * dv
    elif name == "tc_chain_rev":  # reverse chain alone
        by = C * (3 * dk + dv) * esz + C * C * esz + C * f4 + dk * dv * esz + C * dv * esz
        fl = 6 * C * dk * dv + 2 * C * C * dv
    elif name == "tc_chains_bwd":  # recompute + reverse chains in one launch
        by = (C * (2 * dk + dv) * esz + C * f4 + dk * dv * esz + C * dv * esz
              + C * (3 * dk + dv) * esz + C * C * esz + C * f4 + dk * dv * esz + C * dv * esz)
        fl = 4 * C * dk * dv + 6 * C * dk * dv + 2 * C * C * dv
    elif name == "tc_fwd_overlap":  # split forward: Pre and the forward chain, overlapped
        by = (C * (2 * dk + dv) * esz + 2 * C * esz + C * (dk + dv) * esz + C * C * esz + C * f4
              + C * (3 * dk + dv) * esz + C * C * esz + C * f4 + C * dv * esz)
        fl = 4 * C * C * dk + C ** 3 / 3 + 2 * C * C * dk + 2 * C * C * dv + 6 * C * dk * dv + 2 * C * C * dv
    elif name == "tc_grad":
        by = (C * (2 * dk + 2 * dv) * esz + C * esz + C * C * esz + C * f4 + 2 * dk * dv * esz
              + 2 * C * dv * esz + C * (2 * dk + dv) * esz + 2 * C * esz)
        fl = 6 * C * dk * dv + 4 * C * C * dv + 14 * C * C * dk + 4 * C ** 3
    else:
        return None
    return by, fl


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi every 200 ms
    while in context; the lines are kept in memory (or appended to
    $GDN_CLOCKS_CSV when set)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line)

    def __enter__(self):
        import threading

        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)
            out = os.environ.get("GDN_CLOCKS_CSV")
            if out:
                with open(out, "a") as f:
                    f.writelines(self.lines)
        return False

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- the step
class Runner:
    def __init__(self, w, dev, seed_offset=0, reuse=True):
        from chunked_linear_recurrence_gated_gb300 import gdn
        from chunked_linear_recurrence_gated_gb300.inputs import make_workload_inputs

        self.gdn = gdn
        self.w = w
        self.dev = dev
        x = make_workload_inputs(w, device=dev)
        self.x = x
        B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv
        self.o = torch.empty(B, T, H, dv, dtype=w.torch_dtype, device=dev)
        self.dq = torch.empty_like(x["q"])
        self.dk = torch.empty_like(x["k"])
        self.dv = torch.empty_like(x["v"])
        self.dg = torch.empty_like(x["g"])
        self.db = torch.empty_like(x["beta"])
        n = len(w.chunks)
        self.S = [torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev) for _ in range(n + 1)]
        self.S[0].zero_()
        self.dS = [torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev) for _ in range(n)]
        self.bounds = np.concatenate([[0], np.cumsum(w.chunks)]).astype(int)
        Lmax = max(w.chunks)
        shp = gdn.gdn_shape(B, Lmax, H, dk, dv, 1 if w.dtype == "bf16" else 0)
        self.reuse = reuse
        if reuse:
            # the backward reads the per-block products its chunk's forward kept
            self.ws_s = gdn.alloc_workspace(gdn.chunk_workspace_bytes(shp, gdn.GDN_WS_SAVED), dev)
            self.saved = []
            for L in w.chunks:
                s_i = gdn.gdn_shape(B, int(L), H, dk, dv, shp.dtype)
                self.saved.append(gdn.alloc_workspace(gdn.chunk_saved_bytes(s_i), dev))
        else:
            self.ws_f = gdn.alloc_workspace(gdn.chunk_workspace_bytes(shp, False), dev)
            self.ws_b = gdn.alloc_workspace(gdn.chunk_workspace_bytes(shp, True), dev)
        self.launches_per_step = None

    def sl(self, t, i):
        return t[:, self.bounds[i]:self.bounds[i + 1]]

    def fwd_chunk(self, i):
        g, x = self.gdn, self.x
        args = (self.sl(x["q"], i), self.sl(x["k"], i), self.sl(x["v"], i),
                self.sl(x["g"], i), self.sl(x["beta"], i))
        if self.reuse:
            g.gdn_chunk_fwd_save(*args, S_in=self.S[i], saved=self.saved[i],
                                 o=self.sl(self.o, i), S_out=self.S[i + 1], workspace=self.ws_s)
        else:
            g.gdn_chunk_fwd(*args, S_in=self.S[i], o=self.sl(self.o, i), S_out=self.S[i + 1],
                            workspace=self.ws_f)

    def bwd_chunk(self, i):
        g, x = self.gdn, self.x
        n = len(self.w.chunks)
        args = (self.sl(x["q"], i), self.sl(x["k"], i), self.sl(x["v"], i),
                self.sl(x["g"], i), self.sl(x["beta"], i), self.S[i], self.sl(x["do"], i))
        grads = (self.sl(self.dq, i), self.sl(self.dk, i), self.sl(self.dv, i),
                 self.sl(self.dg, i), self.sl(self.db, i))
        dS_out = self.dS[i + 1] if i + 1 < n else None
        if self.reuse:
            g.gdn_chunk_bwd_saved(*args, self.saved[i], dS_out=dS_out, grads=grads,
                                  dS_in=self.dS[i], workspace=self.ws_s)
        else:
            g.gdn_chunk_bwd(*args, dS_out=dS_out, grads=grads, dS_in=self.dS[i],
                            workspace=self.ws_b)

    def step(self):
        n = len(self.w.chunks)
        for i in range(n):
            self.fwd_chunk(i)
        for i in reversed(range(n)):
            self.bwd_chunk(i)

    def fwd_step(self):
        for i in range(len(self.w.chunks)):
            self.fwd_chunk(i)

    def units(self):
        """Token-heads of each call of one step (the units a launch processes)."""
        return [self.w.B * int(L) * self.w.H for L in self.w.chunks]


class VarlenRunner:
    """The packed variable-length workload: one gdn_varlen_fwd and one
    gdn_varlen_bwd call over all sequences (state restarts at every start)."""

    def __init__(self, w, dev):
        from chunked_linear_recurrence_gated_gb300 import gdn
        from chunked_linear_recurrence_gated_gb300.inputs import cu_seqlens, make_workload_inputs

        self.gdn = gdn
        self.w = w
        self.x = make_workload_inputs(w, device=dev)
        self.cu = cu_seqlens(w.seqlens).to(dev)
        nseq = len(w.seqlens)
        self.o = torch.empty(1, w.T, w.H, w.dv, dtype=w.torch_dtype, device=dev)
        self.Sf = torch.empty(nseq, w.H, w.dk, w.dv, dtype=torch.float32, device=dev)
        self.dS0 = torch.empty_like(self.Sf)
        x = self.x
        self.grads = (torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"]),
                      torch.empty_like(x["g"]), torch.empty_like(x["beta"]))
        shp = gdn.shape_of(x["q"], x["v"])
        self.ws_f = gdn.alloc_workspace(gdn.varlen_workspace_bytes(shp, nseq, False), dev)
        self.ws_b = gdn.alloc_workspace(gdn.varlen_workspace_bytes(shp, nseq, True), dev)

    def fwd_step(self):
        x = self.x
        self.gdn.gdn_varlen_fwd(self.cu, x["q"], x["k"], x["v"], x["g"], x["beta"], o=self.o,
                                S_final=self.Sf, workspace=self.ws_f)

    def step(self):
        x = self.x
        self.fwd_step()
        self.gdn.gdn_varlen_bwd(self.cu, x["q"], x["k"], x["v"], x["g"], x["beta"], None,
                                x["do"], grads=self.grads, dS0=self.dS0, workspace=self.ws_b)

    def units(self):
        return [self.w.T * self.w.H]


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def aggregate(ms_step_local, tokens_per_rank, world, device=None):
    """Whole-job throughput of a weak-scaling run: every rank processed its own
    `tokens_per_rank` tokens; the step time is the slowest rank's (max over
    ranks). Returns (ms_per_step, tokens_per_second)."""
    ms = float(ms_step_local)
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    return ms, tokens_per_rank * world / (ms / 1e3)


def time_steps(fn, K, dev):
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    s.record()
    for _ in range(K):
        fn()
    e.record()
    torch.cuda.synchronize(dev)
    return s.elapsed_time(e)


def gpu_local_cpus(dev_index):
    """Host CPUs of the GPU's NUMA node (Linux sysfs via the PCI bus id), or None."""
    try:
        out = subprocess.run(["nvidia-smi", f"--id={dev_index}", "--query-gpu=pci.bus_id",
                              "--format=csv,noheader"], capture_output=True, text=True,
                             timeout=20).stdout.strip()
        dom, rest = out.split(":", 1)
        bus = f"{int(dom, 16):04x}:{rest}".lower()
        with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
            node = int(f.read().strip())
        if node < 0:
            return None
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
        cpus &= os.sched_getaffinity(0)
        return (node, cpus) if cpus else None
    except Exception:
        return None


def e2e_measure(runner, K, dev):
    """Same step through the public API with host buffers: every chunk's inputs
    are copied in from pinned host memory and its results (o and every
    gradient) copied out inside the timed region. The copies run per chunk on
    two copy streams, overlapped with the kernels of the neighbouring chunks.
    The device holds two sets of input buffers, used by alternate steps, so a
    step's inputs are uploaded while the previous step's backward runs and its
    gradients are downloaded (both directions of the host link busy at once,
    as a training loop prefetches its next batch); a step's kernels start only
    after the previous step's results have all been read back."""
    x = runner.x
    keys = ["q", "k", "v", "g", "beta", "do"]
    # pinned buffers on the GPU's own NUMA node (the host link is the bound here)
    saved_aff = os.sched_getaffinity(0)
    local = gpu_local_cpus(dev.index if dev.index is not None else 0)
    if local:
        os.sched_setaffinity(0, local[1])
    host_in = {k: torch.empty(x[k].shape, dtype=x[k].dtype, pin_memory=True) for k in keys}
    for k in keys:
        host_in[k].copy_(x[k])
    outs = [runner.dq, runner.dk, runner.dv, runner.dg, runner.db]
    host_o = torch.empty(runner.o.shape, dtype=runner.o.dtype, pin_memory=True)
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_o.numel() * host_o.element_size() + sum(t.numel() * t.element_size() for t in host_out)
    comp = torch.cuda.current_stream(dev)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    n = len(runner.w.chunks)
    xsets = [x, {k: torch.empty_like(x[k]) for k in keys}]
    free = [None, None]  # per input set: the step that last read it has finished its kernels
    count = [0]

    fwd_keys = ["q", "k", "v", "g", "beta"]

    def one():
        si = count[0] % 2
        count[0] += 1
        xi = xsets[si]
        runner.x = xi
        ready, ready_do = [], [None] * n
        with torch.cuda.stream(s_in):
            if free[si] is not None:
                s_in.wait_event(free[si])
            # forward inputs in chunk order, then dO in the backward's (reverse) order
            for i in range(n):
                for k in fwd_keys:
                    runner.sl(xi[k], i).copy_(runner.sl(host_in[k], i), non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_in)
                ready.append(ev)
            for i in reversed(range(n)):
                runner.sl(xi["do"], i).copy_(runner.sl(host_in["do"], i), non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_in)
                ready_do[i] = ev
        for i in range(n):
            comp.wait_event(ready[i])
            runner.fwd_chunk(i)
            done = torch.cuda.Event()
            done.record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                runner.sl(host_o, i).copy_(runner.sl(runner.o, i), non_blocking=True)
        for i in reversed(range(n)):
            comp.wait_event(ready_do[i])
            runner.bwd_chunk(i)
            done = torch.cuda.Event()
            done.record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                for h, t in zip(host_out, outs):
                    runner.sl(h, i).copy_(runner.sl(t, i), non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(comp)
        free[si] = ev
        comp.wait_stream(s_out)

    one()
    ms = time_steps(one, K, dev)
    runner.x = x
    os.sched_setaffinity(0, saved_aff)
    return ms / K, h2d, d2h, (local[0] if local else None)


def conv_measure(K, warmup, dev, hbm, peak_kind, tokens=0):
    """The causal short convolution carried across chunks (the auxiliary
    local-convolution states), measured on a Gated DeltaNet layer's q / k / v
    convolution of the same 256K-token sequence: fwd over the 8 chained chunks,
    then bwd in reverse order. Algorithmic bytes: fwd reads x and writes y, bwd
    reads x and dy and writes dx (bf16), plus the (W - 1)-row states."""
    from chunked_linear_recurrence_gated_gb300 import gdn
    from chunked_linear_recurrence_gated_gb300.inputs import CONV_BENCH, make_conv_inputs

    cfg = dict(CONV_BENCH)
    if tokens:  # the first chunks up to `tokens` (small profiling cases)
        keep = [c for i, c in enumerate(cfg["chunks"]) if sum(cfg["chunks"][:i + 1]) <= tokens]
        if not keep:
            raise SystemExit("--tokens is smaller than the convolution's first chunk")
        cfg.update(chunks=keep, T=sum(keep))
    B, T, C, W, act = cfg["B"], cfg["T"], cfg["C"], cfg["W"], cfg["act"]
    d = make_conv_inputs(B, T, C, W, dtype=torch.bfloat16, device=dev, with_state=False)
    y = torch.empty_like(d["x"])
    dx = torch.empty_like(d["x"])
    n = len(cfg["chunks"])
    bounds = np.concatenate([[0], np.cumsum(cfg["chunks"])]).astype(int)
    st = [None] + [torch.empty(B, W - 1, C, dtype=torch.bfloat16, device=dev) for _ in range(n)]
    dst = [torch.empty(B, W - 1, C, dtype=torch.bfloat16, device=dev) for _ in range(n)]
    dws = [torch.empty_like(d["w"]) for _ in range(n)]
    dbs = [torch.empty_like(d["b"]) for _ in range(n)]
    shp = gdn.gdn_conv_shape(B, max(cfg["chunks"]), C, W, 1, gdn.CONV_ACT[act])
    ws = gdn.alloc_workspace(gdn.load().gdn_conv_workspace_bytes(ctypes.byref(shp)), dev)
    sl = lambda t, i: t[:, bounds[i]:bounds[i + 1]]

    def step():
        for i in range(n):
            gdn.gdn_conv_fwd(sl(d["x"], i), d["w"], d["b"], st[i], act, y=sl(y, i),
                             state_out=st[i + 1])
        for i in reversed(range(n)):
            gdn.gdn_conv_bwd(sl(d["x"], i), d["w"], d["b"], st[i], sl(d["dy"], i),
                             dst[i + 1] if i + 1 < n else None, act, dx=sl(dx, i), dw=dws[i],
                             db=dbs[i], dstate_in=dst[i], workspace=ws)

    for _ in range(max(warmup, 3)):
        step()
    ms = time_steps(step, K, dev) / K
    timer = gdn.KernelTimer(capacity=512)
    with timer:
        step()
    torch.cuda.synchronize(dev)
    per = {k: sum(v) for k, v in timer.per_kernel().items()}
    elems = B * T * C
    alg = 5 * 2 * elems  # bytes
    kb = {"conv_fwd": 2 * 2 * elems, "conv_bwd": 3 * 2 * elems}
    kernels = {k: {"ms_per_step": v, "alg_gb_per_s": (kb[k] / (v / 1e3) / 1e9) if k in kb else None,
                   "frac": (kb[k] / (v / 1e3) / 1e9 / hbm) if k in kb else None}
               for k, v in per.items()}
    return {"workload": f"qkv short conv B{B} T{T} C{C} W{W} {act} bf16, "
                        f"{n} x {max(cfg['chunks'])} chained",
            "ms_per_step": ms, "tokens_per_s": B * T / (ms / 1e3),
            "alg_bytes_per_step": alg,
            "roofline": {"bound": "hbm", "achieved": alg / (ms / 1e3) / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": alg / (ms / 1e3) / 1e9 / hbm,
                         "peak_source": peak_kind},
            "kernels": kernels}


def cpu_baseline(w, x, max_tokens=32768):
    """The oracle, as it stands, on a bounded sample: all heads of the first chunk."""
    import oracle

    L = min(max_tokens, w.chunks[0] if w.chunks else w.T)
    sub = {k: x[k][:, :L].float().cpu() for k in ("q", "k", "v", "g", "beta", "do")}
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.fwd(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], None, nthreads=threads)
    oracle.bwd(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], None, sub["do"], None,
               nthreads=threads)
    dt = time.perf_counter() - t0
    return {"value": L / dt, "unit": UNIT, "cores": min(threads, w.H * w.B), "kind": "oracle",
            "sample": f"fwd+bwd of the first {L} tokens of the sequence, all {w.H} heads "
                      f"(fp64 token loop, {dt:.1f} s)"}


def workload_config(w, world, recompute):
    cfg = {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
           "state": "fp32",
           "backward": ("recomputes T / W / U and the per-block states from S_in "
                        "(gdn_chunk_bwd)" if recompute else
                        "reads the per-block products its chunk's forward kept "
                        "(gdn_chunk_fwd_save / gdn_chunk_bwd_saved)"),
           "l2": "inputs larger than L2 (no flush)",
           "parallelism": f"dp{world} (independent sequence per GPU)"}
    if w.seqlens is not None:
        cfg["seqlens"] = len(w.seqlens)
    else:
        cfg["chunks"] = w.chunks
    return cfg


def op_roofline(w, ms, which="fwd+bwd"):
    """The op's roofline for `which` (SURVEY 8(d) bytes / flops per token-head):
    the slower of its algorithmic bytes at the measured HBM bandwidth and its
    algorithmic flops at the measured bf16 tensor rate."""
    hbm, bf16, _, _ = peaks()
    fb, bb = alg_bytes_per_token_head(w.dk, w.dv)
    ff, bf = alg_flops_per_token_head(w.dk, w.dv)
    by, fl = (fb + bb, ff + bf) if which == "fwd+bwd" else (fb, ff)
    th = w.B * w.T * w.H
    t_bytes = by * th / (hbm * 1e9)
    t_flops = fl * th / (bf16 * 1e12)
    roof_ms = max(t_bytes, t_flops) * 1e3
    return {"roofline_ms": roof_ms, "bound": "hbm" if t_bytes >= t_flops else "tensor",
            "frac_of_roofline": roof_ms / ms,
            "roofline_tokens_per_s": w.B * w.T / (roof_ms / 1e3)}


# Which phase of the op each kernel belongs to: its roofline credits it with
# that phase's algorithmic bytes for the token-heads it processes.
KERNEL_PHASE = {"tc_grad": "bwd", "simt_grad": "bwd", "tc_chains_bwd": "bwd",
                "tc_chain_rev": "bwd", "simt_st_bwd": "bwd"}


def kernel_roofline(name, per_launch_ms, units_per_launch, w, hbm, peak_kind):
    """Roofline of one kernel: SURVEY 8(d)'s algorithmic bytes per token-head of
    the phase it serves (fwd: q, k, v, g, beta in, o out; bwd: q, k, v, g,
    beta, do in, dq, dk, dv, dg, dbeta out) x the token-heads of each launch,
    over the summed launch time."""
    fb, bb = alg_bytes_per_token_head(w.dk, w.dv)
    per_th = bb if KERNEL_PHASE.get(name, "fwd") == "bwd" else fb
    alg = per_th * sum(units_per_launch)
    t = sum(per_launch_ms) / 1e3
    achieved = alg / t / 1e9
    n = len(per_launch_ms)
    launch_units = sum(units_per_launch) // max(n, 1)
    traffic = measured_traffic(name) if launch_units == 32768 * 16 else None
    return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "traffic": traffic, "kernel": name,
            "alg_bytes_per_launch": alg / max(n, 1), "launch_ms": sum(per_launch_ms) / max(n, 1),
            "alg_bytes_per_token_head": per_th, "phase": KERNEL_PHASE.get(name, "fwd"),
            "peak_source": peak_kind, "timing": "CUDA events on the launch stream"}


def time_mode(runner, K, warmup, dev):
    """ms per fwd+bwd step and per forward-only step of `runner` (CUDA events,
    W warm-up steps first)."""
    for _ in range(max(warmup, 3)):
        runner.step()
    torch.cuda.synchronize(dev)
    ms = time_steps(runner.step, K, dev) / K
    for _ in range(2):
        runner.fwd_step()
    ms_f = time_steps(runner.fwd_step, K, dev) / K
    return ms, ms_f


def per_kernel(runner, dev, nsteps=2):
    """{kernel: [ms of each launch]} of `nsteps` instrumented steps."""
    from chunked_linear_recurrence_gated_gb300 import gdn

    timer = gdn.KernelTimer(capacity=4096)
    with timer:
        for _ in range(nsteps):
            runner.step()
    torch.cuda.synchronize(dev)
    return timer.per_kernel()


SPLIT_SETTINGS = [(1, 0, 1), (1, 0, 2), (2, 0, 2), (4, 0, 2), (8, 0, 2), (16, 0, 2),
                  (2, 300, 2), (2, 500, 2), (2, 700, 2), (2, 900, 2), (4, 0, 1)]


def split_sweep(runner, K, dev):
    """The forward with the chunk split into segments whose Pre kernel runs
    beside the previous segment's state chain (the StateFlow review's
    split-and-overlap of the state transition with the dense kernels): forward
    ms per step for (segments, first segment's share f, 16-column groups per
    chain CTA), against the serial order (1 segment)."""
    from chunked_linear_recurrence_gated_gb300 import gdn

    rows = []
    for seg, pm, rg in SPLIT_SETTINGS:
        gdn.set_fwd_split(seg, pm, rg)
        for _ in range(2):
            runner.fwd_step()
        ms = time_steps(runner.fwd_step, K, dev) / K
        rows.append({"segments": seg, "first_fraction": (pm / 1000) if pm else None,
                     "chain_rg": rg, "fwd_ms": ms})
    gdn.set_fwd_split(0, 0, 0)
    return rows


def other_workloads(dev, K, warmup):
    """fwd and fwd+bwd tokens/s of the other bf16 workloads (mid 8K, hybrid
    alpha = 0.5 with H 32, varlen with dv 256), recomputing backward, against
    their op rooflines."""
    from chunked_linear_recurrence_gated_gb300.inputs import workload

    out = {}
    for idx in (1, 3, 4):
        w = workload(idx)
        r = VarlenRunner(w, dev) if w.seqlens is not None else Runner(w, dev, reuse=False)
        ms, ms_f = time_mode(r, K, warmup, dev)
        out[w.name] = {"ms_per_step": ms, "tokens_per_s": w.B * w.T / (ms / 1e3),
                       "frac_of_roofline": op_roofline(w, ms)["frac_of_roofline"],
                       "fwd_ms": ms_f, "fwd_tokens_per_s": w.B * w.T / (ms_f / 1e3),
                       "fwd_frac_of_roofline": op_roofline(w, ms_f, "fwd")["frac_of_roofline"],
                       "api": "gdn_varlen_fwd/bwd" if w.seqlens is not None else
                              f"gdn_chunk_fwd/bwd over {len(w.chunks)} chained chunks"}
        del r
        torch.cuda.empty_cache()
    return out


def reference_arm(args, w):
    """The oracle timed on the host cores, a bounded sample per step."""
    import oracle
    from chunked_linear_recurrence_gated_gb300.inputs import make_workload_inputs

    x = make_workload_inputs(w, device="cpu")
    L = 2048
    sub = {k: x[k][:, :L].float() for k in ("q", "k", "v", "g", "beta", "do")}
    threads = oracle.default_threads()

    def one():
        oracle.fwd(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], None, nthreads=threads)
        oracle.bwd(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], None, sub["do"], None,
                   nthreads=threads)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = (time.perf_counter() - t0) / args.steps
    value = L / dt
    sample = f"fwd+bwd of the first {L} tokens, all {w.H} heads, per step"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": dict(workload_config(w, args.gpus, not args.kept), sample_tokens=L,
                       runs_on=f"host cores of rank 0 ({threads} threads)"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(threads, w.H),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", type=int, default=WORKLOAD_INDEX,
                    help="workload index (1-3: fixed-length chunked bf16 workloads, "
                         "4: packed varlen)")
    ap.add_argument("--no-conv", action="store_true",
                    help="skip the short-convolution measurement")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the summary of the other workloads")
    ap.add_argument("--no-split-sweep", action="store_true",
                    help="skip the split-forward (state-transition / dense overlap) sweep")
    ap.add_argument("--kept", action="store_true",
                    help="headline on the backward that reads the products its chunk's "
                         "forward kept instead of the recomputing backward")
    ap.add_argument("--tokens", type=int, default=0,
                    help="run only the first N tokens (a whole number of chunks); "
                         "for small profiling cases")
    ap.add_argument("--conv-only", action="store_true",
                    help="time only the short convolution (with --tokens, its first chunks); "
                         "prints its summary; for profiling")
    args = ap.parse_args()

    import dataclasses

    from chunked_linear_recurrence_gated_gb300.inputs import workload

    w = workload(args.workload)
    if args.tokens and w.seqlens is None:
        n = 0
        acc = 0
        while n < len(w.chunks) and acc + w.chunks[n] <= args.tokens:
            acc += w.chunks[n]
            n += 1
        if n == 0:
            raise SystemExit("--tokens is smaller than the first chunk")
        w = dataclasses.replace(w, T=acc, chunks=w.chunks[:n],
                                name=f"{w.name}_first{acc}")
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    recompute = not args.kept

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args, w)))
        return

    from chunked_linear_recurrence_gated_gb300 import gdn

    gdn.load()  # fails loudly if the CUDA library is missing
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)

    if args.conv_only:
        hbm, _, _, peak_kind = peaks()
        conv = conv_measure(max(3, min(args.steps, 10)), args.warmup, dev, hbm, peak_kind,
                            tokens=args.tokens)
        if rank == 0:
            print(json.dumps({"short_conv": conv}))
        return
    varlen = w.seqlens is not None
    runner = VarlenRunner(w, dev) if varlen else Runner(w, dev, reuse=not recompute)
    for _ in range(max(args.warmup, 3)):
        runner.step()
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_start = time.perf_counter()
        while time.perf_counter() - t_start < 0.6:  # let the clock sampler start under load
            runner.step()
            torch.cuda.synchronize(dev)
        barrier(world)
        ms = time_steps(runner.step, args.steps, dev)
    barrier(world)
    ms_step, value = aggregate(ms / args.steps, w.B * w.T, world, device=dev)
    tokens = w.B * w.T * world
    # forward alone (the same calls' first half)
    for _ in range(2):
        runner.fwd_step()
    barrier(world)
    ms_f = time_steps(runner.fwd_step, args.steps, dev)
    ms_fwd, value_fwd = aggregate(ms_f / args.steps, w.B * w.T, world, device=dev)

    # state-transition / dense-kernel overlap in the forward (split fraction sweep)
    f2 = None
    if not varlen and not args.no_split_sweep:
        rows = split_sweep(runner, max(3, min(args.steps, 10)), dev)
        serial = next(r["fwd_ms"] for r in rows if r["segments"] == 1 and r["chain_rg"] == 1)
        best = min(rows, key=lambda r: r["fwd_ms"])
        f2 = {"serial_fwd_ms": serial, "best": best, "best_gain_fwd_ms": serial - best["fwd_ms"],
              "default_fwd_ms": ms_fwd, "settings": rows}

    # per-kernel timing on the launch stream (instrumented replay of the same steps)
    nsteps_timed = min(2, args.steps)
    per = per_kernel(runner, dev, nsteps_timed)
    launches = sum(len(v) for v in per.values()) // nsteps_timed
    totals = {k: sum(v) for k, v in per.items()}
    dom = max(totals, key=totals.get)
    hbm, bf16, bf16_s, peak_kind = peaks()
    calls = runner.units() * nsteps_timed  # token-heads of each call, in order
    nl = len(per[dom])
    units = (calls * ((nl + len(calls) - 1) // len(calls)))[:nl] if nl != len(calls) else calls
    if dom.startswith("simt_"):
        # fp32 FFMA: 152 SMs x 128 lanes x 2 flop x max SM clock (2070 MHz)
        km = kernel_model(dom, w.dk, w.dv)
        alu_peak = 152 * 128 * 2 * 2.070e9 / 1e12
        achieved = km[1] * (sum(units) / 64) / (totals[dom] / 1e3) / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
                "frac": achieved / alu_peak, "traffic": None, "kernel": dom,
                "peak_source": "derived: fp32 FFMA lanes x max clock"}
    else:
        roof = kernel_roofline(dom, per[dom], units, w, hbm, peak_kind)
        km = kernel_model(dom, w.dk, w.dv)
        if km is not None:
            design = km[0] * sum(units) / 64 / (totals[dom] / 1e3) / 1e9
            roof["design_bytes_per_launch"] = km[0] * sum(units) / 64 / nl
            roof["design_frac"] = design / hbm

    e2e = None
    if not args.no_e2e and not varlen:
        barrier(world)
        e_ms, h2d, d2h, node = e2e_measure(runner, max(1, min(args.steps, 5)), dev)
        e_ms, _ = aggregate(e_ms, w.B * w.T, world, device=dev)  # slowest rank
        e2e = {"value": tokens / (e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "copies": "pinned host buffers, per chunk on two copy streams overlapped "
                         "with the kernels; two device input sets, so a step's uploads run "
                         "while the previous step's backward downloads its gradients",
               "steps_timed": max(1, min(args.steps, 5)),
               "host_numa_node": node}
    # the other backward of the same workload (kept products vs recomputing)
    other = None
    if not varlen:
        alt = Runner(w, dev, reuse=recompute)
        a_ms, a_ms_f = time_mode(alt, args.steps, args.warmup, dev)
        a_ms, _ = aggregate(a_ms, w.B * w.T, world, device=dev)
        a_per = per_kernel(alt, dev, nsteps_timed)
        other = {"backward": workload_config(w, world, not recompute)["backward"],
                 "ms_per_step": a_ms, "tokens_per_s": tokens / (a_ms / 1e3),
                 "frac_of_roofline": op_roofline(w, a_ms)["frac_of_roofline"],
                 "kernels_ms_per_step": {k: sum(v) / nsteps_timed for k, v in a_per.items()}}
        del alt
        torch.cuda.empty_cache()
    conv = None
    if not args.no_conv and not args.tokens and not varlen:
        conv = conv_measure(max(3, min(args.steps, 10)), args.warmup, dev, hbm, peak_kind)
    others = None
    if not args.no_others and not args.tokens and args.workload == WORKLOAD_INDEX:
        others = other_workloads(dev, max(3, min(args.steps, 10)), args.warmup)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, runner.x)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": workload_config(w, world, recompute),
            "clocks": clk.summary(),
            "e2e": e2e,
            "gpu_launches": launches * args.steps,
            "roofline": roof,
            "op_roofline": op_roofline(w, ms_step),
            "fwd": {"value": value_fwd, "unit": UNIT, "ms_per_step": ms_fwd,
                    "op_roofline": op_roofline(w, ms_fwd, "fwd")},
            "kernels_ms_per_step": {k: v / nsteps_timed for k, v in totals.items()},
            "f2_overlap": f2,
            "other_backward": other,
            "other_workloads": others,
            "cpu_baseline": cpu,
            "short_conv": conv,
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
