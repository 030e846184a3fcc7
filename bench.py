"""Benchmark of the Event-Tensor MoE megakernel on GB300.

Default workload: the Mixtral-shaped MoE layer (H 4096, 8 experts, top-2,
SwiGLU FFN 14336, bf16 weights ~N(0, 0.02), synthetic seeded inputs).  One
step is one pass over the token sweep T = 1, 2, 4, ..., 512 -- every token
count served by the same compiled kernel, the count read from device memory.
L2 is flushed before every layer call (a 256 MiB write, then a 256 MiB read,
so the call starts from a cold L2 holding clean lines only) and each call is
timed with CUDA events on the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload mixtral|fine|mixtral_block|fine_block|mixtral_chain2|
                              fine_chain2|splitk|mlp]

The *_block workloads run the fused MoE block (RMSNorm, routed experts, a
shared expert of width 2F on the fine-grained shape, residual add) over the
same sweep; they print their own line with their own metric.  The *_chain2
workloads run two such blocks (each with its own weights) chained in one
launch, and the same two blocks as two launches for comparison.

Prints ONE JSON line on rank 0.  With N > 1 (torchrun, one process per GPU)
every rank runs an independent replica of the same sweep ("replicas only":
the layer has no exchange step on one node here); value = tokens of all
ranks / the slowest rank's time.  --impl reference times the CPU oracle on
the host cores (a bounded sample per step) for the same metric.
"""
import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from moe_task_scheduling_gb300 import workloads as wl  # noqa: E402

METRIC = "MoE-layer tokens/s over the token-count sweep (us/layer per T; % of HBM roofline)"
METRIC_BLOCK = ("Fused MoE-block tokens/s over the token-count sweep (RMSNorm + routed and shared "
                "experts + residual; us/block per T; % of HBM roofline)")
# workload -> (configuration, shared-expert width; None = the plain layer)
MOE_WORKLOADS = {"mixtral": (wl.MIXTRAL, None), "fine": (wl.FINE, None),
                 "mixtral_block": (wl.MIXTRAL, 0), "fine_block": (wl.FINE, 2 * wl.FINE.F)}
METRIC_CHAIN = ("Two chained fused MoE blocks in one launch: tokens/s over the token-count sweep "
                "(us per two-block call per T; vs the same blocks as two launches)")
# workload -> (configuration, shared-expert width, layers)
CHAIN_WORKLOADS = {"mixtral_chain2": (wl.MIXTRAL, 0, 2), "fine_chain2": (wl.FINE, 2 * wl.FINE.F, 2)}
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Run before each timed call: write a buffer twice the size of L2 (every
    line of the previous call is evicted), then read another one, so the call
    starts from a cold L2 that holds clean lines only.  With the write alone
    L2 is left full of the flush buffer's dirty lines, and writing those back
    to HBM lands inside the next timed call (measured on GB300: 2.5 % of the
    Mixtral sweep's time)."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        # fp32, so the sum reads the buffer in place (an integer sum would first cast it)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.sum()
# the sources the MoE megakernel is compiled from: a committed ncu traffic
# figure stands for the kernel only while these hash to its recorded value
KERNEL_SOURCES = ["et_device.cuh", "et_gemm.cuh", "et_layout.h", "moe_kernel.cu"]


# ----------------------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def _code_only(text):
    """C++ source without its comments and with whitespace runs collapsed, so
    that a comment-only edit leaves the hash of the compiled code unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # string or character literal, copied whole
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash():
    """Hash of the megakernel's code (comments and layout excluded)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        text = open(os.path.join(ROOT, "moe_task_scheduling_gb300", "csrc", f), encoding="utf-8").read()
        h.update(_code_only(text).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch from a committed ncu summary, only if it was taken
    on the current kernel sources (same source hash)."""
    path = os.path.join(ROOT, "profiles", f"moe_megakernel_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m or not t or m.group(1) != source_hash():
        return None
    return float(t.group(1))


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def smi_index(local):
    """nvidia-smi's index of this process's GPU (CUDA_VISIBLE_DEVICES respected)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if vis.replace(",", "").isdigit():
        return int(vis.split(",")[local if local < len(vis.split(",")) else 0])
    return local


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world, device):
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- MoE workload

def moe_algorithmic_bytes(cfg, T, n_touched, Fs=None):
    """Bytes the layer must move: the expert weights it touches (gate, up, down),
    the router weight, x in and out (the block adds gamma and the shared
    expert's weights).  h, y, x_hat and split-K partials are the
    implementation's own traffic and are not counted."""
    b = (n_touched * 3 * cfg.F * cfg.H * 2 + cfg.H * cfg.E * 2 + 2 * T * cfg.H * 2
         + (cfg.E * 4 if cfg.zipf_s is not None else 0))
    if Fs is not None:
        b += cfg.H * 2 + 3 * Fs * cfg.H * 2
    return b


def moe_algorithmic_flops(cfg, T, Fs=None):
    return 2 * T * cfg.k * 3 * cfg.H * cfg.F + 2 * T * cfg.H * cfg.E + 2 * T * 3 * cfg.H * (Fs or 0)


class MoeBench:
    """The MoE layer (Fs None) or the fused block with a shared expert of width Fs."""

    def __init__(self, cfg, device, Fs=None):
        from moe_task_scheduling_gb300 import etmoe
        self.etmoe = etmoe
        etmoe.load()
        self.cfg = cfg
        self.Fs = Fs
        self.dev = device
        self.inp = wl.moe_inputs(cfg, device=device)
        self.blk = wl.block_extra_inputs(cfg, Fs, device=device) if Fs is not None else None
        if self.blk is not None:  # the skew in units of the router input's (x_hat's) logit std
            self.blk["bias"] = wl.block_router_bias(self.inp["bias"])
        T_max = cfg.T_max
        self.out = torch.empty((T_max, cfg.H), dtype=torch.bfloat16, device=device)
        self.cnt = torch.zeros((cfg.E,), dtype=torch.int32, device=device)
        nbytes = (etmoe.et_moe_workspace_bytes(T_max, cfg.H, cfg.F, cfg.E, cfg.k) if Fs is None else
                  etmoe.et_moe_block_workspace_bytes(T_max, cfg.H, cfg.F, cfg.E, cfg.k, Fs))
        self.ws = etmoe.alloc_workspace(nbytes, device=device)
        self.d_T = torch.zeros(1, dtype=torch.int32, device=device)
        self.flush = L2Flush(device)
        self.stream = torch.cuda.current_stream(device)

    def call(self, x=None, out=None, T=None):
        """One layer call; T from device memory (d_T), or the host count T."""
        i = self.inp
        tkw = dict(T=0, d_T=self.d_T) if T is None else dict(T=T, d_T=None)
        if self.blk is not None:
            b = self.blk
            self.etmoe.et_moe_block(x if x is not None else i["x"], b["gamma"], b["eps"], i["wr"],
                                    b["bias"], i["wg"], i["wu"], i["wd"], b["sg"], b["su"], b["sd"],
                                    out if out is not None else self.out, k=self.cfg.k,
                                    T_max=self.cfg.T_max, expert_counts=self.cnt,
                                    workspace=self.ws, stream=self.stream, **tkw)
            return
        self.etmoe.et_moe_layer(x if x is not None else i["x"], i["wr"], i["bias"], i["wg"], i["wu"],
                                i["wd"], out if out is not None else self.out, k=self.cfg.k,
                                T_max=self.cfg.T_max, expert_counts=self.cnt,
                                workspace=self.ws, stream=self.stream, **tkw)

    def step(self, events=None):
        """One pass over the sweep; returns per-T event pairs if asked."""
        pairs = []
        for T in self.cfg.T_sweep:
            self.flush()
            self.d_T.fill_(T)
            if events:
                s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s.record(self.stream)
                self.call()
                e.record(self.stream)
                pairs.append((T, s, e))
            else:
                self.call()
        return pairs

    def touched(self):
        out = {}
        for T in self.cfg.T_sweep:
            self.d_T.fill_(T)
            self.call()
            torch.cuda.synchronize()
            out[T] = int((self.cnt > 0).sum().item())
        return out

    def e2e(self, steps):
        """Through the public call with host buffers: per T, pinned x -> device,
        the layer (the token count passed from the host, as a caller holding host
        buffers would), out -> pinned host; every copy is inside the timed region.
        As a serving loop would, the copies run on a second stream with double
        buffers, so the next call's upload and the last call's download overlap
        the current layer.  The host outputs of the last step are then checked
        bit for bit against a plain call per T."""
        import torch
        cfg = self.cfg
        dev = self.inp["x"].device
        Ts = list(cfg.T_sweep)
        xh = {T: self.inp["x"][:T].cpu().pin_memory() for T in Ts}
        oh = {T: torch.empty((T, cfg.H), dtype=torch.bfloat16).pin_memory() for T in Ts}
        xd = [torch.empty_like(self.inp["x"]) for _ in range(2)]
        od = [torch.empty_like(self.out) for _ in range(2)]
        ms, cs = self.stream, torch.cuda.Stream(device=dev)
        h2d = sum(T * cfg.H * 2 for T in Ts)
        total = 0.0
        for _ in range(steps):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(ms)
            cs.wait_event(s)
            up, done, down = [None] * len(Ts), [None] * len(Ts), [None] * len(Ts)

            def upload(i):
                with torch.cuda.stream(cs):
                    if i >= 2:
                        cs.wait_event(done[i - 2])  # layer i - 2 has read this x buffer
                    xd[i % 2][:Ts[i]].copy_(xh[Ts[i]], non_blocking=True)
                    up[i] = torch.cuda.Event()
                    up[i].record(cs)

            upload(0)
            for i, T in enumerate(Ts):
                if i + 1 < len(Ts):
                    upload(i + 1)
                ms.wait_event(up[i])
                if i >= 2:
                    ms.wait_event(down[i - 2])  # this out buffer has been read back
                self.call(x=xd[i % 2], out=od[i % 2], T=T)
                done[i] = torch.cuda.Event()
                done[i].record(ms)
                with torch.cuda.stream(cs):
                    cs.wait_event(done[i])
                    oh[T].copy_(od[i % 2][:T], non_blocking=True)
                    down[i] = torch.cuda.Event()
                    down[i].record(cs)
            ms.wait_event(down[-1])
            e.record(ms)
            e.synchronize()
            total += s.elapsed_time(e) / 1e3
        for T in Ts:  # the pipelined results are the plain call's
            self.call(x=self.inp["x"], out=od[0], T=T)
            torch.cuda.synchronize()
            if not torch.equal(od[0][:T].cpu(), oh[T]):
                raise RuntimeError(f"e2e: host output at T={T} differs from a plain call")
        return total, h2d, h2d


class DenseBench:
    """Split-K GEMM (config 2) or the MLP chain (config 3) over their M / B sweeps."""

    def __init__(self, kind, device):
        from moe_task_scheduling_gb300 import etmoe
        self.etmoe = etmoe
        etmoe.load()
        self.kind = kind
        self.dev = device
        self.stream = torch.cuda.current_stream(device)
        self.flush = L2Flush(device)
        self.d_n = torch.zeros(1, dtype=torch.int32, device=device)
        if kind == "splitk":
            c = self.cfg = wl.SPLITK
            self.inp = wl.splitk_inputs(c, device=device)
            self.sweep = c.M_sweep
            self.out = torch.empty((c.M_max, c.N), dtype=torch.bfloat16, device=device)
            self.ws = etmoe.alloc_workspace(etmoe.et_splitk_workspace_bytes(c.M_max, c.N, c.K,
                                                                            c.split), device=device)
        else:
            c = self.cfg = wl.MLP
            self.inp = wl.mlp_inputs(c, device=device)
            self.sweep = c.B_sweep
            self.out = torch.empty((c.B_max, c.H), dtype=torch.bfloat16, device=device)
            self.ws = etmoe.alloc_workspace(etmoe.et_mlp_workspace_bytes(c.B_max, c.H, c.F),
                                            device=device)

    def call(self, clc=False):
        c, i = self.cfg, self.inp
        if self.kind == "splitk":
            f = self.etmoe.et_splitk_gemm_clc if clc else self.etmoe.et_splitk_gemm
            f(i["X"], i["Wt"], self.out, split=c.split, M=0, d_M=self.d_n, M_max=c.M_max,
              workspace=self.ws, stream=self.stream)
        else:
            self.etmoe.et_mlp_chain(i["x"], i["gamma"], c.eps, i["wg"], i["wu"], i["wd"], self.out,
                                    B=0, d_B=self.d_n, B_max=c.B_max, workspace=self.ws,
                                    stream=self.stream)

    def bytes_flops(self, n):
        c = self.cfg
        if self.kind == "splitk":
            return c.N * c.K * 2 + n * c.K * 2 + n * c.N * 2, 2 * n * c.N * c.K
        return 3 * c.H * c.F * 2 + 2 * n * c.H * 2 + c.H * 2, 6 * n * c.H * c.F

    def measure(self, steps, warmup):
        """Median CUDA-event time per size; the split-K GEMM also through the
        Cluster Launch Control work queue (us_clc)."""
        res = []
        variants = [False, True] if self.kind == "splitk" else [False]
        for n in self.sweep:
            self.d_n.fill_(n)
            times = {}
            for clc in variants:
                for _ in range(warmup):
                    self.flush()
                    self.call(clc)
                ts = []
                for _ in range(steps):
                    self.flush()
                    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    s.record(self.stream)
                    self.call(clc)
                    e.record(self.stream)
                    ts.append((s, e))
                torch.cuda.synchronize()
                times[clc] = statistics.median(s.elapsed_time(e) / 1e3 for s, e in ts)
            code, detail = self.etmoe.et_status(self.ws)
            assert code == 0, f"device status {code} ({detail})"
            t = times[False]
            by, fl = self.bytes_flops(n)
            pk = peaks()
            r = {"n": n, "us": round(t * 1e6, 2), "hbm_frac": round(by / t / 1e9 / pk["hbm_gbs"], 4),
                 "tensor_frac": round(fl / t / 1e12 / pk["bf16_tflops"], 4)}
            if True in times:
                r["us_clc"] = round(times[True] * 1e6, 2)
                r["hbm_frac_clc"] = round(by / times[True] / 1e9 / pk["hbm_gbs"], 4)
            res.append(r)
        return res


class ChainBench:
    """n fused blocks chained in one launch (et_moe_chain), and the same blocks
    as n launches (et_moe_block each) on the previous block's output."""

    def __init__(self, cfg, device, Fs, n):
        import dataclasses
        from moe_task_scheduling_gb300 import etmoe
        self.etmoe = etmoe
        etmoe.load()
        self.cfg, self.Fs, self.n, self.dev = cfg, Fs, n, device
        self.inp, self.blk = [], []
        for j in range(n):
            c = dataclasses.replace(cfg, index=cfg.index + 100 * j)
            self.inp.append(wl.moe_inputs(c, device=device))
            self.blk.append(wl.block_extra_inputs(c, Fs, device=device))
            self.blk[-1]["bias"] = wl.block_router_bias(self.inp[-1]["bias"])
        T_max = cfg.T_max
        self.outs = [torch.empty((T_max, cfg.H), dtype=torch.bfloat16, device=device)
                     for _ in range(n)]
        self.descs = []
        for j in range(n):
            i, b = self.inp[j], self.blk[j]
            self.descs.append(etmoe.layer_desc(i["wr"], b["bias"], i["wg"], i["wu"], i["wd"],
                                               self.outs[j], gamma=b["gamma"], eps=b["eps"],
                                               ws_gate=b["sg"], ws_up=b["su"], ws_down=b["sd"]))
        self.ws = etmoe.alloc_workspace(etmoe.et_moe_chain_workspace_bytes(
            self.descs, T_max, cfg.H, cfg.F, cfg.E, cfg.k), device=device)
        self.ws1 = [etmoe.alloc_workspace(etmoe.et_moe_block_workspace_bytes(
            T_max, cfg.H, cfg.F, cfg.E, cfg.k, Fs), device=device) for _ in range(n)]
        self.d_T = torch.zeros(1, dtype=torch.int32, device=device)
        self.flush = L2Flush(device)
        self.stream = torch.cuda.current_stream(device)

    def chain(self, x=None):
        c = self.cfg
        self.etmoe.et_moe_chain(self.descs, self.inp[0]["x"] if x is None else x, H=c.H, F=c.F,
                                E=c.E, k=c.k, T=0, d_T=self.d_T, T_max=c.T_max, workspace=self.ws,
                                stream=self.stream)

    def separate(self):
        c = self.cfg
        x = self.inp[0]["x"]
        for j in range(self.n):
            i, b = self.inp[j], self.blk[j]
            self.etmoe.et_moe_block(x, b["gamma"], b["eps"], i["wr"], b["bias"], i["wg"], i["wu"],
                                    i["wd"], b["sg"], b["su"], b["sd"], self.outs[j], k=c.k, T=0,
                                    d_T=self.d_T, T_max=c.T_max, workspace=self.ws1[j],
                                    stream=self.stream)
            x = self.outs[j]

    def timed(self, fn, T):
        self.flush()
        self.d_T.fill_(T)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(self.stream)
        fn()
        e.record(self.stream)
        return s, e


def run_chain(args, world, rank, local):
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    cfg, Fs, n = CHAIN_WORKLOADS[args.workload]
    b = ChainBench(cfg, device, Fs, n)
    for _ in range(args.warmup):
        for T in cfg.T_sweep:
            b.timed(b.chain, T)
            b.timed(b.separate, T)
    torch.cuda.synchronize()
    gpu_index = local
    barrier(world)
    torch.cuda.synchronize()
    pairs = {T: ([], []) for T in cfg.T_sweep}
    wall0 = time.perf_counter()
    with ClockSampler(gpu_index) as clk:
        for _ in range(args.steps):
            for T in cfg.T_sweep:
                pairs[T][0].append(b.timed(b.chain, T))
                pairs[T][1].append(b.timed(b.separate, T))
        torch.cuda.synchronize()
        barrier(world)
        wall = time.perf_counter() - wall0
    per_T = {T: ([s.elapsed_time(e) / 1e3 for s, e in c], [s.elapsed_time(e) / 1e3 for s, e in d])
             for T, (c, d) in pairs.items()}
    code, detail = b.etmoe.et_status(b.ws)
    assert code == 0, f"device status {code} ({detail})"
    t_chain = sum(sum(c) for c, _ in per_T.values())
    t_sep = sum(sum(d) for _, d in per_T.values())
    tokens = args.steps * sum(cfg.T_sweep)
    t_max = max_over_ranks(t_chain, world, device)
    tok_all = sum_over_ranks(tokens, world, device)
    if rank != 0:
        return None
    pk = peaks()
    sweep, bytes_total = [], 0.0
    for T in cfg.T_sweep:
        c, d = per_T[T]
        tc, td = statistics.median(c), statistics.median(d)
        b.d_T.fill_(T)
        cnts = []
        for j in range(n):  # experts each block touched (from its own run)
            cnt = torch.zeros(cfg.E, dtype=torch.int32, device=device)
            i, bb = b.inp[j], b.blk[j]
            x = b.inp[0]["x"] if j == 0 else b.outs[j - 1]
            b.etmoe.et_moe_block(x, bb["gamma"], bb["eps"], i["wr"], bb["bias"], i["wg"], i["wu"],
                                 i["wd"], bb["sg"], bb["su"], bb["sd"], b.outs[j], k=cfg.k, T=0,
                                 d_T=b.d_T, T_max=cfg.T_max, expert_counts=cnt, workspace=b.ws1[j])
            cnts.append(int((cnt > 0).sum().item()))
        by = sum(moe_algorithmic_bytes(cfg, T, t, Fs) for t in cnts)
        bytes_total += by * len(c)
        sweep.append({"T": T, "us_chain": round(tc * 1e6, 2), "us_two_launches": round(td * 1e6, 2),
                      "saved_us": round((td - tc) * 1e6, 2), "experts_touched": cnts,
                      "hbm_frac": round(by / tc / 1e9 / pk["hbm_gbs"], 4)})
    achieved = bytes_total / t_chain / 1e9
    return {
        "metric": METRIC_CHAIN,
        "value": round(tok_all / t_max, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_max / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) bf16 weights and activations)",
        "config": {"workload": f"{cfg.name}: {n} fused MoE blocks (Fs={Fs}) chained, T sweep "
                               f"{list(cfg.T_sweep)}",
                   "H": cfg.H, "F": cfg.F, "E": cfg.E, "k": cfg.k, "Fs": Fs, "layers": n,
                   "l2": "flushed before every call (chain, or the pair): 256 MiB write, then 256 MiB read",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "two_launches": {"value": round(tokens / t_sep, 1), "unit": "tokens/s",
                         "kind": "the same blocks, one et_moe_block launch each"},
        "sweep": sweep,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": None,
                     "peak_source": pk["source"] + " (hbm copy, burst)",
                     "kernel": "moe_megakernel"},
        "gpu_launches": args.steps * len(cfg.T_sweep),
        "wall_s_timed": round(wall, 3),
        "clocks": clk.summary(),
    }


WARMUP_CHILD = r"""
import hashlib, json, os, sys, time
sys.path.insert(0, os.environ["ET_ROOT"])
import torch
from moe_task_scheduling_gb300 import workloads as wl
cfg = wl.MIXTRAL
Ts = [int(t) for t in os.environ.get("ET_TS", "").split(",") if t] or list(cfg.T_sweep)
dev = torch.device("cuda")
torch.zeros(1, device=dev)
inp = wl.moe_inputs(cfg, device=dev)
out = torch.empty((cfg.T_max, cfg.H), dtype=torch.bfloat16, device=dev)
d_T = torch.full((1,), Ts[0], dtype=torch.int32, device=dev)
torch.cuda.synchronize()
def now():
    torch.cuda.synchronize()
    return time.perf_counter()
t0 = now()
from moe_task_scheduling_gb300 import etmoe
etmoe.load(os.environ.get("ET_LIB") or None)
t_load = now() - t0
ws = etmoe.alloc_workspace(etmoe.et_moe_workspace_bytes(cfg.T_max, cfg.H, cfg.F, cfg.E, cfg.k))
torch.cuda.synchronize()
def call():
    etmoe.et_moe_layer(inp["x"], inp["wr"], inp["bias"], inp["wg"], inp["wu"], inp["wd"], out,
                       k=cfg.k, T=0, d_T=d_T, T_max=cfg.T_max, workspace=ws)
t0 = now(); call(); t_first = now() - t0
t0 = now(); call(); t_second = now() - t0
first_T, steady_T, sha = {}, {}, {}
for T in Ts[1:]:
    d_T.fill_(T)
    t0 = now(); call(); first_T[T] = now() - t0
for T in Ts:
    d_T.fill_(T)
    ts = []
    for _ in range(3):
        t0 = now(); call(); ts.append(now() - t0)
    steady_T[T] = sorted(ts)[1]
    sha[T] = hashlib.sha256(out[:T].cpu().view(torch.int16).numpy().tobytes()).hexdigest()[:16]
assert etmoe.et_status(ws) == (0, 0)
print(json.dumps({"load_s": t_load, "first_s": t_first, "second_s": t_second,
                  "first_T": first_T, "steady_T": steady_T, "out_sha": sha}))
"""

# token counts given their own specialised build in the warm-up comparison
SPECIALISED_TS = (1, 512)


def _warmup_child(env_extra):
    env = dict(os.environ, ET_ROOT=ROOT, **env_extra)
    r = subprocess.run([sys.executable, "-c", WARMUP_CHILD], capture_output=True, text=True,
                       env=env, timeout=600)
    if r.returncode != 0:
        raise RuntimeError("warm-up child failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_warmup(args):
    """Warm-up cost of one kernel for every token count against builds
    specialised per batch size.  Measured: the library's full build (timed
    into a scratch directory); then, in fresh processes, the first layer call
    (library load, kernel attributes, tensor maps, module load, launch) and the
    first call at each new token count against the steady state, host wall
    clock with a device synchronise on both sides.  The alternative is built
    for real at a few token counts: the library with the megakernel compiled
    for one constant T (-DET_FIXED_T), its build timed, its first call timed
    in a fresh process, and its output checked bit for bit against the
    general build at that T."""
    import tempfile
    from moe_task_scheduling_gb300 import build as B
    spec = []
    with tempfile.TemporaryDirectory() as d:
        t0 = time.perf_counter()
        B.build(force=True, out_dir=d)
        t_build = time.perf_counter() - t0
        for T in SPECIALISED_TS:
            sd = os.path.join(d, f"T{T}")
            t0 = time.perf_counter()
            lib = B.build(force=True, out_dir=sd, defines=(f"ET_FIXED_T={T}",))
            t_b = time.perf_counter() - t0
            c = _warmup_child({"ET_LIB": lib, "ET_TS": str(T)})
            spec.append({"T": T, "build_s": round(t_b, 2),
                         "first_call_ms": round(c["first_s"] * 1e3, 3),
                         "steady_ms": round(c["steady_T"][str(T)] * 1e3, 3),
                         "out_sha": c["out_sha"][str(T)]})
    c = _warmup_child({})
    for r in spec:
        r["same_output_as_general_build"] = r.pop("out_sha") == c["out_sha"][str(r["T"])]
    sweep = [{"T": int(T), "first_call_ms": round(c["first_T"].get(T, c["first_s"]) * 1e3, 3),
              "steady_ms": round(c["steady_T"][T] * 1e3, 3)}
             for T in sorted(c["steady_T"], key=int)]
    n_sizes = len(wl.MIXTRAL.T_sweep)
    per_build = statistics.mean(r["build_s"] for r in spec)
    return {
        "metric": "MoE layer warm-up: first call in a fresh process, one compiled kernel for "
                  "every token count (ms)",
        "value": round(c["first_s"] * 1e3, 3), "unit": "ms", "higher_is_better": False,
        "n_gpus": 1, "data": "synthetic (seeded N(0,0.02) bf16 weights)",
        "config": {"workload": "mixtral MoE layer, T = 1 first, then each T of the sweep",
                   "clock": "host wall clock, device synchronised before and after"},
        "library_load_ms": round(c["load_s"] * 1e3, 3),
        "second_call_ms": round(c["second_s"] * 1e3, 3),
        "sweep": sweep,
        "build": {"full_library_s": round(t_build, 2),
                  "specialised_builds": spec,
                  "per_size_builds_for_the_sweep_s": round(n_sizes * per_build, 1),
                  "note": f"one build serves all {n_sizes} token counts of the sweep; builds "
                          f"specialised per size were built and timed at T = "
                          f"{list(SPECIALISED_TS)}, and {n_sizes} of them take {n_sizes} x "
                          f"their mean build time"},
    }


def run_dense(args, local):
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    b = DenseBench(args.workload, device)
    res = b.measure(args.steps, args.warmup)
    return {"workload": args.workload, "sweep": res,
            "note": "per-call CUDA-event median, L2 flushed before each call; not the headline line"}


def run_ours(args, world, rank, local):
    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU for --impl ours"
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    cfg, Fs = MOE_WORKLOADS[args.workload]
    b = MoeBench(cfg, device, Fs)
    touched = b.touched()
    for _ in range(args.warmup):
        b.step()
    torch.cuda.synchronize()
    gpu_index = smi_index(local)
    barrier(world)
    torch.cuda.synchronize()
    per_T = {T: [] for T in cfg.T_sweep}
    wall0 = time.perf_counter()
    with ClockSampler(gpu_index) as clk:
        all_pairs = [b.step(events=True) for _ in range(args.steps)]
        torch.cuda.synchronize()
        barrier(world)
        wall = time.perf_counter() - wall0
        for pairs in all_pairs:
            for T, s, e in pairs:
                per_T[T].append(s.elapsed_time(e) / 1e3)
        e2e_time, h2d, d2h = b.e2e(args.steps)
    kernel_time = sum(sum(v) for v in per_T.values())  # seconds, summed over steps
    tokens = args.steps * sum(cfg.T_sweep)
    t_max = max_over_ranks(kernel_time, world, device)
    tok_all = sum_over_ranks(tokens, world, device)
    e2e_max = max_over_ranks(e2e_time, world, device)
    if rank != 0:
        return None
    pk = peaks()
    sweep = []
    bytes_total = 0.0
    for T in cfg.T_sweep:
        t = statistics.median(per_T[T])
        by = moe_algorithmic_bytes(cfg, T, touched[T], Fs)
        bytes_total += by * len(per_T[T])
        sweep.append({"T": T, "us_per_layer": round(t * 1e6, 2), "us_min": round(min(per_T[T]) * 1e6, 2),
                      "tokens_per_s": round(T / t, 1), "experts_touched": touched[T],
                      "hbm_frac": round(by / t / 1e9 / pk["hbm_gbs"], 4),
                      "tensor_frac": round(moe_algorithmic_flops(cfg, T, Fs) / t / 1e12 /
                                           pk["bf16_tflops"], 4)})
    achieved = bytes_total / kernel_time / 1e9
    traffic = profiled_traffic(args.workload)
    n_launch = args.steps * len(cfg.T_sweep)
    what = "MoE layer" if Fs is None else (f"fused MoE block (shared expert Fs={Fs})" if Fs else
                                           "fused MoE block (no shared expert)")
    line = {
        "metric": METRIC if Fs is None else METRIC_BLOCK,
        "value": round(tok_all / t_max, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_max / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) bf16 weights and activations)",
        "config": {"workload": f"{cfg.name} {what}, T sweep {list(cfg.T_sweep)}",
                   "H": cfg.H, "F": cfg.F, "E": cfg.E, "k": cfg.k,
                   **({} if Fs is None else {"Fs": Fs, "eps": 1e-5}),
                   "l2": "flushed before every layer call: 256 MiB write, then 256 MiB read (cold, clean L2)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "symbolic_T": "one compiled kernel, T read from device memory"},
        "sweep": sweep,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                     "traffic": traffic, "peak_source": pk["source"] + " (hbm copy, burst)",
                     "kernel": "moe_megakernel"},
        "e2e": {"value": round(tok_all / e2e_max, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": n_launch,
        "wall_s_timed": round(wall, 3),
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_per_op:
        line["per_op_baseline"] = per_op_baseline(b, cfg)
        # torch._grouped_mm is not run: on the GPU machine's torch build it failed with an
        # unspecified launch failure on this GPU
        line["per_op_grouped_baseline"] = {
            "unavailable": "torch._grouped_mm failed with an unspecified launch failure on this "
                           "GPU (GPU box torch build); not run"}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(b, cfg, args)
    if world == 1 and args.workload == "mixtral" and not args.no_extra:
        del b
        torch.cuda.empty_cache()
        line.update(secondary_sweeps(args, device))
    return line


def moe_sweep_record(cfg, Fs, device, steps, warmup):
    """A MoE workload's own sweep as a compact record: tokens/s over the sweep,
    per-T microseconds and roofline fractions, the sweep's HBM roofline."""
    b = MoeBench(cfg, device, Fs)
    touched = b.touched()
    for _ in range(warmup):
        b.step()
    torch.cuda.synchronize()
    per_T = {T: [] for T in cfg.T_sweep}
    with ClockSampler(smi_index(device.index or 0)) as clk:
        all_pairs = [b.step(events=True) for _ in range(steps)]
        torch.cuda.synchronize()
    for pairs in all_pairs:
        for T, s0, e0 in pairs:
            per_T[T].append(s0.elapsed_time(e0) / 1e3)
    code, detail = b.etmoe.et_status(b.ws)
    assert code == 0, f"device status {code} ({detail})"
    pk = peaks()
    total = sum(sum(v) for v in per_T.values())
    bytes_total, sweep = 0.0, []
    for T in cfg.T_sweep:
        t = statistics.median(per_T[T])
        by = moe_algorithmic_bytes(cfg, T, touched[T], Fs)
        bytes_total += by * len(per_T[T])
        sweep.append({"T": T, "us": round(t * 1e6, 2), "experts_touched": touched[T],
                      "hbm_frac": round(by / t / 1e9 / pk["hbm_gbs"], 4),
                      "tensor_frac": round(moe_algorithmic_flops(cfg, T, Fs) / t / 1e12 /
                                           pk["bf16_tflops"], 4)})
    achieved = bytes_total / total / 1e9
    rec = {"value": round(steps * sum(cfg.T_sweep) / total, 1), "unit": "tokens/s",
           "workload": f"{cfg.name} H={cfg.H} F={cfg.F} E={cfg.E} k={cfg.k}" +
                       ("" if Fs is None else f", fused block Fs={Fs}"),
           "sweep": sweep,
           "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                        "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                        "peak_source": pk["source"] + " (hbm copy, burst)",
                        "kernel": "moe_megakernel"},
           "gpu_launches": steps * len(cfg.T_sweep), "clocks": clk.summary()}
    del b
    torch.cuda.empty_cache()
    return rec


def dense_sweep_record(kind, device, steps, warmup):
    b = DenseBench(kind, device)
    with ClockSampler(smi_index(device.index or 0)) as clk:
        res = b.measure(steps, warmup)
    variants = 2 if kind == "splitk" else 1
    kernel = "splitk_kernel" if kind == "splitk" else "mlp_chain_kernel"
    rec = {"workload": (f"split-K GEMM Y[M,{b.cfg.N}] = X[M,{b.cfg.K}] W, split {b.cfg.split}"
                        if kind == "splitk" else
                        f"MLP chain H={b.cfg.H} F={b.cfg.F} (RMSNorm, gate/up, SiLU*mul, down)"),
           "kernel": kernel, "sweep": res,
           "gpu_launches": variants * steps * len(res), "clocks": clk.summary()}
    del b
    torch.cuda.empty_cache()
    return rec


def secondary_sweeps(args, device):
    """The other configurations, measured in the same run as the headline:
    the fine-grained skewed layer, the split-K GEMM, the MLP chain, the fused
    Mixtral-shaped block, and the warm-up record."""
    out = {}
    steps, warmup = args.steps, args.warmup
    out["fine"] = moe_sweep_record(wl.FINE, None, device, steps, warmup)
    out["mixtral_block"] = moe_sweep_record(wl.MIXTRAL, 0, device, steps, warmup)
    out["splitk"] = dense_sweep_record("splitk", device, steps, warmup)
    out["mlp"] = dense_sweep_record("mlp", device, steps, warmup)
    if not args.no_warmup_record:
        try:
            out["warmup"] = run_warmup(args)
        except Exception as e:  # a failed build or child is reported, not fatal
            out["warmup"] = {"unavailable": f"{type(e).__name__}: {str(e)[-300:]}"}
    return out


def run_single(args, local):
    """One layer call at token count T after `warmup` identical calls (L2
    flushed before each): the launch an ncu capture selects with -s/-c."""
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    cfg, Fs = MOE_WORKLOADS[args.workload]
    b = MoeBench(cfg, device, Fs)
    b.d_T.fill_(args.single)
    for _ in range(args.warmup + 1):
        b.flush()
        b.call()
    torch.cuda.synchronize()
    code, detail = b.etmoe.et_status(b.ws)
    return {"single": args.single, "workload": args.workload, "launches": args.warmup + 1,
            "status": [code, detail]}


TASK_NAMES = {1: "router", 2: "scan", 3: "permute", 4: "gateup", 5: "down", 6: "combine",
              7: "norm", 9: "shared_gateup", 10: "shared_down"}


def run_trace(args, local):
    """One traced layer call at token count T (after `warmup` untraced calls,
    L2 flushed before each): the kernel's own per-task records (et_opts.trace)
    summarised per task type and role, front-end phase marks, and the
    untraced CUDA-event time of the same call.  Times are us from the first
    CTA's start."""
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    cfg, Fs = MOE_WORKLOADS[args.workload]
    if Fs is not None:
        raise SystemExit("--trace covers the plain MoE layer workloads")
    b = MoeBench(cfg, device, Fs)
    T = args.trace
    b.d_T.fill_(T)
    for _ in range(args.warmup):
        b.flush()
        b.call()
    ts = []
    for _ in range(5):
        b.flush()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(b.stream)
        b.call()
        e.record(b.stream)
        e.synchronize()
        ts.append(s.elapsed_time(e) * 1e3)
    buf = b.etmoe.alloc_trace(200000, device=device)
    b.flush()
    i = b.inp
    b.etmoe.et_moe_layer(i["x"], i["wr"], i["bias"], i["wg"], i["wu"], i["wd"], b.out, k=cfg.k,
                         T=0, d_T=b.d_T, T_max=cfg.T_max, expert_counts=b.cnt, workspace=b.ws,
                         stream=b.stream, trace=buf)
    torch.cuda.synchronize()
    code, detail = b.etmoe.et_status(b.ws)
    assert code == 0, f"device status {code} ({detail})"
    recs = b.etmoe.read_trace(buf)
    t0 = min(r[5] for r in recs if r[1] == 2)

    def us(t):
        return round((t - t0) / 1e3, 2)

    res = {"trace": T, "workload": args.workload, "us_event": round(statistics.median(ts), 2),
           "experts_touched": int((b.cnt > 0).sum().item()), "records": len(recs)}
    setup = sorted(r[6] for r in recs if r[1] == 2)
    ex = [r for r in recs if r[1] == 3]
    res["cta_setup_end"] = [us(setup[0]), us(setup[len(setup) // 2]), us(setup[-1])]
    res["cta_exit"] = [us(min(r[5] for r in ex)), us(max(r[6] for r in ex))]
    for role, name in ((0, "producer"), (1, "workers")):
        d = {}
        for ty in sorted({r[0] for r in recs if r[1] == role}):
            rr = [r for r in recs if r[1] == role and r[0] == ty]
            dur = sorted((r[6] - r[5]) / 1e3 for r in rr)
            d[TASK_NAMES.get(ty, str(ty))] = {
                "n": len(rr), "first_begin": us(min(r[5] for r in rr)),
                "last_end": us(max(r[6] for r in rr)), "dur_median": round(dur[len(dur) // 2], 2),
                "dur_max": round(dur[-1], 2)}
        res[name] = d
    phases = {}
    for r in recs:
        if r[1] == 4:
            ph = phases.setdefault(r[0] - 16, [r[5], r[6], 0])
            ph[0], ph[1], ph[2] = min(ph[0], r[5]), max(ph[1], r[6]), ph[2] + 1
    res["front_end_phases"] = {str(k): [us(v[0]), us(v[1]), v[2]] for k, v in sorted(phases.items())}
    return res


def per_op_layer(inp, cfg, T, blk=None):
    """The MoE layer as a sequence of plain PyTorch ops (one launch each, no
    Triton), with a host sync for the per-expert counts: the same-GPU per-op
    baseline.  Router in fp32, expert GEMMs in bf16 (cuBLAS).  With `blk` the
    fused block: RMSNorm first, the shared expert and the residual after."""
    x0 = inp["x"][:T]
    x = x0
    if blk is not None:
        xf = x0.float()
        x = (xf * torch.rsqrt(xf.square().mean(-1, keepdim=True) + blk["eps"]) *
             blk["gamma"].float()).to(torch.bfloat16)
    logits = x.float() @ inp["wr"].float()
    bias = inp["bias"] if blk is None else blk["bias"]
    if bias is not None:
        logits = logits + bias
    w, idx = torch.topk(torch.softmax(logits, dim=-1), cfg.k, dim=-1)
    w = (w / w.sum(dim=-1, keepdim=True)).reshape(-1)
    flat = idx.reshape(-1)
    order = torch.argsort(flat, stable=True)
    counts = torch.bincount(flat, minlength=cfg.E).tolist()  # host sync
    out = torch.zeros((T, cfg.H), dtype=torch.float32, device=x.device)
    start = 0
    for e, c in enumerate(counts):
        if c == 0:
            continue
        rows = order[start:start + c]
        start += c
        tok = rows // cfg.k
        xe = x[tok]
        h = torch.nn.functional.silu(xe @ inp["wg"][e].T) * (xe @ inp["wu"][e].T)
        y = h @ inp["wd"][e].T
        out.index_add_(0, tok, y.float() * w[rows, None])
    if blk is not None:
        out += x0.float()
        if blk["sg"] is not None:
            hs = torch.nn.functional.silu(x @ blk["sg"].T) * (x @ blk["su"].T)
            out += (hs @ blk["sd"].T).float()
    return out.to(torch.bfloat16), sum(1 for c in counts if c)


def count_launches(fn):
    """GPU work items one call of fn enqueues, counted by the PyTorch profiler:
    kernels, and the memory copies / fills issued as separate operations."""
    from torch.profiler import ProfilerActivity, profile
    try:
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            fn()
            torch.cuda.synchronize()
    except Exception as e:  # the profiler could not start (e.g. already in use)
        return {"unavailable": f"torch.profiler: {type(e).__name__}"}
    kern = copies = 0
    for ev in prof.events():
        if str(getattr(ev, "device_type", "")).endswith("CUDA"):
            name = ev.name.lower()
            if name.startswith(("memcpy", "memset")):
                copies += 1
            else:
                kern += 1
    return {"kernels": kern, "copies": copies}


def per_op_baseline(b, cfg, reps=3):
    """Median CUDA-event time per T of per_op_layer over the same sweep (L2
    flushed before each call, host sync included), as tokens/s."""
    per_T, launches = {}, {}
    for T in cfg.T_sweep:
        ts = []
        for i in range(reps + 1):
            b.flush()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(b.stream)
            _, touched = per_op_layer(b.inp, cfg, T, b.blk)
            e.record(b.stream)
            e.synchronize()
            if i:
                ts.append(s.elapsed_time(e) / 1e3)
        per_T[T] = statistics.median(ts)
    # counted after every timing (the profiler slows what runs after it starts),
    # with one uncounted pass first (its first session records nothing)
    count_launches(lambda: per_op_layer(b.inp, cfg, cfg.T_sweep[0], b.blk))
    for T in cfg.T_sweep:
        launches[T] = count_launches(lambda: per_op_layer(b.inp, cfg, T, b.blk))
    tot = sum(per_T.values())
    return {"value": round(sum(cfg.T_sweep) / tot, 1), "unit": "tokens/s",
            "kind": "same-GPU per-op PyTorch (" + ("RMSNorm, " if b.blk is not None else "") +
                    "router matmul/softmax/topk, stable argsort, bincount host sync, per-expert "
                    "cuBLAS GEMMs, index_add_" +
                    (", shared expert, residual" if b.blk is not None else "") + ")",
            "us_per_layer": {str(T): round(t * 1e6, 1) for T, t in per_T.items()},
            "launches_per_layer": {str(T): n for T, n in launches.items()}}


def cpu_baseline(b, cfg, args):
    """The oracle, as it stands, on the host cores over a bounded sample of the
    same workload (the first `n` tokens of the sweep's largest batch)."""
    import oracle
    n = args.cpu_tokens
    hb = {k: (wl.bits(v) if v is not None and v.dtype == torch.bfloat16 else
              (None if v is None else v.detach().cpu().numpy())) for k, v in b.inp.items()}
    threads = oracle.default_threads()
    run = oracle_call(oracle, hb, block_bits(b.blk), cfg, n, threads)
    t0 = time.perf_counter()
    run()
    dt = time.perf_counter() - t0
    what = "layer" if b.blk is None else "block"
    return {"value": round(n / dt, 3), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} tokens of the {cfg.name} {what} (all routing + outputs), one call, "
                      f"{dt:.1f} s"}


def block_bits(blk):
    if blk is None:
        return None
    return {k: (wl.bits(v) if isinstance(v, torch.Tensor) and v.dtype == torch.bfloat16 else
                (v.detach().cpu().numpy() if isinstance(v, torch.Tensor) else v))
            for k, v in blk.items()}


def oracle_call(oracle, hb, bb, cfg, n, threads):
    """The oracle over the first n tokens: the layer, or the block when bb is given."""
    if bb is None:
        return lambda: oracle.moe_layer(hb["x"][:n], hb["wr"], hb["bias"], hb["wg"], hb["wu"],
                                        hb["wd"], k=cfg.k, nthreads=threads)
    return lambda: oracle.moe_block(hb["x"][:n], bb["gamma"], bb["eps"], hb["wr"], bb["bias"],
                                    hb["wg"], hb["wu"], hb["wd"], bb["sg"], bb["su"], bb["sd"],
                                    k=cfg.k, nthreads=threads)


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, timed on the host cores, one bounded
    sample (args.ref_tokens tokens of the same layer) per step."""
    if rank != 0:
        return None
    import oracle
    if args.workload not in MOE_WORKLOADS:
        return {"impl": "reference", "unavailable": "the reference arm covers the MoE workloads"}
    cfg, Fs = MOE_WORKLOADS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = wl.moe_inputs(cfg, device=dev)
    hb = {k: (wl.bits(v) if v is not None and v.dtype == torch.bfloat16 else
              (None if v is None else v.detach().cpu().numpy())) for k, v in inp.items()}
    bb = None
    if Fs is not None:
        blk = wl.block_extra_inputs(cfg, Fs, device=dev)
        blk["bias"] = wl.block_router_bias(inp["bias"])
        bb = block_bits(blk)
    del inp
    n = args.ref_tokens
    threads = oracle.default_threads()
    one = oracle_call(oracle, hb, bb, cfg, n, threads)
    what = "MoE layer" if Fs is None else f"fused MoE block (Fs={Fs})"

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = time.perf_counter() - t0
    v = round(args.steps * n / dt, 3)
    return {
        "metric": METRIC if Fs is None else METRIC_BLOCK, "value": v, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,0.02) bf16 weights and activations)", "impl": "reference",
        "config": {"workload": f"{cfg.name} {what}, T sweep {list(cfg.T_sweep)}",
                   "H": cfg.H, "F": cfg.F, "E": cfg.E, "k": cfg.k,
                   "sample_per_step": f"{n} tokens"},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n} tokens of the {cfg.name} {what} per step"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(MOE_WORKLOADS) + list(CHAIN_WORKLOADS) +
                    ["splitk", "mlp", "warmup"], default="mixtral")
    ap.add_argument("--cpu-tokens", type=int, default=32)
    ap.add_argument("--ref-tokens", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-op", action="store_true", help="skip the same-GPU per-op baseline")
    ap.add_argument("--no-extra", action="store_true",
                    help="default workload: skip the secondary sweeps (fine, block, split-K, MLP)")
    ap.add_argument("--no-warmup-record", action="store_true",
                    help="default workload: skip the warm-up record among the secondary sweeps")
    ap.add_argument("--trace", type=int, default=None,
                    help="plain MoE workloads: one traced call at this token count, summarised "
                         "(prints the summary, not a bench line)")
    ap.add_argument("--single", type=int, default=None,
                    help="MoE workloads: run warmup+1 calls at this token count and exit "
                         "(for profiler captures; prints no bench line)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.trace is not None:
        line = run_trace(args, local) if rank == 0 else None
    elif args.single is not None:
        if args.workload not in MOE_WORKLOADS:
            ap.error("--single applies to the MoE workloads")
        line = run_single(args, local) if rank == 0 else None
    elif args.impl == "reference":
        line = run_reference(args, world, rank)
    elif args.workload in CHAIN_WORKLOADS:
        line = run_chain(args, world, rank, local)
    elif args.workload == "warmup":
        line = run_warmup(args) if rank == 0 else None
    elif args.workload in ("splitk", "mlp"):
        line = run_dense(args, local) if rank == 0 else None
    else:
        line = run_ours(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
