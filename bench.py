#!/usr/bin/env python3
"""Benchmark of the hashed multi-head N-gram lookup on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference] [--config C]

A step is one pass of the whole lookup over one batch of the workload (default:
the PageGram 200M-parameter bf16 table, 64 x 1024 Zipf(1.1) tokens): canonical IDs,
n-grams, hashes and rows, gather + sign + concat, then the W_V projection with the scalar
gate x + g v (tcgen05). By default both run in one launch (pg_gather_project_gate: the
gather on extra warps of the persistent projection, writing e_t ahead of the tiles that
read it); --path two_kernel runs pg_gather_sign_concat then pg_project_gate, --path fused
pg_lookup_project_gate; the paths not chosen are timed too. With
--config 5 the step is the Engram-27B-shaped module (gather, fused W_V + 4 W_K with
the RMSNorm-sigmoid gate, causal conv + residual).

Rank 0 prints one JSON line. Under torchrun each rank runs its own batch (seeded by
rank; no collective on the data path) and the timing is the max over ranks.
--impl reference times the CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "N-gram memory lookup tokens/s (1 GB300) and % of HBM / tensor roofline"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The fp32 projection runs on the FP32 FMA pipes, not the tensor cores: its peak is derived
# from the unit counts, 152 SMs x 128 FP32 lanes x 2 flop per FMA x 2.07 GHz (maximum SM
# clock), and reported as an ALU bound.
FP32_FFMA_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


# ---------------------------------------------------------------- rank / sharding helpers

# Nominal GB300 figures, reported beside the measured peaks: HBM3e 7.9 TB/s, dense bf16
# 2.25 PFLOP/s; the FP32 FMA peak of the ALU-bound path is already the derived one.
NOMINAL_PEAK = {"hbm": 7900.0, "tensor": 2250.0, "alu": FP32_FFMA_TFLOPS}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_rate(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Units processed by all ranks divided by the slowest rank's time (weak scaling)."""
    return units_per_rank * world / seconds_max


# ---------------------------------------------------------------- peaks and clocks

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed loop runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        load = [r for r in rows if r[2] > 0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i, flag in enumerate(r[3][1:5]) if flag.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(load)}


# ---------------------------------------------------------------- the GPU path

class Pipeline:
    """Resident inputs and outputs of one workload; step() launches the whole path."""

    def __init__(self, cfg: int, dev, rank: int):
        import numpy as np
        import torch

        from hashed_head_gram_gb300 import pg, workloads as W

        self.pg, self.W, self.torch, self.np = pg, W, torch, np
        self.cfg = cfg
        w = self.w = W.make_workload(cfg)
        spec = self.spec = w.tables[0]
        self.desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
        self.dev = dev
        tokens = W.make_tokens(w, rank=rank)
        self.tokens_host = torch.from_numpy(tokens).pin_memory()
        self.tokens = self.tokens_host.to(dev)
        cmap = W.make_canon_map(w)
        self.cmap = None if cmap is None else torch.from_numpy(cmap.view(np.int32)).to(dev)
        self.table = W.make_table(w, spec, dev)
        dn = self.dn = W.make_dense(w, dev)
        self.N, self.din, self.d = w.N, spec.e_width, w.d
        self.tdt = torch.float32 if w.dtype == W.DT_F32 else torch.bfloat16
        self.pdt = pg.F32 if w.dtype == W.DT_F32 else pg.BF16
        self.e = torch.empty(self.N, self.din, dtype=self.tdt, device=dev)
        if w.gate == W.GATE_SCALAR:
            self.out = torch.empty(self.N, self.d, dtype=self.tdt, device=dev)
            self.x_host = dn["x"].cpu().pin_memory()
        elif w.gate == W.GATE_NONE:
            self.out = torch.empty(self.N, self.d, dtype=self.tdt, device=dev)
        else:
            self.v = torch.empty(self.N, self.d, dtype=torch.bfloat16, device=dev)
            self.alpha = torch.empty(w.M, self.N, device=dev)
            self.v_ms = torch.empty(self.N, device=dev)  # mean(v^2) per token, projection -> conv
            nws = pg.workspace_size(self.N, self.din, self.d, w.M, pg.BF16, pg.GATE_CONTEXT)
            self.ws = torch.empty(nws // 4, device=dev)
            self.H0 = dn["H"].clone()
        self.out_host = torch.empty(self.N, self.d, dtype=self.tdt).pin_memory()

    def gather(self):
        self.pg.gather_sign_concat(self.desc, self.tokens, self.table, self.e, self.pdt, canon_map=self.cmap)

    def decode(self, B: int, steps: int = 16, reps: int = 8):
        """Streaming decode on this workload's table and weights: B sequences, one token
        each per step (pg_decode_lookup, the projection with N = B, and in the context-gated
        module pg_decode_conv_residual). `steps` consecutive steps captured in a CUDA graph and
        replayed `reps` times back to back; returns microseconds per step."""
        torch, pg, W, w, dn = self.torch, self.pg, self.W, self.w, self.dn
        tok = torch.from_numpy(W.make_tokens(W.shrink(w, B=B, L=steps)).T.copy()).to(self.dev)   # [steps, B]
        ctx = w.gate == W.GATE_CONTEXT
        st = pg.DecodeState(B, d=self.d if ctx else 0, M=w.M if ctx else 0, dtype=pg.BF16,
                            kernel_size=w.conv_kernel, dilation=w.dilation, device=self.dev)
        e = torch.empty(B, self.din, dtype=torch.bfloat16, device=self.dev)
        v = torch.empty(B, self.d, dtype=torch.bfloat16, device=self.dev)
        if ctx:
            H = dn["H"][:, :B].contiguous() if B <= w.N else torch.zeros(w.M, B, self.d, dtype=torch.bfloat16,
                                                                          device=self.dev)
            alpha = torch.empty(w.M, B, device=self.dev)
            v_ms = torch.empty(B, device=self.dev)
            ws = torch.empty(pg.workspace_size(B, self.din, self.d, w.M, pg.BF16, pg.GATE_CONTEXT) // 4 + 4,
                             device=self.dev)
        else:
            x = dn["x"][:B].contiguous() if "x" in dn and B <= w.N else torch.zeros(B, self.d, dtype=torch.bfloat16,
                                                                                   device=self.dev)

        def step(s):
            pg.decode_lookup(self.desc, st, tok[s], self.table, e, pg.BF16, canon_map=self.cmap)
            if ctx:
                pg.project_gate(e, dn["W"], self.d, pg.GATE_CONTEXT, v, pg.BF16, M=w.M, h=H, gamma_h=dn["gamma_h"],
                                gamma_k=dn["gamma_k"], eps=w.eps, alpha_out=alpha, workspace=ws, v_ms_out=v_ms)
                pg.decode_conv_residual(st, v, alpha, dn["gamma_c"], dn["conv_w"], H, eps=w.eps, v_ms=v_ms)
            elif w.gate == W.GATE_SCALAR:
                pg.project_gate(e, dn["W"], self.d, pg.GATE_SCALAR, v, pg.BF16, g=w.g, x_resid=x)
            else:
                pg.project_gate(e, dn["W"], self.d, pg.GATE_NONE, v, pg.BF16)

        side = torch.cuda.Stream(device=self.dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for s in range(steps):
                step(s)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for s in range(steps):
                step(s)
        graph.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            graph.replay()
        b.record()
        torch.cuda.synchronize()
        if pg.device_error() != 0:
            raise RuntimeError("device error word set during the decode measurement")
        return a.elapsed_time(b) * 1e3 / (reps * steps)

    def project(self):
        pg, w, dn = self.pg, self.w, self.dn
        if w.gate == self.W.GATE_SCALAR:
            pg.project_gate(self.e, dn["W"], self.d, pg.GATE_SCALAR, self.out, self.pdt, g=w.g, x_resid=dn["x"])
        elif w.gate == self.W.GATE_NONE:
            pg.project_gate(self.e, dn["W"], self.d, pg.GATE_NONE, self.out, self.pdt)
        else:
            pg.project_gate(self.e, dn["W"], self.d, pg.GATE_CONTEXT, self.v, pg.BF16, M=w.M, h=dn["H"],
                            gamma_h=dn["gamma_h"], gamma_k=dn["gamma_k"], eps=w.eps, alpha_out=self.alpha,
                            workspace=self.ws, v_ms_out=self.v_ms)

    def conv(self):
        pg, w, dn = self.pg, self.w, self.dn
        pg.conv_residual(w.B, w.L, self.d, w.M, pg.BF16, self.v, self.alpha, dn["gamma_c"], dn["conv_w"], dn["H"],
                         dilation=w.dilation, eps=w.eps, v_ms=self.v_ms)

    def fused(self):
        pg, w, dn = self.pg, self.w, self.dn
        if w.gate == self.W.GATE_SCALAR:
            pg.lookup_project_gate(self.desc, self.tokens, self.table, dn["W"], self.d, pg.GATE_SCALAR, self.out,
                                   canon_map=self.cmap, g=w.g, x_resid=dn["x"])
        else:
            pg.lookup_project_gate(self.desc, self.tokens, self.table, dn["W"], self.d, pg.GATE_CONTEXT, self.v,
                                   canon_map=self.cmap, M=w.M, h=dn["H"], gamma_h=dn["gamma_h"],
                                   gamma_k=dn["gamma_k"], eps=w.eps, alpha_out=self.alpha, workspace=self.ws)

    def overlap(self):
        pg, w, dn = self.pg, self.w, self.dn
        if not hasattr(self, "ws_ov"):
            n = pg.gather_project_workspace_size(self.N, self.d, w.M, w.gate)
            self.ws_ov = self.torch.empty((n + 3) // 4, device=self.dev)
        if w.gate == self.W.GATE_SCALAR:
            pg.gather_project_gate(self.desc, self.tokens, self.table, self.e, dn["W"], self.d, pg.GATE_SCALAR,
                                   self.out, self.ws_ov, canon_map=self.cmap, g=w.g, x_resid=dn["x"])
        elif w.gate == self.W.GATE_NONE:
            pg.gather_project_gate(self.desc, self.tokens, self.table, self.e, dn["W"], self.d, pg.GATE_NONE,
                                   self.out, self.ws_ov, canon_map=self.cmap)
        else:
            pg.gather_project_gate(self.desc, self.tokens, self.table, self.e, dn["W"], self.d, pg.GATE_CONTEXT,
                                   self.v, self.ws_ov, canon_map=self.cmap, M=w.M, h=dn["H"],
                                   gamma_h=dn["gamma_h"], gamma_k=dn["gamma_k"], eps=w.eps, alpha_out=self.alpha,
                                   v_ms_out=self.v_ms)

    def can_fuse(self):
        sp = self.spec
        return (sp.mode != self.W.MODE_FLAT and sp.row_dtype == self.W.DT_BF16 and sp.r == 64
                and self.w.gate != self.W.GATE_NONE and self.w.cfg_id != 4)

    def can_overlap(self):
        return self.can_fuse() and self.d % 256 == 0

    def paths(self):
        """The ways this workload's step can run: the first is the default."""
        if self.can_overlap():
            return ["overlap", "two_kernel", "fused"]
        if self.can_fuse():
            return ["two_kernel", "fused"]
        return ["two_kernel"]

    def stages(self, path="two_kernel"):
        if self.w.cfg_id == 4:   # the 20B NF4 table: the lookup ends at e_t
            return [("gather_sign_concat", self.gather)]
        if path == "overlap":
            st = [("gather_project_gate", self.overlap)]
        elif path == "fused":
            st = [("lookup_project_gate", self.fused)]
        else:
            st = [("gather_sign_concat", self.gather), ("project_gate", self.project)]
        if self.w.gate == self.W.GATE_CONTEXT:
            st.append(("conv_residual", self.conv))
        return st

    def result_tensor(self):
        if self.w.cfg_id == 4:
            return self.e
        return self.dn["H"] if self.w.gate == self.W.GATE_CONTEXT else self.out

    # The end-to-end loop double-buffers what crosses the host link (token IDs and x in,
    # the result out; the branch states H, updated in place, for the context gate).
    def make_slots(self):
        torch = self.torch
        base = {"tokens": self.tokens}
        if hasattr(self, "x_host"):
            base["x"] = self.dn["x"]
        if self.w.gate == self.W.GATE_CONTEXT:
            base["H"] = self.dn["H"]
        elif self.w.cfg_id == 4:
            base["e"] = self.e
        else:
            base["out"] = self.out
        other = {k: torch.empty_like(v) for k, v in base.items()}
        for k in other:
            other[k].copy_(base[k])
        self.slots = [base, other]

    def use_slot(self, k):
        sl = self.slots[k]
        self.tokens = sl["tokens"]
        if "x" in sl:
            self.dn["x"] = sl["x"]
        if "H" in sl:
            self.dn["H"] = sl["H"]
        if "e" in sl:
            self.e = sl["e"]
        if "out" in sl:
            self.out = sl["out"]

    # algorithmic work per launch ("Roofline")
    def algorithmic(self, name):
        N, din, d, w = self.N, self.din, self.d, self.w
        if name == "gather_sign_concat":
            # 2K rows x row bytes (sector-rounded for NF4) + token ID + e_t write, per token
            rb = self.spec.row_bytes if self.spec.row_dtype != self.W.DT_NF4 else 64
            per = len(self.spec.orders) * self.spec.K * rb + 4 + din * self.e.element_size()
            return "hbm", per * N
        if name == "gather_project_gate":
            # one launch doing both kernels' work; its binding roof is HBM (e_t written and
            # read back, 2K rows, IDs, the epilogue operand and the output: 89 us at the
            # measured copy rate on the PageGram 200M workload, against 55 us of tensor work)
            rb = self.spec.row_bytes
            e_b = din * self.e.element_size()
            epi = d * 2 * (2 if w.gate == self.W.GATE_SCALAR else 1 + 2 * w.M)
            return "hbm", (len(self.spec.orders) * self.spec.K * rb + 4 + 2 * e_b + epi) * N
        if name in ("project_gate", "lookup_project_gate"):
            cols = d * (1 + w.M)
            return ("alu" if w.dtype == self.W.DT_F32 else "tensor"), 2.0 * N * din * cols
        # conv: read v, read + write H for every branch
        return "hbm", N * (d * 2 + 2 * w.M * d * 2)


def compulsory_gather_bytes(p) -> float:
    """Distinct 32-byte table sectors the batch touches (rows from pg_canon_hash on
    the GPU) + token IDs + the e_t write: a lower bound on the gather's DRAM traffic."""
    torch, pg = p.torch, p.pg
    rows = torch.empty(p.N, len(p.spec.orders), p.spec.K, dtype=torch.int32, device=p.dev)
    pg.canon_hash(p.desc, p.tokens, rows, canon_map=p.cmap)
    r = rows.view(-1).to(torch.int64) & 0xFFFFFFFF
    rb = p.spec.row_bytes
    first = (r * rb) // 32
    last = (r * rb + rb - 1) // 32
    span = torch.arange((rb + 31) // 32 + 1, device=p.dev)
    cand = first.unsqueeze(1) + span
    cand = cand[cand <= last.unsqueeze(1)]
    distinct = int(torch.unique(cand).numel())
    return distinct * 32.0 + p.N * 4 + p.N * p.din * p.e.element_size()


def flush_l2(buf):
    """Untimed L2 flush between steps: write a buffer larger than L2, then read it back so
    the written lines are written back here, not inside the next timed kernel."""
    buf.add_(1)
    buf.sum(dtype=buf.dtype)


def time_stages(stages, steps, stream, flush):
    """CUDA-event durations (ms) of every stage of `steps` steps; L2 flushed between steps."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        for j, (_, fn) in enumerate(stages):
            fn()
            ev[i][j + 1].record(stream)
        flush_l2(flush)
    torch.cuda.synchronize()
    return [[ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)] for j in range(len(stages))]


def run_gpu(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", torch.cuda.current_device())
    from hashed_head_gram_gb300 import pg

    p = Pipeline(args.config, dev, rank)
    stream = torch.cuda.current_stream()
    flush = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    path = args.path if args.path in p.paths() else p.paths()[0]
    stages = p.stages(path)

    # ---- warm-up
    for _ in range(args.warmup):
        for _, fn in stages:
            fn()
        flush_l2(flush)
    torch.cuda.synchronize()
    if p.w.gate == p.W.GATE_CONTEXT:
        p.dn["H"].copy_(p.H0)
    torch.cuda.synchronize()

    # ---- device-timed loop: events around every stage of every step, L2 flushed between steps
    launches0 = pg.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        t_wall = time.perf_counter()
        stage_ms = time_stages(stages, args.steps, stream, flush)
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    launches = pg.launch_count() - launches0
    step_ms = [sum(stage_ms[j][i] for j in range(len(stages))) for i in range(args.steps)]
    total_s = reduce_max(sum(step_ms) / 1e3, world)
    value = whole_job_rate(p.N * args.steps, world, total_s)

    # ---- end to end through the C ABI with host buffers: every step uploads its token IDs
    #      (and x) from pinned host memory and reads its whole result back; steps are
    #      pipelined (uploads on one copy stream, kernels on the launching stream, read-backs
    #      on another, double-buffered device tensors) as a serving loop would run them
    h2d = p.tokens_host.numel() * 4 + (p.x_host.numel() * 2 if hasattr(p, "x_host") else 0)
    p.make_slots()
    res0 = p.result_tensor()
    res_hosts = [torch.empty_like(res0, device="cpu").pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = max(2, min(args.steps, 200))
    barrier(world)
    torch.cuda.synchronize()
    t_e0, t_e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_e0.record(s_in)
    for i in range(e2e_steps):
        k = i % 2
        sl = p.slots[k]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[k])    # step i-2's kernels are done with slot k's inputs
            sl["tokens"].copy_(p.tokens_host, non_blocking=True)
            if "x" in sl:
                sl["x"].copy_(p.x_host, non_blocking=True)
            ev_in[k].record(s_in)
        stream.wait_event(ev_in[k])
        if i >= 2:
            stream.wait_event(ev_out[k])       # step i-2's result in slot k has been read back
        p.use_slot(k)
        for _, fn in stages:
            fn()
        ev_comp[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[k])
            res_hosts[k].copy_(p.result_tensor(), non_blocking=True)
            ev_out[k].record(s_out)
    t_e1.record(s_out)
    torch.cuda.synchronize()
    p.use_slot(0)
    e2e_s = reduce_max(t_e0.elapsed_time(t_e1) / 1e3, world)
    e2e_value = whole_job_rate(p.N * e2e_steps, world, e2e_s)
    d2h = res0.numel() * res0.element_size()

    # ---- roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    means = {name: statistics.mean(stage_ms[j]) for j, (name, _) in enumerate(stages)}
    dom = max(means, key=means.get)
    bound, work = p.algorithmic(dom)
    dur_s = means[dom] / 1e3
    traffic = traffic_of(args.config, dom)
    if bound == "hbm":
        achieved, peak, unit = work / dur_s / 1e9, float(peaks["hbm_gbs"]), "GB/s"
    elif bound == "alu":
        achieved, peak, unit = work / dur_s / 1e12, round(FP32_FFMA_TFLOPS, 1), "TFLOP/s"
    else:
        achieved, peak, unit = work / dur_s / 1e12, float(peaks["bf16_tflops"]), "TFLOP/s"
    kernels = {}
    for j, (name, _) in enumerate(stages):
        b, wk = p.algorithmic(name)
        ms = means[name]
        if b == "hbm":
            kernels[name] = {"ms": round(ms, 5), "GB/s": round(wk / (ms / 1e3) / 1e9, 1),
                             "frac_hbm": round(wk / (ms / 1e3) / 1e9 / float(peaks["hbm_gbs"]), 4)}
        elif b == "alu":
            kernels[name] = {"ms": round(ms, 5), "TFLOP/s": round(wk / (ms / 1e3) / 1e12, 1),
                             "frac_fp32_ffma": round(wk / (ms / 1e3) / 1e12 / FP32_FFMA_TFLOPS, 4)}
        else:
            kernels[name] = {"ms": round(ms, 5), "TFLOP/s": round(wk / (ms / 1e3) / 1e12, 1),
                             "frac_tensor": round(wk / (ms / 1e3) / 1e12 / float(peaks["bf16_tflops"]), 4)}
    comp = compulsory_gather_bytes(p)
    if "gather_sign_concat" in means:
        g_ms = means["gather_sign_concat"]
        kernels["gather_sign_concat"]["compulsory_bytes"] = comp
        kernels["gather_sign_concat"]["frac_hbm_compulsory"] = round(
            comp / (g_ms / 1e3) / 1e9 / float(peaks["hbm_gbs"]), 4)
    if "lookup_project_gate" in means:
        # e_t never reaches memory: table sectors + IDs + the epilogue operand in + the output
        fb = comp - p.N * p.din * 2 + p.N * p.d * 2 * (2 if p.w.gate == p.W.GATE_SCALAR else 1 + 2 * p.w.M)
        f_ms = means["lookup_project_gate"]
        kernels["lookup_project_gate"]["compulsory_bytes"] = fb
        kernels["lookup_project_gate"]["GB/s_compulsory"] = round(fb / (f_ms / 1e3) / 1e9, 1)
        kernels["lookup_project_gate"]["frac_hbm_compulsory"] = round(
            fb / (f_ms / 1e3) / 1e9 / float(peaks["hbm_gbs"]), 4)
    if "gather_project_gate" in means:
        # e_t written once and read back by the projection (mostly from L2): table sectors +
        # IDs + e_t + the epilogue operand in + the output
        fb = comp + p.N * p.d * 2 * (2 if p.w.gate == p.W.GATE_SCALAR else 1 + 2 * p.w.M)
        o_ms_ = means["gather_project_gate"]
        kernels["gather_project_gate"]["compulsory_bytes"] = fb
        kernels["gather_project_gate"]["GB/s_compulsory"] = round(fb / (o_ms_ / 1e3) / 1e9, 1)
        kernels["gather_project_gate"]["frac_hbm_compulsory"] = round(
            fb / (o_ms_ / 1e3) / 1e9 / float(peaks["hbm_gbs"]), 4)
    other = []
    for op in p.paths():
        if op == path:
            continue
        ost = p.stages(op)
        o_ms = time_stages(ost, max(3, args.steps // 4), stream, flush)
        other.append({"path": op, "ms_per_step": round(sum(statistics.mean(x) for x in o_ms), 5),
                      "kernels": {name: round(statistics.mean(o_ms[j]), 5) for j, (name, _) in enumerate(ost)}})

    # ---- the no-reuse control: the same path on uniform IDs (Zipf workloads only)
    control = None
    if p.w.zipf_s is not None:
        import torch as _t
        zipf_tokens = p.tokens.clone()
        p.tokens.copy_(_t.from_numpy(p.W.make_tokens(p.w, rank=rank, uniform=True)).to(dev))
        u_ms = time_stages(stages, max(3, args.steps // 4), stream, flush)
        u_means = {name: statistics.mean(u_ms[j]) for j, (name, _) in enumerate(stages)}
        u_step = sum(u_means.values())
        comp_u = compulsory_gather_bytes(p)
        if dom == "gather_project_gate":
            comp_u += p.N * p.d * 2 * (2 if p.w.gate == p.W.GATE_SCALAR else 1 + 2 * p.w.M)
        b_u, work_u = p.algorithmic(dom)
        ck = {"ms": round(u_means[dom], 5)}
        if b_u == "hbm":
            ck["frac_hbm"] = round(work_u / (u_means[dom] / 1e3) / 1e9 / float(peaks["hbm_gbs"]), 4)
            if dom in ("gather_sign_concat", "gather_project_gate"):
                ck["compulsory_bytes"] = comp_u
                ck["frac_hbm_compulsory"] = round(comp_u / (u_means[dom] / 1e3) / 1e9 / float(peaks["hbm_gbs"]), 4)
        control = {"ids": "i.i.d. uniform over the vocabulary (no reuse: the compulsory bytes approach the "
                          "algorithmic ones)", "ms_per_step": round(u_step, 5),
                   "tokens_per_s": round(whole_job_rate(p.N, world, reduce_max(u_step / 1e3, world)), 1),
                   "kernels": {dom: ck}}
        p.tokens.copy_(zipf_tokens)
        del zipf_tokens

    decode = []
    if p.w.dtype == p.W.DT_BF16:
        for B in sorted({1, p.w.B, 4096}):
            us = p.decode(B)
            decode.append({"sequences": B, "us_per_step": round(us, 2), "tokens_per_s": round(B / us * 1e6, 1)})

    clocks = clk.summary()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.mean(step_ms), 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if p.w.dtype == p.W.DT_F32 else "bf16",
            "data": "synthetic: seeded Zipf token IDs, int8/64 table values, N(0,0.02) weights, N(0,1) states",
            "config": workload_config(p.w, world),
            "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "how": f"{e2e_steps} steps pipelined: each uploads its inputs from pinned host memory and "
                           "reads its whole result back; uploads, kernels and read-backs of consecutive steps "
                           "overlap on three streams (double-buffered device tensors); no L2 flush (inputs "
                           "> L2 except the tiny workload)"},
            "gpu_launches": launches,
            "roofline": {"bound": bound, "kernel": dom, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "frac_nominal": round(achieved / NOMINAL_PEAK[bound], 4),
                         "peak_source": ("derived: 152 SMs x 128 FP32 lanes x 2 flop x 2.07 GHz" if bound == "alu"
                                         else f"{peak_src} ({'hbm_gbs' if bound == 'hbm' else 'bf16_tflops'})")},
            "kernels": kernels,
            "path": path,
            "other_paths": other,
            "uniform_ids_control": control,
            "decode": {"steps": decode,
                       "how": "streaming decode, one token per sequence and step, on the same table and weights "
                              "(decode lookup -> projection with N = sequences -> decode conv where the module has "
                              "one); 16 consecutive steps in one CUDA graph replayed back to back, no L2 flush "
                              "(table rows cold, W and the state warm, as in serving); not part of value"},
            "clocks": clocks,
            "wall_s_timed_loop": round(t_wall, 4),
        }
        if world == 1 and not args.no_cpu_baseline:
            if p.spec.table_bytes > (8 << 30):
                line["cpu_baseline"] = None   # the table does not fit the host-side oracle leg
            else:
                line["cpu_baseline"] = cpu_baseline(args.config, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ncu-measured DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum),
# keyed by (workload, stage), with the sha256 prefix of the kernel's source file followed by
# the csrc headers (sorted) at the time of the capture; reported only while those sources
# are unchanged (profiles/ holds the captures).
TRAFFIC = {
    (2, "gather_project_gate"): ("pg_project.cu", "2a1469a817ae6a29", 403.618304e6),
    (2, "gather_sign_concat"): ("pg_lookup.cu", "b7b2203aa8b0ee2c", 180.663808e6),
    (2, "project_gate"): ("pg_project.cu", "2a1469a817ae6a29", 307.012096e6),
    (2, "lookup_project_gate"): ("pg_project.cu", "2a1469a817ae6a29", 274.138624e6),
    (4, "gather_sign_concat"): ("pg_lookup.cu", "b7b2203aa8b0ee2c", 190.301952e6),
    (5, "gather_sign_concat"): ("pg_lookup.cu", "b7b2203aa8b0ee2c", 143.117312e6),
    (5, "project_gate"): ("pg_project.cu", "2a1469a817ae6a29", 1069.227776e6),
    (5, "conv_residual"): ("pg_conv.cu", "dedb84e101a08b0d", 1463.943936e6),
}


def source_sha(src):
    """sha256 prefix of csrc/<src> followed by every csrc header, sorted by name."""
    import glob
    import hashlib
    csrc = os.path.join(ROOT, "hashed_head_gram_gb300", "csrc")
    h = hashlib.sha256()
    for path in [os.path.join(csrc, src)] + sorted(glob.glob(os.path.join(csrc, "*.cuh"))):
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_of(cfg, stage):
    entry = TRAFFIC.get((cfg, stage))
    if entry is None:
        return None
    src, sha, nbytes = entry
    try:
        now = source_sha(src)
    except OSError:
        return None
    return nbytes if now == sha else None


def workload_config(w, world):
    t = w.tables[0]
    desc = {2: "PageGram 200M-parameter bf16 table: P_n = 48,823 / 48,821 pages, K=8, S=4, r=64; "
               "Zipf(1.1) IDs over 50,304; W_V 1024->768; scalar gate g=0.5",
            4: "20B-parameter PageGram table in NF4 (34-byte rows, 10.6 GB): P_n = 4,882,811 / 4,882,789, K=8, "
               "S=4; Zipf(1.05) over 128,000 IDs folded to 98,010; gather + NF4 dequant + sign + concat",
            1: "tiny fp32 PageGram table (P_n=64, K=8, S=4, r=64); 4096 uniform IDs over 1024; fp32 W_V 1024->256",
            5: "Engram-27B-shaped module: 16 prime subtables ~2.2266M rows, r=80, bf16; Zipf(1.05) over 128k "
               "with canonical folding; fused W_V + 4 W_K (1280 -> 12800); RMSNorm-sigmoid gate; causal "
               "depthwise conv k=4 dilation 3 + SiLU + residual into 4 branches of d=2560"}.get(w.cfg_id, w.name)
    return {"workload": f"{w.name} (config {w.cfg_id}): {desc}", "batch": f"{w.B}x{w.L}", "tokens_per_gpu": w.N,
            "table_bytes": t.table_bytes, "parallelism": f"dp{world} (independent batches, no collective)",
            "l2": "flushed between timed steps (256 MiB written, then read back, untimed); "
                  "table and activations > L2"}


# ---------------------------------------------------------------- CPU oracle legs

def _oracle_sample(cfg: int, ntok: int):
    """Runs the oracle over the first `ntok` tokens of the workload; returns seconds."""
    import numpy as np
    import torch

    from hashed_head_gram_gb300 import workloads as W
    from oracle import dense, oracle as orc

    w = W.make_workload(cfg)
    spec = w.tables[0]
    tokens = W.make_tokens(w)
    cmap = W.make_canon_map(w)
    L = w.L
    nseq = max(1, (ntok + L - 1) // L)
    tok = tokens[:nseq]
    which = np.arange(min(ntok, nseq * L), dtype=np.int64)
    table = _cpu_table(w, spec)
    dn = _cpu_dense(w)
    t0 = time.perf_counter()
    canon, rows, signs, bad = orc.index(spec, tok, cmap, w.vocab, which)
    rowdata = orc.fetch_rows(table, rows)
    e = orc.assemble(spec, rows, rowdata, signs, orc.F32 if spec.row_dtype == W.DT_F32 else orc.BF16)
    if w.cfg_id == 4:   # the lookup ends at e_t
        return time.perf_counter() - t0, len(which)
    ef = e.astype(np.float64) if spec.row_dtype == W.DT_F32 else orc.bf16_bits_to_f64(e)
    if w.gate == W.GATE_NONE:
        dense.project(ef, dn["W"])
    elif w.gate == W.GATE_SCALAR:
        v = dense.project(ef, dn["W"])
        dense.scalar_gate(dn["x"][:len(which)], v, w.g)
    else:
        v, a = dense.engram_gate(ef, dn["W"], dn["H"][:, :len(which)], dn["gh"], dn["gk"], w.eps, w.M)
        n = len(which) // L * L
        if n:
            dense.conv_residual(v[:n].reshape(-1, L, w.d), a[:, :n].reshape(w.M, -1, L), dn["gc"], dn["cw"],
                                w.dilation, w.eps, dn["H"][:, :n].reshape(w.M, -1, L, w.d))
    return time.perf_counter() - t0, len(which)


_CPU_CACHE = {}


def _cpu_table(w, spec):
    """Host copy of the table rows. The table tensor is generated on the CPU with the
    same seeded generator kind the tests use (only the rows are needed)."""
    import numpy as np
    from hashed_head_gram_gb300 import workloads as W
    key = ("t", w.cfg_id)
    if key not in _CPU_CACHE:
        if spec.table_bytes > (8 << 30):
            raise RuntimeError("table too large for the CPU baseline leg")
        t = W.make_table(w, spec, "cpu")
        _CPU_CACHE[key] = t.view(__import__("torch").uint8).reshape(spec.table_rows, spec.row_bytes).numpy()
    return _CPU_CACHE[key]


def _cpu_dense(w):
    from hashed_head_gram_gb300 import workloads as W
    key = ("d", w.cfg_id)
    if key not in _CPU_CACHE:
        dn = W.make_dense(w, "cpu")
        out = {"W": dn["W"].double().numpy()}
        if "x" in dn:
            out["x"] = dn["x"].double().numpy()
        if "H" in dn:
            out.update(H=dn["H"][:, :8192].double().numpy(), gh=dn["gamma_h"].double().numpy(),
                       gk=dn["gamma_k"].double().numpy(), gc=dn["gamma_c"].double().numpy(),
                       cw=dn["conv_w"].double().numpy())
        _CPU_CACHE[key] = out
    return _CPU_CACHE[key]


def cpu_baseline(cfg: int, seconds: float):
    """The oracle as it stands on the host cores, on a bounded sample of the workload."""
    dt, n = _oracle_sample(cfg, 1024)                     # calibration
    w = __import__("hashed_head_gram_gb300.workloads", fromlist=["x"]).make_workload(cfg)
    cap = 8192 if w.gate == 2 else 1 << 16   # the host copy of the branch states holds 8192 tokens
    want = int(max(1024, min(cap, n * seconds / max(dt, 1e-3))))
    dt, n = _oracle_sample(cfg, want)
    return {"value": round(n / dt, 1), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {n} tokens of the workload batch; C stages single-threaded, numpy fp64 "
                      f"projection/gate on the BLAS thread pool (up to {os.cpu_count()} cores); {dt:.2f} s"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    dt1, n1 = _oracle_sample(args.config, 256)
    budget = 60.0                                         # seconds for the whole run
    per_step = max(64, min(1 << 14, int(n1 * budget / max((args.steps + args.warmup) * dt1, 1e-6))))
    for _ in range(args.warmup):
        _oracle_sample(args.config, per_step)
    total_t, total_n = 0.0, 0
    for _ in range(args.steps):
        dt, n = _oracle_sample(args.config, per_step)
        total_t += dt
        total_n += n
    value = total_n / total_t
    from hashed_head_gram_gb300 import workloads as W
    w = W.make_workload(args.config)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_t / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (same seeded workload as the GPU arm)", "config": workload_config(w, 1),
            "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"{per_step} tokens per step from the workload batch"},
            "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--path", choices=["auto", "overlap", "two_kernel", "fused"], default="auto",
                    help="how the lookup and the projection run: overlap = one launch writing e_t with the "
                         "gather on extra warps of the projection (pg_gather_project_gate); two_kernel = "
                         "pg_gather_sign_concat + pg_project_gate; fused = pg_lookup_project_gate (r = 64 bf16 "
                         "tables); auto = the first that applies, in that order. The others that apply are "
                         "timed too and reported as other_paths")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
