#!/usr/bin/env python3
"""Benchmark of the hashed multi-head N-gram lookup on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference] [--config C]
                    [--workloads all|C,C,...] [--path auto|overlap|two_kernel|fused]
    python bench.py --kernel {gather,project,project_fp8,gather_project,conv,nf4_export,decode,slots} --config C

A step is one pass of the whole lookup over one batch of a workload. The headline
(--config, default 5) is the Engram-27B-shaped module, 8 x 4096 Zipf tokens: canonical
IDs, n-grams, hashes and rows, gather + sign + concat (pg_gather_sign_concat), the fused
W_V + 4 W_K projection with the RMSNorm-sigmoid gate (tcgen05; pg_project_gate), the
causal depthwise conv + SiLU + residual into the 4 branch states (pg_conv_residual). The
other four workloads are measured in the same run (same method, at least 100 timed
steps) and reported under "workloads": the tiny fp32 tables, the PageGram 200M bf16
table (lookup + projection + scalar gate in one launch, pg_gather_project_gate), the
Engram-style 200M table and the 20B NF4 table (the lookup alone).

Rank 0 prints one JSON line. Under torchrun each rank runs its own batch (seeded by
rank; no collective on the data path) and the timing is the max over ranks.
--impl reference times the CPU oracle on the host cores instead (rank 0 only).
--kernel runs one kernel at a time on a workload's shapes (timing and profiling).
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
FP8_OVER_BF16 = 4.5 / 2.25     # nominal dense FP8 / bf16 tensor rates of GB300
ALL_WORKLOADS = (1, 2, 3, 4, 5)
EXTRA_MIN_STEPS = 100          # timed steps of the workloads besides the headline

# Nominal GB300 figures, reported beside the measured peaks: HBM3e 7.9 TB/s, dense bf16
# 2.25 PFLOP/s; the FP32 FMA peak of the ALU-bound path is already the derived one.
NOMINAL_PEAK = {"hbm": 7900.0, "tensor": 2250.0, "tensor_fp8": 4500.0, "alu": FP32_FFMA_TFLOPS}


# ---------------------------------------------------------------- rank / sharding helpers

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

GATHER_KERNELS = ("gather_sign_concat", "gather_project_gate", "lookup_project_gate")


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
        self.rank = rank
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

    def gather(self):
        self.pg.gather_sign_concat(self.desc, self.tokens, self.table, self.e, self.pdt, canon_map=self.cmap)

    def fp8_ready(self):
        """E4M3 operands of the FP8 path: W quantised once (a weight), buffers for e_t's codes."""
        if hasattr(self, "qe"):
            return
        torch, dn = self.torch, self.dn
        self.qe = torch.empty(self.N, self.din, dtype=torch.uint8, device=self.dev)
        self.se = torch.empty(self.N, device=self.dev)
        self.qw = torch.empty(dn["W"].shape, dtype=torch.uint8, device=self.dev)
        self.sw = torch.empty(dn["W"].shape[0], device=self.dev)
        self.pg.fp8_quantize(dn["W"], self.qw, self.sw)
        torch.cuda.synchronize()

    def gather_q8(self):
        self.pg.gather_sign_concat_e4m3(self.desc, self.tokens, self.table, self.qe, self.se, canon_map=self.cmap)

    def project_fp8(self):
        pg, w, dn = self.pg, self.w, self.dn
        if w.gate == self.W.GATE_SCALAR:
            pg.project_gate_fp8(self.qe, self.se, self.qw, self.sw, self.d, pg.GATE_SCALAR, self.out, g=w.g,
                                x_resid=dn["x"])
        else:
            pg.project_gate_fp8(self.qe, self.se, self.qw, self.sw, self.d, pg.GATE_CONTEXT, self.v, M=w.M,
                                h=dn["H"], gamma_h=dn["gamma_h"], gamma_k=dn["gamma_k"], eps=w.eps,
                                alpha_out=self.alpha, workspace=self.ws, v_ms_out=self.v_ms)

    def decode(self, B: int, steps: int = 16, reps: int = 8, one_launch: bool = False):
        """Streaming decode on this workload's table and weights: B sequences, one token
        each per step (pg_decode_lookup, the projection with N = B, and in the context-gated
        module pg_decode_conv_residual; with one_launch, pg_decode_step, B <= 8). `steps`
        consecutive steps captured in a CUDA graph and replayed `reps` times back to back;
        returns microseconds per step."""
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

        if one_launch:
            ws1 = torch.zeros((pg.decode_step_workspace_size(B, self.d, w.M if ctx else 0) + 3) // 4,
                              dtype=torch.int32, device=self.dev)

        def step(s):
            if one_launch:
                if ctx:
                    pg.decode_step(self.desc, st, tok[s], self.table, dn["W"], self.d, pg.GATE_CONTEXT, v, ws1,
                                   canon_map=self.cmap, H=H, gamma_h=dn["gamma_h"], gamma_k=dn["gamma_k"],
                                   gamma_c=dn["gamma_c"], conv_w=dn["conv_w"], eps=w.eps, alpha_out=alpha,
                                   v_ms_out=v_ms)
                else:
                    gate = pg.GATE_SCALAR if w.gate == W.GATE_SCALAR else pg.GATE_NONE
                    pg.decode_step(self.desc, st, tok[s], self.table, dn["W"], self.d, gate, v, ws1,
                                   canon_map=self.cmap, g=w.g, x_resid=x if gate == pg.GATE_SCALAR else None)
                return
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

    def project_conv(self):
        """The context-gated projection and the conv + residual in one launch."""
        pg, w, dn = self.pg, self.w, self.dn
        if not hasattr(self, "ws_pc"):
            n = pg.project_gate_conv_workspace_size(self.N, self.d, w.M)
            self.ws_pc = self.torch.empty((n + 3) // 4, device=self.dev)
        pg.project_gate_conv(w.B, w.L, self.e, dn["W"], self.d, w.M, dn["H"], dn["gamma_h"], dn["gamma_k"],
                             dn["gamma_c"], dn["conv_w"], self.v, self.alpha, self.ws_pc, dilation=w.dilation,
                             eps=w.eps, v_ms_out=self.v_ms)

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

    def can_fp8(self):
        sp = self.spec
        return (sp.mode != self.W.MODE_FLAT and sp.row_dtype == self.W.DT_BF16 and sp.r in (64, 80)
                and self.w.gate != self.W.GATE_NONE and self.d % 256 == 0 and self.din % 256 == 0)

    def can_conv_fuse(self):
        return (self.w.gate == self.W.GATE_CONTEXT and self.w.dtype == self.W.DT_BF16 and self.d % 256 == 0
                and self.din % 64 == 0)

    def paths(self):
        """The ways this workload's step can run: the first is the default (bf16)."""
        out = ["two_kernel"]
        if self.can_conv_fuse():
            out = ["two_kernel", "conv_fused"]
        if self.can_overlap():
            out = ["overlap", "two_kernel", "fused"]
        elif self.can_fuse():
            out = ["two_kernel", "fused"]
        if self.can_fp8():
            out.append("fp8")
        return out

    def stages(self, path="two_kernel"):
        if self.w.cfg_id == 4:   # the 20B NF4 table: the lookup ends at e_t
            return [("gather_sign_concat", self.gather)]
        if path == "overlap":
            st = [("gather_project_gate", self.overlap)]
        elif path == "conv_fused":
            return [("gather_sign_concat", self.gather), ("project_gate_conv", self.project_conv)]
        elif path == "fp8":
            self.fp8_ready()
            st = [("gather_sign_concat_e4m3", self.gather_q8), ("project_gate_fp8", self.project_fp8)]
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

    def epilogue_bytes(self):
        """Per token: the projection's epilogue operand in and result out (scalar gate: x in,
        out; context gate: h of every branch in, v out)."""
        w = self.w
        if w.gate == self.W.GATE_SCALAR:
            return self.d * 2 * 2
        if w.gate == self.W.GATE_CONTEXT:
            return self.d * 2 * (1 + w.M)
        return self.d * 2

    def weight_bytes(self):
        return (1 + self.w.M) * self.d * self.din * (4 if self.w.dtype == self.W.DT_F32 else 2)

    def algorithmic(self, name):
        """(bound, work per launch) with no reuse counted: every row read from HBM as often as
        the method addresses it (sector-rounded for the 34-byte NF4 rows)."""
        N, din, d, w = self.N, self.din, self.d, self.w
        rows = len(self.spec.orders) * (1 if self.spec.mode == self.W.MODE_FLAT else self.spec.K)
        rb = self.spec.row_bytes if self.spec.row_dtype != self.W.DT_NF4 else 64
        e_b = din * self.e.element_size()
        if name == "gather_sign_concat":
            # 2K rows + token ID + e_t write, per token
            return "hbm", (rows * rb + 4 + e_b) * N
        if name == "gather_project_gate":
            # one launch doing the lookup and the projection: rows, ID, e_t written once, the
            # epilogue operand and the output (e_t's read-back by the tiles is the split's own
            # cost, not the method's, and comes mostly from L2); its binding roof is HBM
            return "hbm", (rows * rb + 4 + e_b + self.epilogue_bytes()) * N + self.weight_bytes()
        if name == "lookup_project_gate":
            return "hbm", (rows * rb + 4 + self.epilogue_bytes()) * N + self.weight_bytes()
        if name == "gather_sign_concat_e4m3":
            # 2K rows + token ID + E4M3 e_t (1 byte per element) + its fp32 scale, per token
            return "hbm", (rows * rb + 4 + din + 4) * N
        if name == "project_gate_fp8":
            return "tensor_fp8", 2.0 * N * din * d * (1 + w.M)
        if name in ("project_gate", "project_gate_conv"):
            cols = d * (1 + w.M)
            return ("alu" if w.dtype == self.W.DT_F32 else "tensor"), 2.0 * N * din * cols
        # conv: read v, read + write H for every branch
        return "hbm", N * (d * 2 + 2 * w.M * d * 2)

    def compulsory(self, name, table_sectors_bytes):
        """Lower bound on a kernel's DRAM bytes: the distinct 32-byte table sectors the batch
        touches, token IDs, e_t written (where it leaves the kernel), the epilogue operand and
        output, and W."""
        N = self.N
        e_b = self.din * self.e.element_size()
        if name == "gather_sign_concat":
            return table_sectors_bytes + N * 4 + N * e_b
        if name == "gather_project_gate":
            return table_sectors_bytes + N * (4 + e_b + self.epilogue_bytes()) + self.weight_bytes()
        if name == "lookup_project_gate":
            return table_sectors_bytes + N * (4 + self.epilogue_bytes()) + self.weight_bytes()
        if name == "gather_sign_concat_e4m3":
            return table_sectors_bytes + N * (4 + self.din + 4)
        return None


def table_sector_bytes(p) -> float:
    """Distinct 32-byte table sectors the batch touches (rows from pg_canon_hash on the
    GPU), in bytes."""
    torch, pg = p.torch, p.pg
    heads = 1 if p.spec.mode == p.W.MODE_FLAT else p.spec.K
    rows = torch.empty(p.N, len(p.spec.orders), heads, dtype=torch.int32, device=p.dev)
    pg.canon_hash(p.desc, p.tokens, rows, canon_map=p.cmap)
    r = rows.view(-1).to(torch.int64) & 0xFFFFFFFF
    rb = p.spec.row_bytes
    first = (r * rb) // 32
    last = (r * rb + rb - 1) // 32
    span = torch.arange((rb + 31) // 32 + 1, device=p.dev)
    cand = first.unsqueeze(1) + span
    cand = cand[cand <= last.unsqueeze(1)]
    return float(torch.unique(cand).numel()) * 32.0


def row_references(p, steps, flush) -> dict:
    """The rows the lookup reads, moved by themselves: pg_row_copy (the same row indices,
    from pg_canon_hash before the timed region, the same 16-byte loads, a dense write of each
    row's 16-byte-aligned window; no hashing, signs, dequantisation or concatenation) and
    torch.index_select of the same rows (a library gather). Each timed over `steps`
    launches with the L2 flushed between them."""
    torch, pg = p.torch, p.pg
    heads = 1 if p.spec.mode == p.W.MODE_FLAT else p.spec.K
    rows = torch.empty(p.N, len(p.spec.orders), heads, dtype=torch.int32, device=p.dev)
    pg.canon_hash(p.desc, p.tokens, rows, canon_map=p.cmap)
    rows = rows.view(-1)
    n = rows.numel()
    rb = p.spec.row_bytes
    wb = pg.row_copy_window(rb)
    ob = max(wb, p.e.element_size() * (p.spec.r if p.spec.mode != p.W.MODE_FLAT else p.din))  # e_t bytes per row
    out = torch.empty(n, ob, dtype=torch.uint8, device=p.dev)
    idx = rows.to(torch.int64) & 0xFFFFFFFF
    wide = torch.int64 if rb % 8 == 0 else torch.int16
    tab = p.table.view(torch.uint8).view(-1)[: p.spec.table_rows * rb].view(wide).view(p.spec.table_rows, -1)
    sel = torch.empty(n, tab.shape[1], dtype=wide, device=p.dev)

    def timed(fn):
        for _ in range(3):
            fn()
            flush_l2(flush)
        ms = []
        for _ in range(steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            flush_l2(flush)
            ms.append((a, b))
        torch.cuda.synchronize()
        return statistics.mean(x.elapsed_time(y) for x, y in ms)

    t_copy = timed(lambda: pg.row_copy(p.table, rb, rows, out, ob))
    t_sel = timed(lambda: torch.index_select(tab, 0, idx, out=sel))
    del out, sel, tab, idx, rows
    return {
        "rows": n, "row_bytes": rb,
        "row_copy": {"ms": round(t_copy, 5), "rows_per_s": round(n / (t_copy / 1e3), 1), "window_bytes": wb,
                     "out_row_bytes": ob, "GB/s_read_plus_write": round(n * (wb + ob) / (t_copy / 1e3) / 1e9, 1),
                     "how": f"pg_row_copy of the batch's rows (indices from pg_canon_hash): each row's "
                            f"{wb}-byte aligned window read with 16-byte loads and written densely as a {ob}-byte "
                            f"row (the lookup's output bytes per row), {steps} launches, L2 flushed between them"},
        "torch_index_select": {"ms": round(t_sel, 5), "rows_per_s": round(n / (t_sel / 1e3), 1),
                               "how": "torch.index_select of the same rows into a dense buffer (library gather)"},
    }


def compulsory_gather_bytes(p) -> float:
    """Distinct 32-byte table sectors + token IDs + the e_t write: a lower bound on the
    gather's DRAM traffic."""
    return p.compulsory("gather_sign_concat", table_sector_bytes(p))


def flush_l2(buf):
    """Untimed L2 flush between steps: write a buffer larger than L2, then read it back so
    the written lines are written back here, not inside the next timed kernel."""
    buf.add_(1)
    buf.sum(dtype=buf.dtype)


def time_stages(stages, steps, stream, flush):
    """CUDA-event durations (ms) of every stage of `steps` steps; L2 flushed between steps.
    The first step also starts behind a flush, so the device is busy while the host enqueues
    it (otherwise the host's launch latency of its first kernel lands between its events)."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(steps)]
    flush_l2(flush)
    for i in range(steps):
        ev[i][0].record(stream)
        for j, (_, fn) in enumerate(stages):
            fn()
            ev[i][j + 1].record(stream)
        flush_l2(flush)
    torch.cuda.synchronize()
    return [[ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)] for j in range(len(stages))]


def warm(stages, n, flush, sync=True):
    import torch
    for _ in range(n):
        for _, fn in stages:
            fn()
        flush_l2(flush)
    if sync:
        torch.cuda.synchronize()


def kernel_entry(p, name, ms, peaks, comp_sectors):
    """Per-kernel rates: no-reuse algorithmic rate and fraction, plus the compulsory-byte
    fraction for the gathering kernels."""
    b, wk = p.algorithmic(name)
    s = ms / 1e3
    if b == "hbm":
        out = {"ms": round(ms, 5), "GB/s": round(wk / s / 1e9, 1),
               "frac_hbm": round(wk / s / 1e9 / float(peaks["hbm_gbs"]), 4)}
        cb = p.compulsory(name, comp_sectors)
        if cb is not None:
            out["frac_hbm"] = round(wk / s / 1e9 / float(peaks["hbm_gbs"]), 4)
            out["frac_hbm_note"] = "no-reuse bytes (every addressed row from HBM): can exceed 1 under Zipf reuse"
            out["compulsory_bytes"] = cb
            out["GB/s_compulsory"] = round(cb / s / 1e9, 1)
            out["frac_hbm_compulsory"] = round(cb / s / 1e9 / float(peaks["hbm_gbs"]), 4)
        return out
    if b == "alu":
        return {"ms": round(ms, 5), "TFLOP/s": round(wk / s / 1e12, 1),
                "frac_fp32_ffma": round(wk / s / 1e12 / FP32_FFMA_TFLOPS, 4)}
    if b == "tensor_fp8":
        # FP8 peak = the measured bf16 peak x the nominal FP8 / bf16 ratio (4.5 / 2.25)
        return {"ms": round(ms, 5), "TFLOP/s": round(wk / s / 1e12, 1),
                "frac_tensor_fp8_burst": round(wk / s / 1e12 / (FP8_OVER_BF16 * float(peaks["bf16_tflops"])), 4),
                "frac_tensor_fp8_sustained": round(wk / s / 1e12 / (FP8_OVER_BF16 * float(
                    peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))), 4)}
    return {"ms": round(ms, 5), "TFLOP/s": round(wk / s / 1e12, 1),
            "frac_tensor_burst": round(wk / s / 1e12 / float(peaks["bf16_tflops"]), 4),
            "frac_tensor_sustained": round(wk / s / 1e12 / float(peaks.get("bf16_tflops_sustained",
                                                                            peaks["bf16_tflops"])), 4)}


def roofline_of(p, name, ms, peaks, peak_src, comp_sectors, cfg):
    """The roofline object of one kernel: achieved = its algorithmic bytes (compulsory
    bytes for the gathering kernels: distinct table sectors, IDs, e_t, epilogue operands)
    or flops per launch / its mean CUDA-event duration."""
    bound, work = p.algorithmic(name)
    s = ms / 1e3
    out = {"bound": bound, "kernel": name}
    if bound == "hbm":
        cb = p.compulsory(name, comp_sectors)
        byts = cb if cb is not None else work
        peak = float(peaks["hbm_gbs"])
        out.update(achieved=round(byts / s / 1e9, 2), peak=peak, unit="GB/s", frac=round(byts / s / 1e9 / peak, 4),
                   bytes_per_launch=byts,
                   basis=("compulsory bytes: distinct 32-byte table sectors + IDs + e_t + epilogue operands + W"
                          if cb is not None else "algorithmic bytes (each read and written once)"),
                   peak_source=f"{peak_src} (hbm_gbs: STREAM-style copy)")
        if cb is not None:
            out["achieved_no_reuse"] = round(work / s / 1e9, 2)
            out["frac_no_reuse"] = round(work / s / 1e9 / peak, 4)
    elif bound == "alu":
        achieved = work / s / 1e12
        out.update(achieved=round(achieved, 2), peak=round(FP32_FFMA_TFLOPS, 1), unit="TFLOP/s",
                   frac=round(achieved / FP32_FFMA_TFLOPS, 4),
                   peak_source="derived: 152 SMs x 128 FP32 lanes x 2 flop x 2.07 GHz")
    else:
        achieved = work / s / 1e12
        ratio = FP8_OVER_BF16 if bound == "tensor_fp8" else 1.0   # FP8: measured bf16 x nominal ratio
        sus = ratio * float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
        out.update(achieved=round(achieved, 2), peak=sus, unit="TFLOP/s", frac=round(achieved / sus, 4),
                   frac_burst=round(achieved / (ratio * float(peaks["bf16_tflops"])), 4),
                   peak_burst=ratio * float(peaks["bf16_tflops"]),
                   peak_source=f"{peak_src} (bf16_tflops_sustained: cuBLAS bf16 back to back under the power cap; "
                               "the kernel runs inside a step of several launches)")
    out["frac_nominal"] = round(out["achieved"] / NOMINAL_PEAK[bound], 4)
    out["traffic"] = traffic_of(cfg, name)
    return out


def measure_workload(cfg, args, dev, rank, world, steps, headline):
    """Times one workload's step (device-resident inputs), its alternative paths, the
    uniform-ID control, streaming decode and the end-to-end loop; returns a dict."""
    import torch
    from hashed_head_gram_gb300 import pg

    p = Pipeline(cfg, dev, rank)
    stream = torch.cuda.current_stream()
    flush = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    path = args.path if args.path in p.paths() else p.paths()[0]
    stages = p.stages(path)

    # ---- warm-up
    warm(stages, args.warmup, flush)
    if p.w.gate == p.W.GATE_CONTEXT:
        p.dn["H"].copy_(p.H0)
    torch.cuda.synchronize()

    # ---- device-timed loop: events around every stage of every step, L2 flushed between steps
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        # two more untimed steps, enqueued without a synchronisation, keep the device busy
        # from the sampler's start-up pause into the first timed step (its clocks up)
        warm(stages, 2, flush, sync=False)
        if p.w.gate == p.W.GATE_CONTEXT:
            p.dn["H"].copy_(p.H0)
        launches0 = pg.launch_count()
        t_wall = time.perf_counter()
        stage_ms = time_stages(stages, steps, stream, flush)
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    launches = pg.launch_count() - launches0
    step_ms = [sum(stage_ms[j][i] for j in range(len(stages))) for i in range(steps)]
    total_s = reduce_max(sum(step_ms) / 1e3, world)
    value = whole_job_rate(p.N * steps, world, total_s)

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
    e2e_steps = max(2, min(steps, 200))
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
    del res_hosts

    # ---- per-kernel rates and the roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    means = {name: statistics.mean(stage_ms[j]) for j, (name, _) in enumerate(stages)}
    dom = max(means, key=means.get)
    sectors = table_sector_bytes(p)
    kernels = {name: kernel_entry(p, name, ms, peaks, sectors) for name, ms in means.items()}
    roofline = roofline_of(p, dom, means[dom], peaks, peak_src, sectors, cfg)
    if dom != "gather_sign_concat" and "gather_sign_concat" in means:
        kernels["gather_sign_concat"]["roofline"] = roofline_of(p, "gather_sign_concat", means["gather_sign_concat"],
                                                                peaks, peak_src, sectors, cfg)
    rows_ref = None if args.quick else row_references(p, steps, flush)

    # ---- the other paths of this workload, each warmed up and timed over the same steps
    other = []
    for op in ([] if args.quick else p.paths()):
        if op == path:
            continue
        ost = p.stages(op)
        warm(ost, args.warmup, flush)
        o_ms = time_stages(ost, steps, stream, flush)
        om = {name: statistics.mean(o_ms[j]) for j, (name, _) in enumerate(ost)}
        other.append({"path": op, "ms_per_step": round(sum(om.values()), 5),
                      "kernels": {name: kernel_entry(p, name, ms, peaks, sectors) for name, ms in om.items()}})
    if p.w.gate == p.W.GATE_CONTEXT:
        p.dn["H"].copy_(p.H0)
    if rows_ref is not None:  # the gather kernel (default or two-kernel path) against its rows moved alone
        g_ms = means.get("gather_sign_concat")
        for op in other:
            if g_ms is None and "gather_sign_concat" in op["kernels"]:
                g_ms = op["kernels"]["gather_sign_concat"]["ms"]
        if g_ms is not None:
            rows_ref["gather_sign_concat_ms"] = round(g_ms, 5)
            rows_ref["gather_over_row_copy"] = round(g_ms / rows_ref["row_copy"]["ms"], 3)

    # ---- the no-reuse control: the same path on uniform IDs (Zipf workloads only)
    control = None
    if p.w.zipf_s is not None and not args.quick:
        zipf_tokens = p.tokens.clone()
        p.tokens.copy_(torch.from_numpy(p.W.make_tokens(p.w, rank=rank, uniform=True)).to(dev))
        warm(stages, args.warmup, flush)
        u_ms = time_stages(stages, steps, stream, flush)
        u_means = {name: statistics.mean(u_ms[j]) for j, (name, _) in enumerate(stages)}
        u_sectors = table_sector_bytes(p)
        control = {"ids": "i.i.d. uniform over the vocabulary (no reuse: the compulsory bytes approach the "
                          "algorithmic ones)", "ms_per_step": round(sum(u_means.values()), 5),
                   "tokens_per_s": round(whole_job_rate(p.N, world, reduce_max(sum(u_means.values()) / 1e3, world)), 1),
                   "kernels": {name: kernel_entry(p, name, ms, peaks, u_sectors) for name, ms in u_means.items()}}
        p.tokens.copy_(zipf_tokens)
        del zipf_tokens
        if p.w.gate == p.W.GATE_CONTEXT:
            p.dn["H"].copy_(p.H0)

    decode = []
    if p.w.dtype == p.W.DT_BF16 and not args.quick:
        for B in sorted({1, 4, p.w.B, 4096}):
            us = p.decode(B)
            entry = {"sequences": B, "us_per_step": round(us, 2), "tokens_per_s": round(B / us * 1e6, 1)}
            if B <= 8 and p.d % 8 == 0:
                one = p.decode(B, one_launch=True)
                entry.update({"one_launch_us_per_step": round(one, 2),
                              "one_launch_tokens_per_s": round(B / one * 1e6, 1)})
            decode.append(entry)
    if pg.device_error() != 0:
        raise RuntimeError(f"device error word set: {pg.device_error()}")

    out = {
        "value": round(value, 1), "unit": "tokens/s", "steps": steps, "ms_per_step": round(statistics.mean(step_ms), 5),
        "dtype": "f32" if p.w.dtype == p.W.DT_F32 else ("e4m3 projection operands, bf16 outputs" if path == "fp8"
                                                        else "bf16"),
        "config": workload_config(p.w, world),
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": f"{e2e_steps} steps pipelined: each uploads its inputs from pinned host memory and "
                       "reads its whole result back; uploads, kernels and read-backs of consecutive steps "
                       "overlap on three streams (double-buffered device tensors); no L2 flush (inputs "
                       "> L2 except the tiny workload)"},
        "gpu_launches": launches,
        "roofline": roofline,
        "kernels": kernels,
        "path": path,
        "other_paths": other,
        "uniform_ids_control": control,
        "rows_moved_alone": rows_ref,
        "decode": {"steps": decode,
                   "how": "streaming decode, one token per sequence and step, on the same table and weights "
                          "(decode lookup -> projection with N = sequences -> decode conv where the module has "
                          "one: us_per_step; up to 8 sequences also the whole step as one launch, "
                          "pg_decode_step: one_launch_us_per_step); 16 consecutive steps in one CUDA graph "
                          "replayed back to back, no L2 flush (table rows cold, W and the state warm, as in "
                          "serving); not part of value"},
        "clocks": clk.summary(),
        "wall_s_timed_loop": round(t_wall, 4),
    }
    del p, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def run_gpu(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", torch.cuda.current_device())

    head = measure_workload(args.config, args, dev, rank, world, args.steps, headline=True)
    extras = {}
    for cfg in args.extra:
        extras[str(cfg)] = measure_workload(cfg, args, dev, rank, world, max(args.steps, EXTRA_MIN_STEPS),
                                            headline=False)

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
            "data": "synthetic: seeded Zipf token IDs, int8/64 table values, N(0,0.02) weights, N(0,1) states",
            "config": head["config"], "e2e": head["e2e"], "gpu_launches": head["gpu_launches"],
            "roofline": head["roofline"], "clocks": head["clocks"],
        }
        for k in ("kernels", "path", "other_paths", "uniform_ids_control", "rows_moved_alone", "decode",
                  "wall_s_timed_loop"):
            line[k] = head[k]
        if extras:
            line["workloads"] = extras
            line["workloads_how"] = (f"the other workloads, each timed like the headline over max(steps, "
                                     f"{EXTRA_MIN_STEPS}) steps after the same warm-up; not part of value")
        if world == 1 and not args.no_cpu_baseline:
            cpu = cpu_baselines([args.config] + list(args.extra), args.cpu_seconds)
            line["cpu_baseline"] = cpu.get(args.config)
            for cfg in args.extra:
                extras[str(cfg)]["cpu_baseline"] = cpu.get(cfg)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ncu-measured DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum),
# keyed by (workload, stage), with the sha256 prefix of the kernel's source file followed by
# the csrc headers (sorted) at the time of the capture; reported only while those sources
# are unchanged (profiles/ holds the captures).
TRAFFIC = {
    (5, "gather_sign_concat"): ("pg_lookup.cu", "0aaf20a91f99f372", 143.618560e6),
    (5, "project_gate"): ("pg_project.cu", "6f3f8ef4a91dcf5d", 1058.875136e6),
    (5, "conv_residual"): ("pg_conv.cu", "7f5d18ad0d0a8728", 1466.197760e6),
    (2, "gather_project_gate"): ("pg_project.cu", "6f3f8ef4a91dcf5d", 406.578688e6),
    (4, "gather_sign_concat"): ("pg_lookup.cu", "0aaf20a91f99f372", 190.824960e6),
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


WORKLOAD_DESC = {
    1: "tiny fp32 PageGram table (P_n=64, K=8, S=4, r=64); 4096 uniform IDs over 1024; fp32 W_V 1024->256",
    2: "PageGram 200M-parameter bf16 table: P_n = 48,823 / 48,821 pages, K=8, S=4, r=64; Zipf(1.1) IDs over "
       "50,304; W_V 1024->768; scalar gate g=0.5",
    3: "Engram-style 200M-parameter bf16 table: 16 prime subtables ~195k rows, r=64; same tokens as the PageGram "
       "200M workload; W_V 1024->768; scalar gate g=0.5",
    4: "20B-parameter PageGram table in NF4 (34-byte rows, 10.6 GB): P_n = 4,882,811 / 4,882,789, K=8, S=4; "
       "Zipf(1.05) over 128,000 IDs folded to 98,010; gather + NF4 dequant + sign + concat",
    5: "Engram-27B-shaped module: 16 prime subtables ~2.2266M rows, r=80, bf16 (5.7 GB); Zipf(1.05) over 128k "
       "with canonical folding; fused W_V + 4 W_K (1280 -> 12800); RMSNorm-sigmoid gate; causal depthwise conv "
       "k=4 dilation 3 + SiLU + residual into 4 branches of d=2560",
}


def workload_config(w, world):
    t = w.tables[0]
    return {"workload": f"{w.name} (config {w.cfg_id}): {WORKLOAD_DESC.get(w.cfg_id, w.name)}",
            "batch": f"{w.B}x{w.L}", "tokens_per_gpu": w.N,
            "table_bytes": t.table_bytes, "parallelism": f"dp{world} (independent batches, no collective)",
            "l2": "flushed between timed steps (256 MiB written, then read back, untimed); "
                  "table and activations > L2"}


# ---------------------------------------------------------------- CPU oracle legs
#
# The oracle, as it stands, on the host cores: every stage of the path over a bounded
# sample of a workload (the first n tokens of its batch: the prefix of the first sequence,
# or whole sequences), each stage timed on its own. With T threads the sample is split
# into T contiguous token ranges run concurrently (the C stages and numpy's fp64 kernels
# release the GIL; BLAS is held to one thread per range); the conv's ranges start 9
# positions early so every output sees its full causal window.

def host_cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return None


class OracleLeg:
    """Inputs of one workload's CPU leg, prepared once; run() times one pass."""

    TABLE_MATERIALISE_BYTES = 1 << 30

    def __init__(self, cfg: int, threads: int):
        import numpy as np
        import torch

        from hashed_head_gram_gb300 import workloads as W
        from oracle import dense, oracle as orc

        self.np, self.W, self.orc, self.dense = np, W, orc, dense
        w = self.w = W.make_workload(cfg)
        self.spec = w.tables[0]
        self.threads = threads
        self.tokens = W.make_tokens(w)
        self.cmap = W.make_canon_map(w)
        self.pool = None
        if threads > 1:
            from concurrent.futures import ThreadPoolExecutor
            self.pool = ThreadPoolExecutor(threads)
        spec = self.spec
        if spec.table_bytes <= self.TABLE_MATERIALISE_BYTES:
            t = W.make_table(w, spec, "cpu")
            self.table = t.view(torch.uint8).reshape(spec.table_rows, spec.row_bytes).numpy()
            self.table_note = "the whole table in host memory"
        else:
            self.table = None
            self.table_note = ("the sample's distinct rows in a compact host table (row ids remapped between the "
                               "index and gather stages, untimed): the full table does not fit the leg")
        self.dn_t = W.make_dense(w, "cpu")
        self.n = 0

    def prepare(self, n: int):
        """Sample = the first n tokens (n <= L: a prefix of sequence 0; else whole sequences)."""
        np, w = self.np, self.w
        n = max(1, min(n, w.N))
        if n > w.L:
            n = n // w.L * w.L
        self.n = n
        self.nseq = (n + w.L - 1) // w.L
        self.tok = np.ascontiguousarray(self.tokens[:self.nseq])
        parts = np.array_split(np.arange(n, dtype=np.int64), self.threads)
        self.which = [p for p in parts if len(p)]
        if self.table is None:
            _, rows, _, _ = self.orc.index(self.spec, self.tok, self.cmap, self.w.vocab, np.arange(n, dtype=np.int64))
            flat = rows.reshape(-1)
            self.uniq = np.unique(flat[flat != self.orc.NO_ROW])
            rng = np.random.default_rng(self.w.cfg_id)
            rb = self.spec.row_bytes
            if self.spec.row_dtype == self.W.DT_NF4:
                ct = rng.integers(0, 256, (len(self.uniq), rb), dtype=np.uint8)
                sc = (1.0 + rng.integers(0, 1024, len(self.uniq)) / 1024.0).astype(np.float16).view(np.uint8)
                ct[:, 32:34] = sc.reshape(-1, 2)
            else:
                q = rng.integers(-128, 128, (len(self.uniq), self.spec.r)).astype(np.float32) / 64
                bits = q.view(np.uint32) if self.spec.row_dtype == self.W.DT_F32 else \
                    (q.view(np.uint32) >> 16).astype(np.uint16)
                ct = np.ascontiguousarray(bits).view(np.uint8).reshape(len(self.uniq), rb)
            self.compact = ct
        dn, M, d = self.dn_t, w.M, w.d
        self.Wd = dn["W"].double().numpy()
        if "x" in dn:
            self.x = dn["x"][:n].double().numpy()
        if "H" in dn:
            self.H = dn["H"][:, :n].double().numpy()
            self.gh, self.gk = dn["gamma_h"].double().numpy(), dn["gamma_k"].double().numpy()
            self.gc, self.cw = dn["gamma_c"].double().numpy(), dn["conv_w"].double().numpy()
        return n

    def _map(self, fn, items):
        return list(self.pool.map(fn, items)) if self.pool is not None else [fn(x) for x in items]

    def run(self):
        """One pass of every stage over the sample; returns {stage: seconds}."""
        np, orc, dense, w, spec = self.np, self.orc, self.dense, self.w, self.spec
        t = {}
        t0 = time.perf_counter()
        idx = self._map(lambda wh: orc.index(spec, self.tok, self.cmap, w.vocab, wh), self.which)
        t["index"] = time.perf_counter() - t0
        rows = [r for (_, r, _, _) in idx]
        table = self.table
        if table is None:   # remap to the compact table (untimed: not the oracle's work)
            table = self.compact
            remapped = []
            for r in rows:
                rr = np.full(r.shape, orc.NO_ROW, np.uint32)
                ok = r != orc.NO_ROW
                rr[ok] = np.searchsorted(self.uniq, r[ok]).astype(np.uint32)
                remapped.append(rr)
            rows = remapped
        odt = orc.F32 if spec.row_dtype == self.W.DT_F32 else orc.BF16
        t0 = time.perf_counter()
        es = self._map(lambda a: orc.assemble(spec, a[0], orc.fetch_rows(table, a[0]), a[1][2], odt),
                       list(zip(rows, idx)))
        t["gather"] = time.perf_counter() - t0
        if w.cfg_id == 4:   # the lookup ends at e_t
            return t
        ctx = w.gate == self.W.GATE_CONTEXT

        def dense_part(a):
            e, wh = a
            ef = e.astype(np.float64) if odt == orc.F32 else orc.bf16_bits_to_f64(e)
            if w.gate == self.W.GATE_NONE:
                return dense.project(ef, self.Wd)
            if w.gate == self.W.GATE_SCALAR:
                return dense.scalar_gate(self.x[wh[0]:wh[-1] + 1], dense.project(ef, self.Wd), w.g)
            return dense.engram_gate(ef, self.Wd, self.H[:, wh[0]:wh[-1] + 1], self.gh, self.gk, w.eps, w.M)

        t0 = time.perf_counter()
        res = self._map(dense_part, list(zip(es, self.which)))
        t["project_gate"] = time.perf_counter() - t0
        if not ctx:
            return t
        v = np.concatenate([r[0] for r in res])
        alpha = np.concatenate([r[1] for r in res], axis=1)
        segs = conv_segments(self.n, w.L, self.threads, (w.conv_kernel - 1) * w.dilation)
        t0 = time.perf_counter()
        self._map(lambda sg: conv_range(dense, sg, v, alpha, self.gc, self.cw, w.dilation, w.eps, self.H), segs)
        t["conv"] = time.perf_counter() - t0
        return t


def conv_segments(n, L, threads, halo):
    """Token ranges for the conv over the first n flat tokens of sequences of length L:
    each sequence split into enough pieces for `threads` workers; (a0, a, b) = the piece
    [a, b) computed from a0 = max(sequence start, a - halo), so that every output in it
    sees its whole causal window."""
    import numpy as np
    nseq = (n + L - 1) // L
    per_seq = max(1, -(-threads // nseq))
    segs = []
    for s in range(nseq):
        lo, hi = s * L, min(n, (s + 1) * L)
        for piece in np.array_split(np.arange(lo, hi), per_seq):
            if len(piece):
                a = int(piece[0])
                segs.append((max(lo, a - halo), a, int(piece[-1]) + 1))
    return segs


def conv_range(dense, seg, v, alpha, gc, cw, dilation, eps, H):
    """The oracle's conv + residual over one (a0, a, b) range of flat tokens: H + Y at [a, b)."""
    a0, a, b = seg
    out = dense.conv_residual(v[a0:b][None], alpha[:, a0:b][:, None], gc, cw, dilation, eps, H[:, a0:b][:, None])
    return out[:, 0, a - a0:]


def _leg_summary(leg, passes, stat=statistics.median):
    """tokens/s per stage and for the whole path (per-token time = the sum of the stages')."""
    n = leg.n
    stages = {k: stat([p[k] for p in passes]) for k in passes[0]}
    total = sum(stages.values())
    return {"value": round(n / total, 1), "unit": "tokens/s", "threads": leg.threads,
            "stages_tokens_per_s": {k: round(n / s, 1) for k, s in stages.items()},
            "sample_tokens": n, "passes": len(passes), "seconds_per_pass": round(total, 3)}


def oracle_leg(cfg: int, threads: int, seconds: float):
    """Sized sample (about `seconds` per pass after a 64-token calibration), one warm pass,
    then the median of a few passes."""
    leg = OracleLeg(cfg, threads)
    leg.prepare(64 * threads)
    leg.run()
    cal = leg.run()
    per_tok = sum(cal.values()) / leg.n
    cap = 16384 if leg.w.gate == leg.W.GATE_CONTEXT else 65536
    leg.prepare(int(min(cap, max(64 * threads, seconds / max(per_tok, 1e-9)))))
    leg.run()
    passes = [leg.run() for _ in range(3)]
    out = _leg_summary(leg, passes)
    out["table"] = leg.table_note
    return out


def run_oracle_legs(args):
    """Child process of cpu_baselines(): BLAS is held to one thread by the environment the
    parent set before this interpreter started."""
    res = {}
    for cfg in [int(c) for c in args.oracle_legs.split(",")]:
        res[cfg] = oracle_leg(cfg, args.threads, args.cpu_seconds)
    print(json.dumps(res), flush=True)


def _one_thread_env(threads):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
              "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[k] = "1"
    env["PG_ORACLE_THREADS"] = str(threads)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    env["CUDA_VISIBLE_DEVICES"] = ""
    return env


def cpu_baselines(cfgs, seconds):
    """The oracle on the host cores for each workload, at 1 thread and at nproc threads, in
    child processes (BLAS threads fixed at start-up; no GPU)."""
    nproc = os.cpu_count() or 1
    model = host_cpu_model()
    out = {}
    legs = {}
    for threads in sorted({1, nproc}):
        cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--oracle-legs",
               ",".join(str(c) for c in cfgs), "--threads", str(threads), "--cpu-seconds", str(seconds)]
        r = subprocess.run(cmd, capture_output=True, text=True, env=_one_thread_env(threads), timeout=1800)
        if r.returncode != 0:
            raise RuntimeError(f"oracle leg failed ({threads} threads):\n{r.stderr[-3000:]}")
        legs[threads] = {int(k): v for k, v in json.loads(r.stdout.strip().splitlines()[-1]).items()}
    for cfg in cfgs:
        one, many = legs[1][cfg], legs[nproc][cfg]
        out[cfg] = {"value": many["value"], "unit": "tokens/s", "cores": nproc, "kind": "oracle",
                    "threads_1": one, "threads_nproc": many, "cpu_model": model,
                    "sample": (f"first {many['sample_tokens']} tokens of the workload batch ({one['sample_tokens']} "
                               f"at 1 thread); every stage of the path "
                               f"({', '.join(many['stages_tokens_per_s'])}) timed on its own, median of 3 passes, "
                               f"whole-path rate from the summed per-token times; {many['table']}")}
    return out


def run_reference(args):
    """The reference arm: the oracle as it stands on the host cores (nproc threads by
    default), one pass over a bounded sample of the workload per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    threads = args.threads or (os.cpu_count() or 1)
    leg = OracleLeg(args.config, threads)
    leg.prepare(64 * threads)
    leg.run()
    cal = leg.run()
    per_tok = sum(cal.values()) / leg.n
    budget = 90.0                                         # seconds for the warm-up and timed steps
    per_step = budget / (args.steps + args.warmup)
    cap = 16384 if leg.w.gate == leg.W.GATE_CONTEXT else 65536
    leg.prepare(int(min(cap, max(64, per_step / max(per_tok, 1e-9)))))
    for _ in range(args.warmup):
        leg.run()
    passes = [leg.run() for _ in range(args.steps)]
    total_t = sum(sum(p.values()) for p in passes)
    value = leg.n * args.steps / total_t
    summ = _leg_summary(leg, passes, stat=statistics.mean)
    from hashed_head_gram_gb300 import workloads as W
    w = W.make_workload(args.config)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_t / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (same seeded workload as the GPU arm)", "config": workload_config(w, 1),
            "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "cpu_model": host_cpu_model(), "stages_tokens_per_s": summ["stages_tokens_per_s"],
                             "sample": f"{leg.n} tokens per step (the first of the workload batch), every stage "
                                       f"of the path on {threads} threads; {leg.table_note}"},
            "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- single-kernel cases

def _kflush(buf):
    buf.add_(1)
    buf.sum(dtype=buf.dtype)  # read back: the written lines leave L2 here, not in the next launch


def _ktime(fn, iters: int, dev) -> float:
    """Median CUDA-event time (us) of fn over `iters` launches, L2 flushed between them."""
    import torch
    flush = torch.zeros(64 << 20, dtype=torch.int32, device=dev)
    for _ in range(3):
        fn()
        _kflush(flush)
    torch.cuda.synchronize()
    marks = []
    for _ in range(iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        _kflush(flush)
        marks.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in marks) * 1e3


def run_kernel_case(args):
    """One kernel at a time on a workload's shapes, through the C ABI exactly as the
    benchmark launches it (the conv and projection cases need no table, so they hold at
    most a few GB on the device). Prints the median time per launch and the rate."""
    import torch

    from hashed_head_gram_gb300 import pg, workloads as W

    dev = torch.device("cuda", torch.cuda.current_device())
    w = W.make_workload(args.config)
    spec = w.tables[0]
    g = torch.Generator(device=dev).manual_seed(12345)
    dt = torch.float32 if w.dtype == W.DT_F32 else torch.bfloat16
    code = pg.F32 if w.dtype == W.DT_F32 else pg.BF16
    N, din, d, M = w.N, spec.e_width, w.d, w.M
    kind = args.kernel
    if kind == "decode":
        _kernel_decode(w, args, dev, g)
        return
    if kind == "slots":
        _kernel_slots(args, dev, g)
        return
    if kind in ("gather", "gather_project"):
        if args.table_rows_scale < 1.0:
            spec = _scaled_spec(W, spec, args.table_rows_scale)
        desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
        tokens = torch.from_numpy(W.make_tokens(w)).to(dev)
        cm = W.make_canon_map(w)
        cm = None if cm is None else torch.from_numpy(cm.view("int32")).to(dev)
        table = W.make_table(w, spec, dev)
        e = torch.empty(N, din, dtype=dt, device=dev)
    if kind == "gather":
        us = _ktime(lambda: pg.gather_sign_concat(desc, tokens, table, e, code, canon_map=cm), args.iters, dev)
        rb = spec.row_bytes if spec.row_dtype != W.DT_NF4 else 64
        heads = 1 if spec.mode == W.MODE_FLAT else spec.K
        byts = N * (len(spec.orders) * heads * rb + 4 + din * e.element_size())
        print(f"gather_sign_concat config {w.cfg_id} (table {spec.table_bytes / 1e9:.2f} GB): {us:.1f} us, "
              f"{byts / us / 1e3:.0f} GB/s (no-reuse bytes)")
    elif kind == "nf4_export":
        x = torch.randn(args.rows, 64, device=dev, generator=g)
        out = torch.empty(args.rows, 34, dtype=torch.uint8, device=dev)
        us = _ktime(lambda: pg.nf4_quantize(x, out), args.iters, dev)
        byts = args.rows * (64 * 4 + 34)
        print(f"nf4_quantize {args.rows} rows: {us:.1f} us, {byts / us / 1e3:.0f} GB/s, {args.rows / us:.1f} M rows/s")
    elif kind == "gather_project":
        if w.gate != W.GATE_SCALAR:
            raise SystemExit("the one-launch case runs the scalar-gated workloads (configs 2, 3)")
        Wm = (torch.randn(d, din, device=dev, generator=g) * 0.02).to(dt)
        x = torch.randn(N, d, device=dev, generator=g).to(dt)
        v = torch.empty(N, d, dtype=dt, device=dev)
        ws = torch.empty(pg.gather_project_workspace_size(N, d, 0, pg.GATE_SCALAR) // 4 + 1, device=dev)
        us = _ktime(lambda: pg.gather_project_gate(desc, tokens, table, e, Wm, d, pg.GATE_SCALAR, v, ws, canon_map=cm,
                                                   g=w.g, x_resid=x), args.iters, dev)
        print(f"gather_project_gate config {w.cfg_id}: {us:.1f} us, {2.0 * N * din * d / us / 1e6:.1f} TFLOP/s, "
              f"{N / us:.1f} M tokens/s")
    elif kind == "project_fp8":
        e = (torch.randint(-128, 128, (N, din), device=dev, generator=g).float() / 64).to(torch.bfloat16)
        Wm = (torch.randn((1 + M) * d, din, device=dev, generator=g) * 0.02).to(torch.bfloat16)
        qe = torch.empty(N, din, dtype=torch.uint8, device=dev)
        se = torch.empty(N, device=dev)
        qw = torch.empty((1 + M) * d, din, dtype=torch.uint8, device=dev)
        sw = torch.empty((1 + M) * d, device=dev)
        pg.fp8_quantize(Wm, qw, sw)
        v = torch.empty(N, d, dtype=torch.bfloat16, device=dev)
        quant = lambda: pg.fp8_quantize(e, qe, se)
        quant()
        if w.gate == W.GATE_CONTEXT:
            H = torch.randn(M, N, d, device=dev, generator=g).to(torch.bfloat16)
            one = torch.ones(d, device=dev)
            alpha = torch.empty(M, N, device=dev)
            ws = torch.empty(pg.workspace_size(N, din, d, M, pg.BF16, pg.GATE_CONTEXT) // 4, device=dev)
            fn = lambda: pg.project_gate_fp8(qe, se, qw, sw, d, pg.GATE_CONTEXT, v, M=M, h=H, gamma_h=one,
                                             gamma_k=one, alpha_out=alpha, workspace=ws)
        else:
            x = torch.randn(N, d, device=dev, generator=g).to(torch.bfloat16)
            fn = lambda: pg.project_gate_fp8(qe, se, qw, sw, d, pg.GATE_SCALAR, v, g=w.g, x_resid=x)
        us = _ktime(fn, args.iters, dev)
        uq = _ktime(quant, args.iters, dev)
        print(f"project_gate_fp8 config {w.cfg_id}: {us:.1f} us, {2.0 * N * din * (1 + M) * d / us / 1e6:.1f} "
              f"TFLOP/s; fp8_quantize of e: {uq:.1f} us")
    elif kind == "project":
        e = (torch.randint(-128, 128, (N, din), device=dev, generator=g).float() / 64).to(dt)
        Wm = (torch.randn((1 + M) * d, din, device=dev, generator=g) * 0.02).to(dt)
        v = torch.empty(N, d, dtype=dt, device=dev)
        if w.gate == W.GATE_CONTEXT:
            H = torch.randn(M, N, d, device=dev, generator=g).to(dt)
            one = torch.ones(d, device=dev)
            alpha = torch.empty(M, N, device=dev)
            ws = torch.empty(pg.workspace_size(N, din, d, M, code, pg.GATE_CONTEXT) // 4, device=dev)
            fn = lambda: pg.project_gate(e, Wm, d, pg.GATE_CONTEXT, v, code, M=M, h=H, gamma_h=one, gamma_k=one,
                                         alpha_out=alpha, workspace=ws)
        elif w.gate == W.GATE_SCALAR:
            x = torch.randn(N, d, device=dev, generator=g).to(dt)
            fn = lambda: pg.project_gate(e, Wm, d, pg.GATE_SCALAR, v, code, g=w.g, x_resid=x)
        else:
            fn = lambda: pg.project_gate(e, Wm, d, pg.GATE_NONE, v, code)
        us = _ktime(fn, args.iters, dev)
        print(f"project_gate config {w.cfg_id}: {us:.1f} us, {2.0 * N * din * (1 + M) * d / us / 1e6:.1f} TFLOP/s")
    elif kind == "project_conv":
        if w.gate != W.GATE_CONTEXT:
            raise SystemExit("the projection + conv runs in the context-gated module (config 5)")
        e = (torch.randint(-128, 128, (N, din), device=dev, generator=g).float() / 64).to(dt)
        Wm = (torch.randn((1 + M) * d, din, device=dev, generator=g) * 0.02).to(dt)
        v = torch.empty(N, d, dtype=dt, device=dev)
        H = torch.randn(M, N, d, device=dev, generator=g).to(dt)
        one = torch.ones(d, device=dev)
        cw = torch.randn(d, w.conv_kernel, device=dev, generator=g) * 0.25
        alpha = torch.empty(M, N, device=dev)
        v_ms = torch.empty(N, device=dev)
        ws = torch.empty(pg.project_gate_conv_workspace_size(N, d, M) // 4 + 1, device=dev)
        us = _ktime(lambda: pg.project_gate_conv(w.B, w.L, e, Wm, d, M, H, one, one, one, cw, v, alpha, ws,
                                                 dilation=w.dilation, eps=w.eps, v_ms_out=v_ms), args.iters, dev)
        print(f"project_gate_conv config {w.cfg_id}: {us:.1f} us, {2.0 * N * din * (1 + M) * d / us / 1e6:.1f} "
              f"TFLOP/s (projection flops)")
    elif kind == "conv":
        if w.gate != W.GATE_CONTEXT:
            raise SystemExit("the conv runs in the context-gated module (config 5)")
        v = torch.randn(N, d, device=dev, generator=g).to(dt)
        alpha = torch.rand(M, N, device=dev, generator=g)
        gc = torch.ones(d, device=dev)
        cw = torch.randn(d, w.conv_kernel, device=dev, generator=g) * 0.25
        H = torch.randn(M, N, d, device=dev, generator=g).to(dt)
        v_ms = (v.float() ** 2).mean(dim=1)  # as the projection hands it over in the module
        us = _ktime(lambda: pg.conv_residual(w.B, w.L, d, M, code, v, alpha, gc, cw, H, dilation=w.dilation,
                                             eps=w.eps, v_ms=v_ms), args.iters, dev)
        byts = N * d * v.element_size() * (1 + 2 * M)
        print(f"conv_residual config {w.cfg_id}: {us:.1f} us, {byts / us / 1e3:.0f} GB/s")
    if pg.device_error() != 0:
        raise SystemExit("device error word set")


def _scaled_spec(W, spec, scale):
    """The workload's table with its page / subtable counts scaled down (same layout and
    row format): for captures that must hold only a few GB on the device."""
    import dataclasses
    if spec.mode == W.MODE_PAGEGRAM:
        return dataclasses.replace(spec, pages=W.largest_primes(int(spec.pages[0] * scale), len(spec.orders)))
    p = W.largest_primes(int(spec.rows[0][0] * scale), len(spec.orders) * spec.K)
    return dataclasses.replace(spec, rows=[p[i * spec.K:(i + 1) * spec.K] for i in range(len(spec.orders))])


def _kernel_decode(w, args, dev, g):
    """Streaming decode steps, one token per sequence: pg_decode_lookup, the projection
    (N = B) and, in the context-gated module, pg_decode_conv_residual. Timed per step
    (eager, L2 flushed between steps) and as a CUDA graph of 16 consecutive steps replayed
    back to back (the table rows stay cold, W and the state stay in L2 as in serving)."""
    import torch

    from hashed_head_gram_gb300 import pg, workloads as W

    spec = w.tables[0]
    if args.small_table:
        import dataclasses
        if spec.mode == W.MODE_PAGEGRAM:
            spec = dataclasses.replace(spec, pages=W.largest_primes(25000, len(spec.orders)))
        else:
            p = W.largest_primes(100000, len(spec.orders) * spec.K)
            spec = dataclasses.replace(spec, rows=[p[i * spec.K:(i + 1) * spec.K] for i in range(len(spec.orders))])
    d, M, din = w.d, w.M, spec.e_width
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    cm = W.make_canon_map(w)
    cm = None if cm is None else torch.from_numpy(cm.view("int32")).to(dev)
    table = W.make_table(w, spec, dev)
    Wm = (torch.randn((1 + M) * d, din, device=dev, generator=g) * 0.02).to(torch.bfloat16)
    steps = 16
    for B in [int(x) for x in args.batch.split(",")]:
        tokens = torch.randint(0, w.vocab, (steps, B), device=dev, generator=g, dtype=torch.int32)
        e = torch.empty(B, din, dtype=torch.bfloat16, device=dev)
        v = torch.empty(B, d, dtype=torch.bfloat16, device=dev)
        ctx = w.gate == W.GATE_CONTEXT
        state = pg.DecodeState(B, d=d if ctx else 0, M=M if ctx else 0, dtype=pg.BF16, kernel_size=w.conv_kernel,
                               dilation=w.dilation, device=dev)
        if ctx:
            H = torch.randn(M, B, d, device=dev, generator=g).to(torch.bfloat16)
            one = torch.ones(d, device=dev)
            cw = torch.randn(d, w.conv_kernel, device=dev, generator=g) * 0.25
            alpha = torch.empty(M, B, device=dev)
            v_ms = torch.empty(B, device=dev)
            ws = torch.empty(pg.workspace_size(B, din, d, M, pg.BF16, pg.GATE_CONTEXT) // 4 + 4, device=dev)
            calls = [
                lambda s: pg.decode_lookup(desc, state, tokens[s], table, e, pg.BF16, canon_map=cm),
                lambda s: pg.project_gate(e, Wm, d, pg.GATE_CONTEXT, v, pg.BF16, M=M, h=H, gamma_h=one, gamma_k=one,
                                          alpha_out=alpha, workspace=ws, v_ms_out=v_ms),
                lambda s: pg.decode_conv_residual(state, v, alpha, one, cw, H, eps=w.eps, v_ms=v_ms),
            ]
            names = ["decode_lookup", "project_gate(context)", "decode_conv_residual"]
        else:
            x = torch.randn(B, d, device=dev, generator=g).to(torch.bfloat16)
            gate = pg.GATE_SCALAR if w.gate == W.GATE_SCALAR else pg.GATE_NONE
            calls = [
                lambda s: pg.decode_lookup(desc, state, tokens[s], table, e, pg.BF16, canon_map=cm),
                lambda s: pg.project_gate(e, Wm, d, gate, v, pg.BF16, g=w.g,
                                          x_resid=x if gate == pg.GATE_SCALAR else None),
            ]
            names = ["decode_lookup", "project_gate"]
        step = lambda s=0: [c(s) for c in calls]
        eager = _ktime(step, args.iters, dev)
        parts = [_ktime(lambda c=c: c(0), args.iters, dev) for c in calls]
        side = torch.cuda.Stream(device=dev)
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
        reps = max(1, args.iters // 4)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            graph.replay()
        b.record()
        torch.cuda.synchronize()
        per_step = a.elapsed_time(b) * 1e3 / (reps * steps)
        if pg.device_error() != 0:
            raise SystemExit("device error word set")
        print(f"decode config {w.cfg_id} B={B}: eager step {eager:.1f} us "
              f"({' + '.join(f'{n} {u:.1f}' for n, u in zip(names, parts))}); "
              f"graph {per_step:.1f} us/step, {B / per_step:.3f} M tokens/s")
        if B <= 8:
            # the same step as one launch (pg_decode_step)
            ws1 = torch.zeros((pg.decode_step_workspace_size(B, d, M if ctx else 0) + 3) // 4, dtype=torch.int32,
                              device=dev)
            if ctx:
                one_call = lambda s: pg.decode_step(desc, state, tokens[s], table, Wm, d, pg.GATE_CONTEXT, v, ws1,
                                                    canon_map=cm, H=H, gamma_h=one, gamma_k=one, gamma_c=one,
                                                    conv_w=cw, eps=w.eps, alpha_out=alpha, v_ms_out=v_ms)
            else:
                one_call = lambda s: pg.decode_step(desc, state, tokens[s], table, Wm, d, gate, v, ws1, canon_map=cm,
                                                    g=w.g, x_resid=x if gate == pg.GATE_SCALAR else None)
            eager1 = _ktime(lambda: one_call(0), args.iters, dev)
            graph1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph1):
                for s in range(steps):
                    one_call(s)
            graph1.replay()
            torch.cuda.synchronize()
            a.record()
            for _ in range(reps):
                graph1.replay()
            b.record()
            torch.cuda.synchronize()
            per1 = a.elapsed_time(b) * 1e3 / (reps * steps)
            if pg.device_error() != 0:
                raise SystemExit("device error word set")
            print(f"decode config {w.cfg_id} B={B}: one launch (pg_decode_step) eager {eager1:.1f} us; "
                  f"graph {per1:.1f} us/step, {B / per1:.3f} M tokens/s")


def _kernel_slots(args, dev, g):
    """The PageGram report's slot sweep S in {1, 4, 8, 15, 60} on the PageGram 200M
    workload (bf16 table, P_n chosen so the budget stays fixed): the lookup and the
    one-launch lookup + projection timed per S, and the correlated-collision statistic
    (pg_collision_counts over 4M distinct bigrams) next to its (K - 1) / S expectation."""
    import torch

    from hashed_head_gram_gb300 import pg, workloads as W

    w = W.make_workload(2)
    tokens = torch.from_numpy(W.make_tokens(w)).to(dev)
    N, d = w.N, w.d
    e = torch.empty(N, 1024, dtype=torch.bfloat16, device=dev)
    Wm = (torch.randn(d, 1024, device=dev, generator=g) * 0.02).to(torch.bfloat16)
    x = torch.randn(N, d, device=dev, generator=g).to(torch.bfloat16)
    v = torch.empty(N, d, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(pg.gather_project_workspace_size(N, d, 0, pg.GATE_SCALAR) // 4 + 1, device=dev)
    n = 4_000_000
    for S in W.SLOT_SWEEP:
        spec = W.pagegram_slots(S)
        desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
        table = W.make_table(w, spec, dev)
        ug = _ktime(lambda: pg.gather_sign_concat(desc, tokens, table, e, pg.BF16), args.iters, dev)
        uf = _ktime(lambda: pg.gather_project_gate(desc, tokens, table, e, Wm, d, pg.GATE_SCALAR, v, ws, g=w.g,
                                                   x_resid=x), args.iters, dev)
        grams = torch.from_numpy(W.distinct_ngrams(n, 2, w.vocab, seed=100 + S)).to(dev)
        rows = torch.empty(2 * n, 2, spec.K, dtype=torch.int32, device=dev)
        pg.canon_hash(desc, grams, rows)
        span = spec.pages[0] * spec.K * S
        cws = torch.empty(pg.collision_workspace_size(n, span), dtype=torch.uint8, device=dev)
        counts = torch.empty(spec.K, dtype=torch.int64, device=dev)
        uc = _ktime(lambda: pg.collision_counts(rows.view(-1)[2 * spec.K:], n, spec.K, 4 * spec.K, 0, span, counts,
                                                cws), 3, dev)
        c = counts.cpu().tolist()
        del table
        if pg.device_error() != 0:
            raise SystemExit("device error word set")
        print(f"S={S:2d} P_n={spec.pages}: gather {ug:.1f} us ({N / ug:.0f} M tok/s), gather+project one launch "
              f"{uf:.1f} us ({N / uf:.0f} M tok/s); collisions over {n} bigrams: {c[0]} head-0 pairs, "
              f"extra shared heads {sum(c[1:]) / max(c[0], 1):.4f} (K-1)/S = {7 / S:.4f}; counted in {uc:.0f} us")


# ---------------------------------------------------------------- entry

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", type=int, default=5, choices=list(ALL_WORKLOADS),
                    help="the headline workload (default 5, the Engram-27B-shaped module)")
    ap.add_argument("--workloads", default="all",
                    help="'all' (the headline and the other four) or a comma list of workloads to measure besides "
                         "the headline ('none' for the headline alone)")
    ap.add_argument("--path", choices=["auto", "overlap", "two_kernel", "fused", "fp8", "conv_fused"], default="auto",
                    help="how the lookup and the projection run: overlap = one launch writing e_t with the "
                         "gather on extra warps of the projection (pg_gather_project_gate); two_kernel = "
                         "pg_gather_sign_concat + pg_project_gate; fused = pg_lookup_project_gate (r = 64 bf16 "
                         "tables); fp8 = pg_gather_sign_concat_e4m3 + pg_project_gate_fp8 (E4M3 operands); auto = "
                         "the first bf16 path that applies, in that order. The others that apply are timed too "
                         "and reported as other_paths")
    ap.add_argument("--cpu-seconds", type=float, default=1.0,
                    help="CPU oracle legs: seconds of work per timed pass")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="the default path only (no other paths, uniform-ID control or decode): for profiler captures")
    ap.add_argument("--threads", type=int, default=0, help="reference arm: host threads (default: all cores)")
    ap.add_argument("--oracle-legs", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--kernel", choices=["gather", "project", "project_fp8", "project_conv", "gather_project", "conv",
                                         "nf4_export",
                                         "decode", "slots"], default=None,
                    help="time one kernel on the workload's shapes instead of the benchmark")
    ap.add_argument("--iters", type=int, default=20, help="--kernel: timed launches")
    ap.add_argument("--batch", default="1,16,256,4096", help="--kernel decode: sequences per step (comma list)")
    ap.add_argument("--small-table", action="store_true",
                    help="--kernel decode: the table with ~100k-row subtables / pages (for ncu captures)")
    ap.add_argument("--table-rows-scale", type=float, default=1.0,
                    help="--kernel gather / gather_project: scale the table's pages / subtable rows (for ncu "
                         "captures of a few GB)")
    ap.add_argument("--rows", type=int, default=8 << 20, help="--kernel nf4_export: fp32 head rows to export")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.oracle_legs:
        run_oracle_legs(args)
        return
    if args.kernel:
        run_kernel_case(args)
        return
    if args.workloads == "all":
        args.extra = [c for c in ALL_WORKLOADS if c != args.config]
    elif args.workloads == "none":
        args.extra = []
    else:
        args.extra = [int(c) for c in args.workloads.split(",") if int(c) != args.config]
    if args.impl == "reference":
        if not os.environ.get("PG_ORACLE_THREADS"):
            # one BLAS thread per token range: the environment must be set before numpy loads
            env = _one_thread_env(args.threads or (os.cpu_count() or 1))
            for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
                      "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS"):
                os.environ[k] = env[k]
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
