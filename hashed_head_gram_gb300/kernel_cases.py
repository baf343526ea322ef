"""Single-kernel runs on a workload's shapes, for timing and profiling one kernel at a time.

    python -m hashed_head_gram_gb300.kernel_cases {gather,project,project_fp8,gather_project,conv,nf4_export,decode,slots} --config C [--iters N]

Inputs are synthetic and seeded (the conv and projection cases need no table, so they
hold at most a few GB on the device); each launch goes through the C ABI exactly as the
benchmark's. Prints the median CUDA-event time per launch (L2 flushed between launches,
untimed) and the achieved rate.
"""
from __future__ import annotations

import argparse
import statistics

import torch

from . import pg
from . import workloads as W


def _flush(buf):
    buf.add_(1)
    buf.sum(dtype=buf.dtype)  # read back: the written lines leave L2 here, not in the next launch


def _time(fn, iters: int, dev) -> float:
    flush = torch.zeros(64 << 20, dtype=torch.int32, device=dev)
    fn()
    _flush(flush)
    torch.cuda.synchronize()
    marks = []
    for _ in range(iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        _flush(flush)
        marks.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in marks) * 1e3


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("kernel", choices=["gather", "project", "project_fp8", "gather_project", "conv", "nf4_export",
                                       "decode", "slots"])
    ap.add_argument("--batch", default="1,16,256,4096", help="decode: sequences per step (comma list)")
    ap.add_argument("--small-table", action="store_true",
                    help="decode: the table with ~100k-row subtables / pages (for ncu captures)")
    ap.add_argument("--rows", type=int, default=8 << 20, help="nf4_export: fp32 head rows to export")
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--iters", type=int, default=20)
    args = ap.parse_args(argv)
    dev = torch.device("cuda", torch.cuda.current_device())
    w = W.make_workload(args.config)
    spec = w.tables[0]
    g = torch.Generator(device=dev).manual_seed(12345)
    dt = torch.float32 if w.dtype == W.DT_F32 else torch.bfloat16
    code = pg.F32 if w.dtype == W.DT_F32 else pg.BF16
    N, din, d, M = w.N, spec.e_width, w.d, w.M
    if args.kernel == "decode":
        _decode(w, args, dev, g)
        return
    if args.kernel == "slots":
        _slots(args, dev, g)
        return
    if args.kernel == "gather":
        desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
        tokens = torch.from_numpy(W.make_tokens(w)).to(dev)
        cm = W.make_canon_map(w)
        cm = None if cm is None else torch.from_numpy(cm.view("int32")).to(dev)
        table = W.make_table(w, spec, dev)
        e = torch.empty(N, din, dtype=dt, device=dev)
        us = _time(lambda: pg.gather_sign_concat(desc, tokens, table, e, code, canon_map=cm), args.iters, dev)
        rb = spec.row_bytes if spec.row_dtype != W.DT_NF4 else 64
        byts = N * (len(spec.orders) * spec.K * rb + 4 + din * e.element_size())
        print(f"gather_sign_concat config {w.cfg_id}: {us:.1f} us, {byts / us / 1e3:.0f} GB/s (algorithmic)")
    elif args.kernel == "nf4_export":
        # NF4 export of fp32 head rows (64 wide) into 34-byte rows (pg_nf4_quantize)
        x = torch.randn(args.rows, 64, device=dev, generator=g)
        out = torch.empty(args.rows, 34, dtype=torch.uint8, device=dev)
        us = _time(lambda: pg.nf4_quantize(x, out), args.iters, dev)
        byts = args.rows * (64 * 4 + 34)
        print(f"nf4_quantize {args.rows} rows: {us:.1f} us, {byts / us / 1e3:.0f} GB/s, {args.rows / us:.1f} M rows/s")
    elif args.kernel == "gather_project":
        # lookup + scalar-gated projection in one launch (pg_gather_project_gate)
        if w.gate != W.GATE_SCALAR:
            raise SystemExit("the one-launch case runs the scalar-gated workloads (configs 2, 3)")
        desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
        tokens = torch.from_numpy(W.make_tokens(w)).to(dev)
        cm = W.make_canon_map(w)
        cm = None if cm is None else torch.from_numpy(cm.view("int32")).to(dev)
        table = W.make_table(w, spec, dev)
        e = torch.empty(N, din, dtype=dt, device=dev)
        Wm = (torch.randn(d, din, device=dev, generator=g) * 0.02).to(dt)
        x = torch.randn(N, d, device=dev, generator=g).to(dt)
        v = torch.empty(N, d, dtype=dt, device=dev)
        ws = torch.empty(pg.gather_project_workspace_size(N, d, 0, pg.GATE_SCALAR) // 4 + 1, device=dev)
        us = _time(lambda: pg.gather_project_gate(desc, tokens, table, e, Wm, d, pg.GATE_SCALAR, v, ws, canon_map=cm,
                                                  g=w.g, x_resid=x), args.iters, dev)
        print(f"gather_project_gate config {w.cfg_id}: {us:.1f} us, {2.0 * N * din * d / us / 1e6:.1f} TFLOP/s, "
              f"{N / us:.1f} M tokens/s")
    elif args.kernel == "project_fp8":
        # the projection on E4M3 operands (pg_fp8_quantize of e and W, then pg_project_gate_fp8);
        # timed: the projection alone, and the quantisation of e that a step adds to it
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
        us = _time(fn, args.iters, dev)
        uq = _time(quant, args.iters, dev)
        print(f"project_gate_fp8 config {w.cfg_id}: {us:.1f} us, {2.0 * N * din * (1 + M) * d / us / 1e6:.1f} "
              f"TFLOP/s; fp8_quantize of e: {uq:.1f} us")
    elif args.kernel == "project":
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
        us = _time(fn, args.iters, dev)
        print(f"project_gate config {w.cfg_id}: {us:.1f} us, {2.0 * N * din * (1 + M) * d / us / 1e6:.1f} TFLOP/s")
    else:
        if w.gate != W.GATE_CONTEXT:
            raise SystemExit("the conv runs in the context-gated module (config 5)")
        v = torch.randn(N, d, device=dev, generator=g).to(dt)
        alpha = torch.rand(M, N, device=dev, generator=g)
        gc = torch.ones(d, device=dev)
        cw = torch.randn(d, w.conv_kernel, device=dev, generator=g) * 0.25
        H = torch.randn(M, N, d, device=dev, generator=g).to(dt)
        v_ms = (v.float() ** 2).mean(dim=1)  # as the projection hands it over in the module
        us = _time(lambda: pg.conv_residual(w.B, w.L, d, M, code, v, alpha, gc, cw, H, dilation=w.dilation,
                                            eps=w.eps, v_ms=v_ms), args.iters, dev)
        byts = N * d * v.element_size() * (1 + 2 * M)
        print(f"conv_residual config {w.cfg_id}: {us:.1f} us, {byts / us / 1e3:.0f} GB/s")


def _decode(w, args, dev, g):
    """Streaming decode steps, one token per sequence: pg_decode_lookup, the projection
    (N = B) and, in the context-gated module, pg_decode_conv_residual. Timed per step
    (eager, L2 flushed between steps) and as a CUDA graph of 16 consecutive steps replayed
    back to back (the table rows stay cold, W and the state stay in L2 as in serving)."""
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
        eager = _time(step, args.iters, dev)
        parts = [_time(lambda c=c: c(0), args.iters, dev) for c in calls]
        # a graph of `steps` consecutive steps
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
        print(f"decode config {w.cfg_id} B={B}: eager step {eager:.1f} us ({' + '.join(f'{n} {u:.1f}' for n, u in zip(names, parts))}); "
              f"graph {per_step:.1f} us/step, {B / per_step:.3f} M tokens/s")


def _slots(args, dev, g):
    """The PageGram report's slot sweep S in {1, 4, 8, 15, 60} on workload 2 (200M-parameter
    bf16 table, P_n chosen so the budget stays fixed): the lookup (pg_gather_sign_concat)
    and the one-launch lookup + projection (pg_gather_project_gate) timed per S, and the
    correlated-collision statistic (pg_collision_counts over 4M distinct bigrams) next to
    its (K - 1) / S expectation."""
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
        ug = _time(lambda: pg.gather_sign_concat(desc, tokens, table, e, pg.BF16), args.iters, dev)
        uf = _time(lambda: pg.gather_project_gate(desc, tokens, table, e, Wm, d, pg.GATE_SCALAR, v, ws, g=w.g,
                                                  x_resid=x), args.iters, dev)
        grams = torch.from_numpy(W.distinct_ngrams(n, 2, w.vocab, seed=100 + S)).to(dev)
        rows = torch.empty(2 * n, 2, spec.K, dtype=torch.int32, device=dev)
        pg.canon_hash(desc, grams, rows)
        span = spec.pages[0] * spec.K * S
        cws = torch.empty(pg.collision_workspace_size(n, span), dtype=torch.uint8, device=dev)
        counts = torch.empty(spec.K, dtype=torch.int64, device=dev)
        uc = _time(lambda: pg.collision_counts(rows.view(-1)[2 * spec.K:], n, spec.K, 4 * spec.K, 0, span, counts,
                                               cws), 3, dev)
        c = counts.cpu().tolist()
        del table
        if pg.device_error() != 0:
            raise SystemExit("device error word set")
        print(f"S={S:2d} P_n={spec.pages}: gather {ug:.1f} us ({N / ug:.0f} M tok/s), gather+project one launch "
              f"{uf:.1f} us ({N / uf:.0f} M tok/s); collisions over {n} bigrams: {c[0]} head-0 pairs, "
              f"extra shared heads {sum(c[1:]) / max(c[0], 1):.4f} (K-1)/S = {7 / S:.4f}; counted in {uc:.0f} us")


if __name__ == "__main__":
    main()
