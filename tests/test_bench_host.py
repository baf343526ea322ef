"""bench.py's host-side bookkeeping (no GPU): the recorded per-kernel DRAM traffic is
reported only while the kernel's sources are the ones it was captured on, and the
roofline peaks it divides by."""
import json
import os
import shutil

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_is_reported_only_for_the_captured_sources(tmp_path, monkeypatch):
    (cfg, stage), (src, sha, nbytes) = next(iter(bench.TRAFFIC.items()))
    now = bench.source_sha(src)
    assert len(now) == 16 and all(c in "0123456789abcdef" for c in now)
    assert bench.traffic_of(cfg, stage) == (nbytes if now == sha else None)
    assert bench.traffic_of(99, "no such stage") is None
    # a changed header changes every kernel's hash: the figure is withdrawn
    csrc = os.path.join(ROOT, "hashed_head_gram_gb300", "csrc")
    copy = tmp_path / "repo"
    shutil.copytree(csrc, copy / "hashed_head_gram_gb300" / "csrc")
    monkeypatch.setattr(bench, "ROOT", str(copy))
    assert bench.source_sha(src) == now
    hdr = copy / "hashed_head_gram_gb300" / "csrc" / "pg_internal.cuh"
    hdr.write_text(hdr.read_text() + "\n// changed\n")
    assert bench.source_sha(src) != now
    monkeypatch.setitem(bench.TRAFFIC, (cfg, stage), (src, now, nbytes))   # captured on the old sources
    assert bench.traffic_of(cfg, stage) is None


def test_peaks_measured_and_nominal():
    peaks, where = bench.load_peaks()
    assert float(peaks["hbm_gbs"]) > 1000 and float(peaks["bf16_tflops"]) > 100
    assert bench.NOMINAL_PEAK["hbm"] == 7900.0 and bench.NOMINAL_PEAK["tensor"] == 2250.0
    assert abs(bench.NOMINAL_PEAK["alu"] - 152 * 128 * 2 * 2.07e9 / 1e12) < 1e-9


def test_whole_job_rate_counts_every_rank():
    assert bench.whole_job_rate(1000, 1, 2.0) == 500.0
    assert bench.whole_job_rate(1000, 4, 2.0) == 2000.0


def test_oracle_conv_ranges_reproduce_the_whole_sequences():
    # the CPU leg splits the conv over token ranges that start `halo` positions early;
    # stitched together they equal the oracle's conv over whole sequences
    import numpy as np
    from oracle import dense
    rng = np.random.default_rng(3)
    L, nseq, d, M, dil, k = 37, 3, 16, 2, 3, 4
    n = L * nseq
    v = rng.standard_normal((n, d))
    alpha = rng.random((M, n))
    H = rng.standard_normal((M, n, d))
    gc, cw = rng.random(d) + 0.5, rng.standard_normal((d, k)) * 0.25
    ref = dense.conv_residual(v.reshape(nseq, L, d), alpha.reshape(M, nseq, L), gc, cw, dil, 1e-6,
                              H.reshape(M, nseq, L, d)).reshape(M, n, d)
    for threads in (1, 2, 5, 16):
        segs = bench.conv_segments(n, L, threads, (k - 1) * dil)
        covered = np.concatenate([np.arange(a, b) for _, a, b in segs])
        assert (np.sort(covered) == np.arange(n)).all()
        got = np.zeros_like(ref)
        for sg in segs:
            got[:, sg[1]:sg[2]] = bench.conv_range(dense, sg, v, alpha, gc, cw, dil, 1e-6, H)
        assert np.allclose(got, ref, rtol=0, atol=1e-12)
    # a prefix of one sequence (n < L)
    segs = bench.conv_segments(20, L, 4, (k - 1) * dil)
    assert segs[0] == (0, 0, 5) and all(a0 == max(0, a - 9) for a0, a, _ in segs)


def test_reference_arm_prints_one_contract_line():
    # `bench.py --impl reference` times the CPU oracle on the headline workload and prints one
    # JSON line with the GPU arm's metric, unit and direction, and no host<->device bytes
    import subprocess
    import sys
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["higher_is_better"] is True and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["config"]["workload"].startswith("engram27b-module-bf16")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
