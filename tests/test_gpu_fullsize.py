"""Full-size parity: every workload at its full batch and table size, run through
the same C-ABI calls the benchmark times; the oracle recomputes sampled tokens one
by one (bit-exact e_t, fp outputs within rel-L2)."""
import numpy as np
import pytest
import torch

from hashed_head_gram_gb300 import workloads as W
from oracle import dense
from oracle import oracle as orc
from tests._helpers import BF16_TOL, F32_TOL, bits16, canon_tensor, oracle_e, rel_l2, to_f64

pytestmark = pytest.mark.gpu


def _pg():
    from hashed_head_gram_gb300 import pg
    return pg


def _samples(w, n=96, seed=0):
    rng = np.random.default_rng(seed)
    t = np.concatenate([[0, 1, 2, 3, 8, 9, 10, w.L - 1], rng.integers(0, w.L, n - 8)])
    b = rng.integers(0, w.B, n)
    b[:8] = [0, 0, w.B - 1, 1 % w.B, 0, w.B - 1, 0, w.B - 1]
    return b.astype(np.int64), t.astype(np.int64)


def _gather(pg, w, spec, dev, out_dtype, table=None):
    tokens = W.make_tokens(w)
    cmap = W.make_canon_map(w)
    if table is None:
        table = W.make_table(w, spec, dev)
    e = torch.empty(w.N, spec.e_width, dtype=torch.float32 if out_dtype == orc.F32 else torch.bfloat16,
                    device=dev)
    err = torch.empty(1, dtype=torch.int32, device=dev)
    pg.gather_sign_concat(pg.table_desc(spec, w.vocab, w.canon_vocab), torch.from_numpy(tokens).to(dev), table,
                          e, out_dtype, canon_map=canon_tensor(cmap, dev), err_index=err)
    torch.cuda.synchronize()
    assert err.item() == -1
    return tokens, cmap, table, e


def test_full_config1_all_modes(cuda):
    pg = _pg()
    w = W.make_workload(1)
    Wv = W.make_dense(w, cuda)["W"]
    for spec in w.tables:
        tokens, cmap, table, e = _gather(pg, w, spec, cuda, orc.F32)
        ref = oracle_e(spec, tokens, cmap, w.vocab, table, orc.F32)
        assert np.array_equal(e.cpu().numpy().view(np.uint32), ref.view(np.uint32))
        if spec.mode == W.MODE_FLAT:
            continue       # flat rows are already d wide: no W_V
        v = torch.empty(w.N, w.d, device=cuda)
        pg.project_gate(e, Wv, w.d, pg.GATE_NONE, v, pg.F32)
        assert rel_l2(to_f64(v), dense.project(ref, to_f64(Wv))) <= F32_TOL


@pytest.mark.parametrize("cfg,ti", [(2, 0), (3, 0), (3, 1)])
def test_full_200M_tables_with_scalar_gate(cuda, cfg, ti):
    pg = _pg()
    w = W.make_workload(cfg)
    spec = w.tables[ti]
    tokens, cmap, table, e = _gather(pg, w, spec, cuda, orc.BF16)
    dn = W.make_dense(w, cuda)
    out = torch.empty(w.N, w.d, dtype=torch.bfloat16, device=cuda)
    Wv = None if spec.mode == W.MODE_FLAT else dn["W"]
    pg.project_gate(e, Wv, w.d, pg.GATE_SCALAR, out, pg.BF16, g=w.g, x_resid=dn["x"])
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    b, t = _samples(w)
    which = b * w.L + t
    ref_e = oracle_e(spec, tokens, cmap, w.vocab, table, orc.BF16, which=which)
    assert np.array_equal(bits16(e[torch.from_numpy(which).to(cuda)]), ref_e)
    ef = orc.bf16_bits_to_f64(ref_e)
    v_ref = ef if Wv is None else dense.project(ef, to_f64(Wv))
    x = to_f64(dn["x"][torch.from_numpy(which).to(cuda)])
    got = to_f64(out[torch.from_numpy(which).to(cuda)])
    assert rel_l2(got, dense.scalar_gate(x, v_ref, w.g)) <= BF16_TOL
    assert rel_l2(got - x, w.g * v_ref) <= BF16_TOL          # the memory term alone


def test_full_20B_nf4_gather(cuda):
    pg = _pg()
    w = W.make_workload(4)
    spec = w.tables[0]
    tokens, cmap, table, e = _gather(pg, w, spec, cuda, orc.BF16)
    b, t = _samples(w, n=512)
    which = b * w.L + t
    ref = oracle_e(spec, tokens, cmap, w.vocab, table, orc.BF16, which=which)
    assert np.array_equal(bits16(e[torch.from_numpy(which).to(cuda)]), ref)
    # no output row left unwritten: a second gather into a NaN-filled buffer agrees
    e2 = torch.full_like(e, float("nan"))
    pg.gather_sign_concat(pg.table_desc(spec, w.vocab, w.canon_vocab), torch.from_numpy(tokens).to(cuda),
                          table, e2, orc.BF16, canon_map=canon_tensor(cmap, cuda))
    assert torch.equal(e.view(torch.int16), e2.view(torch.int16))


def test_full_engram27b_module(cuda):
    pg = _pg()
    w = W.make_workload(5)
    spec = w.tables[0]
    tokens, cmap, table, e = _gather(pg, w, spec, cuda, orc.BF16)
    dn = W.make_dense(w, cuda)
    N, din, d, M = w.N, spec.e_width, w.d, w.M
    H = dn["H"]
    H0 = H.clone()
    v = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    alpha = torch.empty(M, N, device=cuda)
    v_ms = torch.empty(N, device=cuda)   # the module as the benchmark runs it: mean(v^2) handed over
    ws = torch.empty(pg.workspace_size(N, din, d, M, pg.BF16, pg.GATE_CONTEXT) // 4, device=cuda)
    pg.project_gate(e, dn["W"], d, pg.GATE_CONTEXT, v, pg.BF16, M=M, h=H, gamma_h=dn["gamma_h"],
                    gamma_k=dn["gamma_k"], eps=w.eps, alpha_out=alpha, workspace=ws, v_ms_out=v_ms)
    pg.conv_residual(w.B, w.L, d, M, pg.BF16, v, alpha, dn["gamma_c"], dn["conv_w"], H, dilation=w.dilation,
                     eps=w.eps, v_ms=v_ms)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    Wf = to_f64(dn["W"])
    got_H, ref_H, got_v, ref_v, got_a, ref_a = [], [], [], [], [], []
    for b, t in zip(*_samples(w, n=40)):
        t0 = max(0, t - 9)
        which = b * w.L + np.arange(t0, t + 1)
        ref_e = oracle_e(spec, tokens, cmap, w.vocab, table, orc.BF16, which=which)
        assert np.array_equal(bits16(e[torch.from_numpy(which).to(cuda)]), ref_e)
        wi = torch.from_numpy(which).to(cuda)
        h_win = to_f64(H0[:, wi])
        vv, aa = dense.engram_gate(orc.bf16_bits_to_f64(ref_e), Wf, h_win, to_f64(dn["gamma_h"]),
                                   to_f64(dn["gamma_k"]), w.eps, M)
        Hn = dense.conv_residual(vv[None], aa[:, None], to_f64(dn["gamma_c"]), to_f64(dn["conv_w"]), w.dilation,
                                 w.eps, h_win[:, None])
        got_H.append(to_f64(H[:, wi[-1]]))
        ref_H.append(Hn[:, 0, -1])
        got_v.append(to_f64(v[wi[-1]]))
        ref_v.append(vv[-1])
        got_a.append(to_f64(alpha[:, wi[-1]]))
        ref_a.append(aa[:, -1])
    assert rel_l2(np.stack(got_v), np.stack(ref_v)) <= BF16_TOL
    assert rel_l2(np.stack(got_a), np.stack(ref_a)) <= BF16_TOL
    assert rel_l2(np.stack(got_H), np.stack(ref_H)) <= BF16_TOL
    upd_g = np.stack(got_H) - np.stack([to_f64(H0[:, bb * w.L + tt]) for bb, tt in zip(*_samples(w, n=40))])
    upd_r = np.stack(ref_H) - np.stack([to_f64(H0[:, bb * w.L + tt]) for bb, tt in zip(*_samples(w, n=40))])
    assert rel_l2(upd_g, upd_r) <= 5e-2                       # the Y term alone
