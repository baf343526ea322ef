"""pg_lookup_project_gate (gather fused into the tcgen05 projection): bit-identical to
pg_gather_sign_concat followed by pg_project_gate, and within tolerance of the oracle."""
import dataclasses

import numpy as np
import pytest
import torch

from hashed_head_gram_gb300 import workloads as W
from oracle import dense
from oracle import oracle as orc
from tests._helpers import BF16_TOL, canon_tensor, oracle_e, rel_l2, shrink_table, to_f64

pytestmark = pytest.mark.gpu


def _pg():
    from hashed_head_gram_gb300 import pg
    return pg


def _two_call(pg, desc, spec, tok, table, cm, Wd, d, gate, dn, M=0, ws=None):
    N = tok.numel()
    e = torch.empty(N, spec.e_width, dtype=torch.bfloat16, device=tok.device)
    pg.gather_sign_concat(desc, tok, table, e, pg.BF16, canon_map=cm)
    v = torch.empty(N, d, dtype=torch.bfloat16, device=tok.device)
    alpha = torch.empty(max(M, 1), N, device=tok.device)
    pg.project_gate(e, Wd, d, gate, v, pg.BF16, M=M, g=0.5, x_resid=dn.get("x"), h=dn.get("H"),
                    gamma_h=dn.get("gamma_h"), gamma_k=dn.get("gamma_k"), alpha_out=alpha if M else None,
                    workspace=ws)
    return e, v, alpha


def _fused(pg, desc, tok, table, cm, Wd, d, gate, dn, M=0, ws=None, err=None):
    N = tok.numel()
    v = torch.empty(N, d, dtype=torch.bfloat16, device=tok.device)
    alpha = torch.empty(max(M, 1), N, device=tok.device)
    pg.lookup_project_gate(desc, tok, table, Wd, d, gate, v, canon_map=cm, M=M, g=0.5, x_resid=dn.get("x"),
                           h=dn.get("H"), gamma_h=dn.get("gamma_h"), gamma_k=dn.get("gamma_k"),
                           alpha_out=alpha if M else None, workspace=ws, err_index=err)
    return v, alpha


@pytest.mark.parametrize("cfg,ti,B,L", [(2, 0, 3, 143), (3, 0, 2, 200), (2, 0, 1, 64), (5, 0, 2, 150)])
def test_fused_scalar_and_none_gates_match_two_calls(cuda, cfg, ti, B, L):
    pg = _pg()
    w = W.shrink(W.make_workload(cfg), B=B, L=L)
    spec = shrink_table(w.tables[ti])
    if spec.r != 64:   # the Engram-27B table has r = 80: same tokens and map, r = 64 rows
        spec = dataclasses.replace(spec, r=64)
    d = 768
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    tokens = W.make_tokens(w)
    cmap = W.make_canon_map(w)
    table = W.make_table(w, spec, "cpu")
    g = torch.Generator().manual_seed(3)
    Wv = (torch.randn(d, spec.e_width, generator=g) * 0.02).to(torch.bfloat16)
    x = torch.randn(w.N, d, generator=g).to(torch.bfloat16)
    tok, tab, cm = torch.from_numpy(tokens).to(cuda), table.to(cuda), canon_tensor(cmap, cuda)
    dn = {"x": x.to(cuda)}
    for gate in (pg.GATE_SCALAR, pg.GATE_NONE):
        e, v2, _ = _two_call(pg, desc, spec, tok, tab, cm, Wv.to(cuda), d, gate, dn)
        err = torch.empty(1, dtype=torch.int32, device=cuda)
        v1, _ = _fused(pg, desc, tok, tab, cm, Wv.to(cuda), d, gate, dn, err=err)
        torch.cuda.synchronize()
        assert pg.device_error() == 0 and err.item() == -1
        assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))
    # and against the oracle (scalar gate)
    v1, _ = _fused(pg, desc, tok, tab, cm, Wv.to(cuda), d, pg.GATE_SCALAR, dn)
    ref_e = oracle_e(spec, tokens, cmap, w.vocab, table, orc.BF16)
    ref = dense.scalar_gate(x.double().numpy(), dense.project(orc.bf16_bits_to_f64(ref_e), Wv.double().numpy()), 0.5)
    assert rel_l2(to_f64(v1), ref) <= BF16_TOL


@pytest.mark.parametrize("d,M", [(256, 2), (384, 1)])
def test_fused_context_gate_matches_two_calls(cuda, d, M):
    pg = _pg()
    w = W.shrink(W.make_workload(2), B=2, L=150)
    spec = shrink_table(w.tables[0])
    desc = pg.table_desc(spec, w.vocab)
    tokens = W.make_tokens(w)
    table = W.make_table(w, spec, "cpu").to(cuda)
    g = torch.Generator().manual_seed(4)
    Wm = (torch.randn((1 + M) * d, spec.e_width, generator=g) * 0.02).to(torch.bfloat16).to(cuda)
    dn = {"H": torch.randn(M, w.N, d, generator=g).to(torch.bfloat16).to(cuda),
          "gamma_h": (torch.rand(d, generator=g) + 0.5).to(cuda), "gamma_k": (torch.rand(d, generator=g) + 0.5).to(cuda)}
    ws = torch.empty(pg.workspace_size(w.N, spec.e_width, d, M, pg.BF16, pg.GATE_CONTEXT) // 4, device=cuda)
    tok = torch.from_numpy(tokens).to(cuda)
    _, v2, a2 = _two_call(pg, desc, spec, tok, table, None, Wm, d, pg.GATE_CONTEXT, dn, M=M, ws=ws)
    v1, a1 = _fused(pg, desc, tok, table, None, Wm, d, pg.GATE_CONTEXT, dn, M=M, ws=ws)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16)) and torch.equal(a1, a2)


def test_fused_rejects_what_it_does_not_cover(cuda):
    pg = _pg()
    w = W.shrink(W.make_workload(3), B=1, L=32)
    x = torch.zeros(w.N, 768, dtype=torch.bfloat16, device=cuda)
    v = torch.empty_like(x)
    tok = torch.from_numpy(W.make_tokens(w)).to(cuda)
    flat = shrink_table(w.tables[1])                         # flat rows are 768 wide
    with pytest.raises(pg.PgError) as ex:
        pg.lookup_project_gate(pg.table_desc(flat, w.vocab), tok, W.make_table(w, flat, cuda),
                               torch.zeros(768, 768, dtype=torch.bfloat16, device=cuda), 768, pg.GATE_SCALAR, v,
                               g=0.5, x_resid=x)
    assert ex.value.status == 6
    w4 = W.shrink(W.make_workload(4), B=1, L=32)
    nf4 = shrink_table(w4.tables[0])
    with pytest.raises(pg.PgError) as ex:
        pg.lookup_project_gate(pg.table_desc(nf4, w4.vocab), torch.from_numpy(W.make_tokens(w4)).to(cuda),
                               W.make_table(w4, nf4, cuda), torch.zeros(768, 1024, dtype=torch.bfloat16, device=cuda),
                               768, pg.GATE_SCALAR, v, g=0.5, x_resid=x)
    assert ex.value.status == 6


def test_fused_reports_out_of_range_tokens(cuda):
    pg = _pg()
    w = W.shrink(W.make_workload(2), B=2, L=100)
    spec = shrink_table(w.tables[0])
    tokens = W.make_tokens(w).copy()
    tokens[1, 40] = w.vocab + 3
    d = 256
    dn = {"x": torch.zeros(w.N, d, dtype=torch.bfloat16, device=cuda)}
    err = torch.empty(1, dtype=torch.int32, device=cuda)
    _fused(pg, pg.table_desc(spec, w.vocab), torch.from_numpy(tokens).to(cuda), W.make_table(w, spec, cuda), None,
           torch.zeros(d, spec.e_width, dtype=torch.bfloat16, device=cuda), d, pg.GATE_SCALAR, dn, err=err)
    torch.cuda.synchronize()
    assert err.item() == 140


def test_fused_full_pagegram_200M_workload(cuda):
    pg = _pg()
    w = W.make_workload(2)
    spec = w.tables[0]
    desc = pg.table_desc(spec, w.vocab)
    tokens = W.make_tokens(w)
    tok = torch.from_numpy(tokens).to(cuda)
    table = W.make_table(w, spec, cuda)
    dn = W.make_dense(w, cuda)
    e, v2, _ = _two_call(pg, desc, spec, tok, table, None, dn["W"], w.d, pg.GATE_SCALAR, dn)
    v1, _ = _fused(pg, desc, tok, table, None, dn["W"], w.d, pg.GATE_SCALAR, dn)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))
    rng = np.random.default_rng(5)
    which = np.sort(rng.choice(w.N, 256, replace=False))
    ref_e = oracle_e(spec, tokens, None, w.vocab, table, orc.BF16, which=which)
    wi = torch.from_numpy(which).to(cuda)
    ref = dense.scalar_gate(to_f64(dn["x"][wi]), dense.project(orc.bf16_bits_to_f64(ref_e), to_f64(dn["W"])), w.g)
    assert rel_l2(to_f64(v1[wi]), ref) <= BF16_TOL
