"""pg_gather_project_gate (the lookup on extra warps of the tcgen05 projection, writing e_t
and the projection in one launch): e_t, v, alpha and mean(v^2) bit-identical to
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
    v_ms = torch.empty(N, device=tok.device)
    pg.project_gate(e, Wd, d, gate, v, pg.BF16, M=M, g=0.5, x_resid=dn.get("x"), h=dn.get("H"),
                    gamma_h=dn.get("gamma_h"), gamma_k=dn.get("gamma_k"), alpha_out=alpha if M else None,
                    workspace=ws, v_ms_out=v_ms if M else None)
    return e, v, alpha, v_ms


def _one_call(pg, desc, spec, tok, table, cm, Wd, d, gate, dn, M=0, err=None, ws=None):
    N = tok.numel()
    e = torch.full((N, spec.e_width), 7, dtype=torch.bfloat16, device=tok.device)  # every row overwritten
    v = torch.empty(N, d, dtype=torch.bfloat16, device=tok.device)
    alpha = torch.empty(max(M, 1), N, device=tok.device)
    v_ms = torch.empty(N, device=tok.device)
    if ws is None:
        ws = torch.empty(pg.gather_project_workspace_size(N, d, M, gate) // 4 + 1, device=tok.device)
    pg.gather_project_gate(desc, tok, table, e, Wd, d, gate, v, ws, canon_map=cm, M=M, g=0.5, x_resid=dn.get("x"),
                           h=dn.get("H"), gamma_h=dn.get("gamma_h"), gamma_k=dn.get("gamma_k"),
                           alpha_out=alpha if M else None, v_ms_out=v_ms if M else None, err_index=err)
    return e, v, alpha, v_ms


def _bits(t):
    return t.view(torch.int16)


def _case(cfg, ti, B, L):
    w = W.shrink(W.make_workload(cfg), B=B, L=L)
    spec = shrink_table(w.tables[ti])
    if spec.r != 64:   # the Engram-27B table has r = 80: same tokens and map, r = 64 rows
        spec = dataclasses.replace(spec, r=64)
    return w, spec


# (8, 128) and (9, 256): token counts that are whole multiples of the ready-counter unit
@pytest.mark.parametrize("cfg,ti,B,L", [(2, 0, 3, 143), (3, 0, 2, 200), (2, 0, 1, 64), (5, 0, 2, 150),
                                        (2, 0, 1, 5), (2, 0, 8, 128), (3, 0, 9, 256)])
def test_scalar_and_none_gates_match_two_calls(cuda, cfg, ti, B, L):
    pg = _pg()
    w, spec = _case(cfg, ti, B, L)
    d = 768
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    tokens = W.make_tokens(w)
    cmap = W.make_canon_map(w)
    table = W.make_table(w, spec, "cpu")
    g = torch.Generator().manual_seed(3)
    Wv = (torch.randn(d, spec.e_width, generator=g) * 0.02).to(torch.bfloat16).to(cuda)
    x = torch.randn(w.N, d, generator=g).to(torch.bfloat16)
    tok, tab, cm = torch.from_numpy(tokens).to(cuda), table.to(cuda), canon_tensor(cmap, cuda)
    dn = {"x": x.to(cuda)}
    for gate in (pg.GATE_SCALAR, pg.GATE_NONE):
        e2, v2, _, _ = _two_call(pg, desc, spec, tok, tab, cm, Wv, d, gate, dn)
        err = torch.empty(1, dtype=torch.int32, device=cuda)
        e1, v1, _, _ = _one_call(pg, desc, spec, tok, tab, cm, Wv, d, gate, dn, err=err)
        torch.cuda.synchronize()
        assert pg.device_error() == 0 and err.item() == -1
        assert torch.equal(_bits(e1), _bits(e2))
        assert torch.equal(_bits(v1), _bits(v2))
    # and against the oracle (scalar gate)
    e1, v1, _, _ = _one_call(pg, desc, spec, tok, tab, cm, Wv, d, pg.GATE_SCALAR, dn)
    ref_e = oracle_e(spec, tokens, cmap, w.vocab, table, orc.BF16)
    assert torch.equal(_bits(e1).cpu(), torch.from_numpy(ref_e.view(np.int16)).reshape(e1.shape))
    ref = dense.scalar_gate(x.double().numpy(), dense.project(orc.bf16_bits_to_f64(ref_e), to_f64(Wv)), 0.5)
    assert rel_l2(to_f64(v1), ref) <= BF16_TOL


# heads per token other than the workloads' 16 (units of 32 tokens x 16 rows): 2 heads give
# units of 128 tokens (256 rows), 12 and 24 units of 32 and 16 tokens (384 rows: the last
# gather warps of a unit have no rows), 32 units of 16 tokens (Din = 2048, the call's largest)
@pytest.mark.parametrize("mode,K,orders", [(W.MODE_PAGEGRAM, 1, [2, 3]), (W.MODE_PAGEGRAM, 4, [2, 3, 4]),
                                           (W.MODE_ENGRAM, 8, [1, 2, 3]), (W.MODE_PAGEGRAM, 16, [2, 3])])
def test_head_counts_other_than_sixteen(cuda, mode, K, orders):
    pg = _pg()
    w = W.shrink(W.make_workload(2), B=2, L=333)
    base = w.tables[0]
    if mode == W.MODE_PAGEGRAM:
        spec = dataclasses.replace(base, K=K, S=4, orders=list(orders), pages=[97, 89, 83][:len(orders)], rows=[])
    else:
        pr = W.largest_primes(1999, len(orders) * K)
        spec = dataclasses.replace(base, mode=W.MODE_ENGRAM, K=K, S=1, orders=list(orders), pages=[],
                                   rows=[pr[i * K:(i + 1) * K] for i in range(len(orders))])
    d = 256
    desc = pg.table_desc(spec, w.vocab)
    tokens = W.make_tokens(w)
    table = W.make_table(w, spec, "cpu")
    g = torch.Generator().manual_seed(5)
    Wv = (torch.randn(d, spec.e_width, generator=g) * 0.02).to(torch.bfloat16).to(cuda)
    x = torch.randn(w.N, d, generator=g).to(torch.bfloat16)
    tok, tab = torch.from_numpy(tokens).to(cuda), table.to(cuda)
    dn = {"x": x.to(cuda)}
    e2, v2, _, _ = _two_call(pg, desc, spec, tok, tab, None, Wv, d, pg.GATE_SCALAR, dn)
    err = torch.empty(1, dtype=torch.int32, device=cuda)
    e1, v1, _, _ = _one_call(pg, desc, spec, tok, tab, None, Wv, d, pg.GATE_SCALAR, dn, err=err)
    torch.cuda.synchronize()
    assert pg.device_error() == 0 and err.item() == -1
    assert torch.equal(_bits(e1), _bits(e2)) and torch.equal(_bits(v1), _bits(v2))
    ref_e = oracle_e(spec, tokens, None, w.vocab, table, orc.BF16)
    assert torch.equal(_bits(e1).cpu(), torch.from_numpy(ref_e.view(np.int16)).reshape(e1.shape))
    ref = dense.scalar_gate(x.double().numpy(), dense.project(orc.bf16_bits_to_f64(ref_e), to_f64(Wv)), 0.5)
    assert rel_l2(to_f64(v1), ref) <= BF16_TOL


@pytest.mark.parametrize("d,M", [(256, 2), (512, 1)])
def test_context_gate_matches_two_calls(cuda, d, M):
    pg = _pg()
    w, spec = _case(2, 0, 2, 150)
    desc = pg.table_desc(spec, w.vocab)
    tokens = W.make_tokens(w)
    table = W.make_table(w, spec, "cpu").to(cuda)
    g = torch.Generator().manual_seed(4)
    Wm = (torch.randn((1 + M) * d, spec.e_width, generator=g) * 0.02).to(torch.bfloat16).to(cuda)
    dn = {"H": torch.randn(M, w.N, d, generator=g).to(torch.bfloat16).to(cuda),
          "gamma_h": (torch.rand(d, generator=g) + 0.5).to(cuda), "gamma_k": (torch.rand(d, generator=g) + 0.5).to(cuda)}
    ws2 = torch.empty(pg.workspace_size(w.N, spec.e_width, d, M, pg.BF16, pg.GATE_CONTEXT) // 4, device=cuda)
    tok = torch.from_numpy(tokens).to(cuda)
    e2, v2, a2, m2 = _two_call(pg, desc, spec, tok, table, None, Wm, d, pg.GATE_CONTEXT, dn, M=M, ws=ws2)
    e1, v1, a1, m1 = _one_call(pg, desc, spec, tok, table, None, Wm, d, pg.GATE_CONTEXT, dn, M=M)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    assert torch.equal(_bits(e1), _bits(e2)) and torch.equal(_bits(v1), _bits(v2))
    assert torch.equal(a1[:M], a2[:M]) and torch.equal(m1, m2)


def test_workspace_reuse_gives_identical_results(cuda):
    # the call zeroes its ready and claim counters itself: back-to-back calls on one workspace
    pg = _pg()
    w, spec = _case(2, 0, 4, 256)
    desc = pg.table_desc(spec, w.vocab)
    tok = torch.from_numpy(W.make_tokens(w)).to(cuda)
    table = W.make_table(w, spec, cuda)
    d = 512
    g = torch.Generator().manual_seed(6)
    Wv = (torch.randn(d, spec.e_width, generator=g) * 0.02).to(torch.bfloat16).to(cuda)
    ws = torch.empty(pg.gather_project_workspace_size(w.N, d, 0, pg.GATE_NONE) // 4, device=cuda)
    outs = [_one_call(pg, desc, spec, tok, table, None, Wv, d, pg.GATE_NONE, {}, ws=ws) for _ in range(3)]
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    for e, v, _, _ in outs[1:]:
        assert torch.equal(_bits(e), _bits(outs[0][0])) and torch.equal(_bits(v), _bits(outs[0][1]))


def test_rejects_what_it_does_not_cover(cuda):
    pg = _pg()
    ws = torch.empty(1 << 16, device=cuda)

    def call(w, spec, d, Din, wsp=ws):
        tokens = torch.from_numpy(W.make_tokens(w)).to(cuda)
        e = torch.empty(tokens.numel(), Din, dtype=torch.bfloat16, device=cuda)
        v = torch.empty(tokens.numel(), d, dtype=torch.bfloat16, device=cuda)
        with pytest.raises(pg.PgError) as ex:
            pg.gather_project_gate(pg.table_desc(spec, w.vocab), tokens, W.make_table(w, spec, cuda), e,
                                   torch.zeros(d, Din, dtype=torch.bfloat16, device=cuda), d, pg.GATE_NONE, v, wsp)
        return ex.value.status

    w3 = W.shrink(W.make_workload(3), B=1, L=32)
    flat = shrink_table(w3.tables[1])                        # flat rows are 768 wide
    assert call(w3, flat, 768, flat.e_width) == 6
    w2 = W.shrink(W.make_workload(2), B=1, L=32)
    pagegram = shrink_table(w2.tables[0])
    assert call(w2, pagegram, 384, pagegram.e_width) == 6                              # d % 256 != 0
    assert call(w2, pagegram, 512, pagegram.e_width, wsp=torch.empty(4, device=cuda)) == 8   # workspace


def test_reports_out_of_range_tokens(cuda):
    pg = _pg()
    w, spec = _case(2, 0, 2, 100)
    tokens = W.make_tokens(w).copy()
    tokens[1, 40] = w.vocab + 3
    d = 256
    err = torch.empty(1, dtype=torch.int32, device=cuda)
    _one_call(pg, pg.table_desc(spec, w.vocab), spec, torch.from_numpy(tokens).to(cuda), W.make_table(w, spec, cuda),
              None, torch.zeros(d, spec.e_width, dtype=torch.bfloat16, device=cuda), d, pg.GATE_NONE, {}, err=err)
    torch.cuda.synchronize()
    assert err.item() == 140


@pytest.mark.parametrize("bad", [[(7, 5)], [(1, 100), (7, 5)], [(6, 0)]])
def test_reports_the_smallest_out_of_range_position(cuda, bad):
    # bad IDs in the last sequences of a batch of 8: the smallest flat position is reported
    pg = _pg()
    w, spec = _case(2, 0, 8, 128)
    tokens = W.make_tokens(w).copy()
    for b, t in bad:
        tokens[b, t] = w.vocab + 1 + t
    d = 256
    err = torch.empty(1, dtype=torch.int32, device=cuda)
    _one_call(pg, pg.table_desc(spec, w.vocab), spec, torch.from_numpy(tokens).to(cuda), W.make_table(w, spec, cuda),
              None, torch.zeros(d, spec.e_width, dtype=torch.bfloat16, device=cuda), d, pg.GATE_NONE, {}, err=err)
    torch.cuda.synchronize()
    assert err.item() == min(b * 128 + t for b, t in bad)


def test_full_pagegram_200M_workload(cuda):
    pg = _pg()
    w = W.make_workload(2)
    spec = w.tables[0]
    desc = pg.table_desc(spec, w.vocab)
    tokens = W.make_tokens(w)
    tok = torch.from_numpy(tokens).to(cuda)
    table = W.make_table(w, spec, cuda)
    dn = W.make_dense(w, cuda)
    e2, v2, _, _ = _two_call(pg, desc, spec, tok, table, None, dn["W"], w.d, pg.GATE_SCALAR, dn)
    e1, v1, _, _ = _one_call(pg, desc, spec, tok, table, None, dn["W"], w.d, pg.GATE_SCALAR, dn)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    assert torch.equal(_bits(e1), _bits(e2)) and torch.equal(_bits(v1), _bits(v2))
    rng = np.random.default_rng(5)
    which = np.sort(rng.choice(w.N, 256, replace=False))
    ref_e = oracle_e(spec, tokens, None, w.vocab, table, orc.BF16, which=which)
    wi = torch.from_numpy(which).to(cuda)
    assert torch.equal(_bits(e1[wi]).cpu(), torch.from_numpy(ref_e.view(np.int16)).reshape(len(which), -1))
    ref = dense.scalar_gate(to_f64(dn["x"][wi]), dense.project(orc.bf16_bits_to_f64(ref_e), to_f64(dn["W"])), w.g)
    assert rel_l2(to_f64(v1[wi]), ref) <= BF16_TOL
