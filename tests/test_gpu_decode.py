"""Streaming decode (one new token per sequence and call) against the full-sequence oracle.

A decode state carries each sequence's last canonical IDs and its last (k-1)*dil conv
inputs; position t of a decoded sequence must give what the oracle gives for position t
of the whole sequence (the causality pin makes that well defined). Lookups are compared
bit for bit, the dense chain within the bf16 / fp32 tolerances, and the decode conv bit
for bit against pg_conv_residual on the same inputs."""
import numpy as np
import pytest
import torch

from hashed_head_gram_gb300 import workloads as W
from oracle import dense
from oracle import oracle as orc
from tests._helpers import (BF16_TOL, F32_TOL, bits16, canon_tensor, oracle_e, rel_l2, shrink_table,
                            to_f64)

pytestmark = pytest.mark.gpu

CASES = [(cfg, i) for cfg in range(1, 6) for i in range(len(W.make_workload(cfg).tables))]


def _pg():
    from hashed_head_gram_gb300 import pg
    return pg


def _gen(seed):
    return torch.Generator().manual_seed(seed)


def _out_dtype(spec):
    return orc.F32 if spec.row_dtype == orc.F32 else orc.BF16


def _torch_dtype(code):
    return torch.float32 if code == orc.F32 else torch.bfloat16


def _same(got: torch.Tensor, ref: np.ndarray, code) -> bool:
    if code == orc.F32:
        return np.array_equal(got.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    return np.array_equal(bits16(got), ref)


def _decode_lookups(pg, desc, state, tokens_bt, table, code, cmap, cuda):
    """Runs T decode lookups over tokens [B, T]; returns e [T, B, width] on the GPU."""
    B, T = tokens_bt.shape
    tok = torch.from_numpy(np.ascontiguousarray(tokens_bt.T)).to(cuda)   # [T, B]
    out = []
    err = torch.empty(1, dtype=torch.int32, device=cuda)
    for t in range(T):
        e = torch.empty(B, _pg().table_geometry(desc)[2], dtype=_torch_dtype(code), device=cuda)
        pg.decode_lookup(desc, state, tok[t].contiguous(), table, e, code, canon_map=canon_tensor(cmap, cuda),
                         err_index=err)
        assert err.item() == -1
        out.append(e)
    return torch.stack(out)


@pytest.mark.parametrize("cfg,ti", CASES)
def test_decode_lookup_matches_the_oracle_at_every_position(cuda, cfg, ti):
    pg = _pg()
    B, T = 5, 11   # T > the 4-slot ID ring, so every slot is reused
    w = W.shrink(W.make_workload(cfg), B=B, L=T)
    spec = shrink_table(w.tables[ti])
    tokens, cmap = W.make_tokens(w), W.make_canon_map(w)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    table = W.make_table(w, spec, "cpu")
    code = _out_dtype(spec)
    ref = oracle_e(spec, tokens, cmap, w.vocab, table, code).reshape(B, T, -1)
    state = pg.DecodeState(B)
    e = _decode_lookups(pg, desc, state, tokens, table.to(cuda), code, cmap, cuda)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    for t in range(T):
        assert _same(e[t], np.ascontiguousarray(ref[:, t]), code), t
    assert (state.pos.cpu() == T).all()
    # the ID ring holds the canonical IDs of the last 4 positions, slot p mod 4
    canon = tokens if cmap is None else cmap[tokens].astype(np.int64)
    ids = state.ids.cpu().numpy().view(np.uint32)
    for p in range(T - 4, T):
        assert np.array_equal(ids[:, p % 4], canon[:, p].astype(np.uint32))


@pytest.mark.parametrize("cfg,ti", [(2, 0), (4, 0), (3, 0), (3, 1)])
def test_decode_lookup_f32_output_of_narrow_rows(cuda, cfg, ti):
    pg = _pg()
    B, T = 3, 6
    w = W.shrink(W.make_workload(cfg), B=B, L=T)
    spec = shrink_table(w.tables[ti])
    tokens, cmap = W.make_tokens(w), W.make_canon_map(w)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    table = W.make_table(w, spec, "cpu")
    ref = oracle_e(spec, tokens, cmap, w.vocab, table, orc.F32).reshape(B, T, -1)
    state = pg.DecodeState(B)
    e = _decode_lookups(pg, desc, state, tokens, table.to(cuda), orc.F32, cmap, cuda)
    for t in range(T):
        assert _same(e[t], np.ascontiguousarray(ref[:, t]), orc.F32)


def test_sequences_at_different_positions_and_restarts(cuda):
    # continuous batching: sequence 1 restarts at step 4, sequence 2 at step 7; each
    # restarted sequence must read as a fresh one (no IDs from before the restart)
    pg = _pg()
    B, T = 4, 12
    w = W.shrink(W.make_workload(2), B=B, L=T)
    spec = shrink_table(w.tables[0])
    tokens = W.make_tokens(w)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    table = W.make_table(w, spec, "cpu")
    tab = table.to(cuda)
    state = pg.DecodeState(B)
    restarts = {4: [1], 7: [2]}
    start = np.zeros(B, int)
    got = []
    for t in range(T):
        if t in restarts:
            pg.decode_reset(state, torch.tensor(restarts[t], dtype=torch.int32, device=cuda))
            for b in restarts[t]:
                start[b] = t
        e = torch.empty(B, spec.e_width, dtype=torch.bfloat16, device=cuda)
        pg.decode_lookup(desc, state, torch.from_numpy(tokens[:, t].copy()).to(cuda), tab, e, orc.BF16)
        got.append((e, start.copy()))
    torch.cuda.synchronize()
    for b in range(B):
        for t, (e, st) in enumerate(got):
            seq = tokens[b:b + 1, st[b]:t + 1]
            ref = oracle_e(spec, seq, None, w.vocab, table, orc.BF16)[-1]
            assert np.array_equal(bits16(e[b]), ref), (b, t)
    assert state.pos.cpu().tolist() == [T, T - 4, T - 7, T]


def test_reset_slot_out_of_range_is_reported(cuda):
    pg = _pg()
    state = pg.DecodeState(3)
    pg.device_error(clear=True)
    state.pos.fill_(5)
    pg.decode_reset(state, torch.tensor([2, 3, -1, 0], dtype=torch.int32, device=cuda))
    torch.cuda.synchronize()
    assert state.pos.cpu().tolist() == [0, 5, 0]
    assert pg.device_error(clear=True) == 256


def test_negative_position_is_reported_and_the_sequence_left_alone(cuda):
    pg = _pg()
    B = 3
    w = W.shrink(W.make_workload(2), B=B, L=1)
    spec = shrink_table(w.tables[0])
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    tab = W.make_table(w, spec, "cpu").to(cuda)
    state = pg.DecodeState(B, d=256, M=2)
    pg.device_error(clear=True)
    state.pos.copy_(torch.tensor([0, -7, 2], dtype=torch.int32))
    e = torch.full((B, spec.e_width), 3.0, dtype=torch.bfloat16, device=cuda)
    pg.decode_lookup(desc, state, torch.tensor([1, 2, 3], dtype=torch.int32, device=cuda), tab, e, orc.BF16)
    torch.cuda.synchronize()
    assert pg.device_error(clear=True) == 512
    assert (e[1].float() == 3.0).all() and not (e[0].float() == 3.0).all()
    assert state.pos.cpu().tolist() == [1, -7, 3]
    H = torch.randn(2, B, 256, generator=_gen(3)).to(torch.bfloat16).to(cuda)
    H0 = H.clone()
    v = torch.randn(B, 256, generator=_gen(4)).to(torch.bfloat16).to(cuda)
    pg.decode_conv_residual(state, v, torch.rand(2, B, device=cuda), torch.ones(256, device=cuda),
                            torch.randn(256, 4, device=cuda), H)
    torch.cuda.synchronize()
    assert pg.device_error(clear=True) == 512
    assert torch.equal(H[:, 1].view(torch.int16), H0[:, 1].view(torch.int16))
    assert not torch.equal(H[:, 0].view(torch.int16), H0[:, 0].view(torch.int16))
    assert state.pos.cpu().tolist() == [1, -7, 3]                  # the conv leaves pos alone
    # a conv before any lookup (pos 0: no consumed token) is reported the same way
    fresh = pg.DecodeState(B, d=256, M=2)
    pg.decode_conv_residual(fresh, v, torch.rand(2, B, device=cuda), torch.ones(256, device=cuda),
                            torch.randn(256, 4, device=cuda), H)
    torch.cuda.synchronize()
    assert pg.device_error(clear=True) == 512


def test_out_of_range_token_is_reported_and_read_as_id_0(cuda):
    pg = _pg()
    B = 4
    w = W.shrink(W.make_workload(2), B=B, L=2)
    spec = shrink_table(w.tables[0])
    tokens = W.make_tokens(w)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    table = W.make_table(w, spec, "cpu")
    state = pg.DecodeState(B)
    err = torch.empty(1, dtype=torch.int32, device=cuda)
    bad = tokens.copy()
    bad[2, 1] = w.vocab + 5
    bad[3, 1] = -1
    for t in range(2):
        e = torch.empty(B, spec.e_width, dtype=torch.bfloat16, device=cuda)
        pg.decode_lookup(desc, state, torch.from_numpy(bad[:, t].copy()).to(cuda), table.to(cuda), e, orc.BF16,
                         err_index=err)
    torch.cuda.synchronize()
    assert err.item() == 2
    fixed = bad.copy()
    fixed[2, 1] = 0
    fixed[3, 1] = 0
    ref = oracle_e(spec, fixed, None, w.vocab, table, orc.BF16).reshape(B, 2, -1)[:, 1]
    assert np.array_equal(bits16(e), np.ascontiguousarray(ref))


def test_decode_host_checks(cuda):
    pg = _pg()
    w = W.make_workload(2)
    spec = shrink_table(w.tables[0])
    desc = pg.table_desc(spec, w.vocab)
    lookup_only = pg.DecodeState(2)
    tab = W.make_table(w, spec, "cpu").to(cuda)
    e = torch.empty(2, spec.e_width, dtype=torch.bfloat16, device=cuda)
    with pytest.raises(pg.PgError) as ex:        # a conv call on a state without a conv part
        pg.decode_conv_residual(lookup_only, e[:, :256].contiguous(), torch.rand(1, 2, device=cuda),
                                torch.ones(256, device=cuda), torch.ones(256, 4, device=cuda),
                                torch.empty(1, 2, 256, dtype=torch.bfloat16, device=cuda))
    assert ex.value.status == 2
    toy = pg.table_desc(spec, w.vocab)
    toy.hash_kind = pg.HASH_TOY
    with pytest.raises(pg.PgError) as ex:
        pg.decode_lookup(toy, lookup_only, torch.zeros(2, dtype=torch.int32, device=cuda), tab, e, orc.BF16)
    assert ex.value.status in (2, 6)
    with pytest.raises(pg.PgError) as ex:        # a state whose ring depth disagrees with its conv
        st = pg.DecodeState(2, d=256, M=1)
        st.c.depth = 5
        pg.decode_conv_residual(st, e[:, :256].contiguous(), torch.rand(1, 2, device=cuda),
                                torch.ones(256, device=cuda), torch.ones(256, 4, device=cuda),
                                torch.empty(1, 2, 256, dtype=torch.bfloat16, device=cuda))
    assert ex.value.status == 2


def _conv_inputs(B, T, d, M, ks, seed, dtype):
    g = _gen(seed)
    v = torch.randn(B, T, d, generator=g).to(dtype)
    alpha = torch.rand(M, B, T, generator=g)
    gc = torch.rand(d, generator=g) + 0.5
    w = torch.randn(d, ks, generator=g) * 0.25
    H = torch.randn(M, B, T, d, generator=g).to(dtype)
    return v, alpha, gc, w, H


# (kernel 4, dilation 3) is the Engram notes' conv (ring depth 9); the others cover a
# 1-tap conv (no ring), dilation 1 and the deepest ring (3 * 8 = 24 positions)
@pytest.mark.parametrize("B,T,d,M,ks,dil,dtype", [
    (3, 14, 2560, 4, 4, 3, torch.bfloat16),
    (2, 30, 256, 2, 4, 8, torch.bfloat16),
    (4, 7, 64, 1, 2, 1, torch.float32),
    (1, 5, 8192, 3, 1, 3, torch.bfloat16),
    (2, 12, 768, 8, 3, 2, torch.float32),
    (2, 13, 256, 8, 4, 3, torch.bfloat16),     # 4 taps x (8 + 1) = 36 tap scalars per sequence
])
@pytest.mark.parametrize("given_ms", [False, True])
def test_decode_conv_is_bit_identical_to_the_full_conv(cuda, B, T, d, M, ks, dil, dtype, given_ms):
    pg = _pg()
    v, alpha, gc, w, H = _conv_inputs(B, T, d, M, ks, 60 + d, dtype)
    v_ms = (v.double() ** 2).mean(dim=2).float() if given_ms else None    # [B, T]
    Hf = H.reshape(M, B * T, d).contiguous().to(cuda)
    pg.conv_residual(B, T, d, M, pg.dtype_code(dtype), v.reshape(B * T, d).to(cuda),
                     alpha.reshape(M, B * T).contiguous().to(cuda), gc.to(cuda), w.to(cuda), Hf, dilation=dil,
                     v_ms=None if v_ms is None else v_ms.reshape(-1).to(cuda))
    state = pg.DecodeState(B, d=d, M=M, dtype=pg.dtype_code(dtype), kernel_size=ks, dilation=dil)
    assert state.c.depth == ((ks - 1) * dil + 1 if ks > 1 else 0)
    outs = []
    for t in range(T):
        Ht = H[:, :, t].contiguous().to(cuda)
        state.pos.fill_(t + 1)               # as the step's lookup leaves it: token t consumed
        pg.decode_conv_residual(state, v[:, t].contiguous().to(cuda), alpha[:, :, t].contiguous().to(cuda),
                                gc.to(cuda), w.to(cuda), Ht, eps=1e-6,
                                v_ms=None if v_ms is None else v_ms[:, t].contiguous().to(cuda))
        outs.append(Ht)
    torch.cuda.synchronize()
    Hf = Hf.reshape(M, B, T, d)
    view = torch.int16 if dtype == torch.bfloat16 else torch.int32
    for t in range(T):
        assert torch.equal(outs[t].view(view), Hf[:, :, t].view(view)), t
    assert (state.pos.cpu() == T).all()
    ref = dense.conv_residual(v.double().numpy(), alpha.double().numpy(), gc.double().numpy(), w.double().numpy(),
                              dil, 1e-6, H.double().numpy())
    got = np.stack([to_f64(o) for o in outs], axis=2)
    assert rel_l2(got, ref) <= (BF16_TOL if dtype == torch.bfloat16 else F32_TOL)


def _decode_context_step(pg, desc, state, tok_t, tab, Wm, d, M, H_t, gc, cw, cuda, ws):
    B = tok_t.numel()
    e = torch.empty(B, Wm.shape[1], dtype=torch.bfloat16, device=cuda)
    pg.decode_lookup(desc, state, tok_t, tab, e, orc.BF16)
    v = torch.empty(B, d, dtype=torch.bfloat16, device=cuda)
    alpha = torch.empty(M, B, device=cuda)
    v_ms = torch.empty(B, device=cuda)
    g1 = torch.ones(d, device=cuda)
    pg.project_gate(e, Wm, d, pg.GATE_CONTEXT, v, pg.BF16, M=M, h=H_t, gamma_h=g1, gamma_k=g1, alpha_out=alpha,
                    workspace=ws, v_ms_out=v_ms)
    pg.decode_conv_residual(state, v, alpha, gc, cw, H_t, v_ms=v_ms)
    return v, alpha


def test_decode_steps_of_the_engram_module_match_the_oracle(cuda):
    # the Engram-27B module's shapes (d = 2560, M = 4 branches, 2 x 8 heads of width 80,
    # kernel 4, dilation 3) on small prime subtables: lookup -> fused W_V + 4 W_K projection
    # and context gates -> conv + residual, one token per sequence and step
    pg = _pg()
    B, T = 3, 13
    w = W.shrink(W.make_workload(5), B=B, L=T)
    spec = shrink_table(w.tables[0])
    tokens = W.make_tokens(w)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    table = W.make_table(w, spec, "cpu")
    d, M = w.d, w.M
    Din = spec.e_width
    Wm = (torch.randn((1 + M) * d, Din, generator=_gen(70)) * 0.02).to(torch.bfloat16)
    H = torch.randn(M, B, T, d, generator=_gen(71)).to(torch.bfloat16)
    cw = torch.randn(d, 4, generator=_gen(72)) * 0.25
    gc = torch.ones(d)
    state = pg.DecodeState(B, d=d, M=M, dtype=pg.BF16)
    ws = torch.empty(pg.workspace_size(B, Din, d, M, pg.BF16, pg.GATE_CONTEXT) // 4 + 4, device=cuda)
    tab, Wd, gcd, cwd = table.to(cuda), Wm.to(cuda), gc.to(cuda), cw.to(cuda)
    vs, als, Hs = [], [], []
    for t in range(T):
        Ht = H[:, :, t].contiguous().to(cuda)
        v, alpha = _decode_context_step(pg, desc, state, torch.from_numpy(tokens[:, t].copy()).to(cuda), tab, Wd,
                                        d, M, Ht, gcd, cwd, cuda, ws)
        vs.append(v), als.append(alpha), Hs.append(Ht)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    e_ref = oracle_e(spec, tokens, None, w.vocab, table, orc.BF16)
    e_ref = orc.bf16_bits_to_f64(e_ref)                                   # [B*T, Din]
    v_ref, a_ref = dense.engram_gate(e_ref, Wm.double().numpy(), H.double().numpy().reshape(M, B * T, d),
                                     np.ones(d), np.ones(d), 1e-6, M)
    H_ref = dense.conv_residual(v_ref.reshape(B, T, d), a_ref.reshape(M, B, T), np.ones(d), cw.double().numpy(),
                                3, 1e-6, H.double().numpy())
    v_got = np.stack([to_f64(x) for x in vs], axis=1)                      # [B, T, d]
    a_got = np.stack([to_f64(x) for x in als], axis=2)                     # [M, B, T]
    H_got = np.stack([to_f64(x) for x in Hs], axis=2)                      # [M, B, T, d]
    assert rel_l2(v_got, v_ref.reshape(B, T, d)) <= BF16_TOL
    assert np.abs(a_got - a_ref.reshape(M, B, T)).max() < 2e-3
    assert rel_l2(H_got, H_ref) <= BF16_TOL
    upd = H_got - H.double().numpy()
    assert rel_l2(upd, H_ref - H.double().numpy()) <= 5e-2


def test_decode_steps_of_the_pagegram_scalar_path_match_the_oracle(cuda):
    # PageGram 200M shapes (2 x 8 heads of width 64, d = 768, g = 0.5) with NF4 and bf16
    # rows: lookup (advancing) -> W_V projection with the scalar gate x + g W_V e_t
    pg = _pg()
    for cfg in (2, 4):
        B, T = 4, 9
        w = W.shrink(W.make_workload(cfg), B=B, L=T)
        spec = shrink_table(w.tables[0])
        tokens = W.make_tokens(w)
        desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
        table = W.make_table(w, spec, "cpu")
        d, Din = 768, spec.e_width
        Wm = (torch.randn(d, Din, generator=_gen(80)) * 0.02).to(torch.bfloat16)
        x = torch.randn(B, T, d, generator=_gen(81)).to(torch.bfloat16)
        state = pg.DecodeState(B)
        tab, Wd = table.to(cuda), Wm.to(cuda)
        outs = []
        for t in range(T):
            e = torch.empty(B, Din, dtype=torch.bfloat16, device=cuda)
            pg.decode_lookup(desc, state, torch.from_numpy(tokens[:, t].copy()).to(cuda), tab, e, orc.BF16)
            out = torch.empty(B, d, dtype=torch.bfloat16, device=cuda)
            pg.project_gate(e, Wd, d, pg.GATE_SCALAR, out, pg.BF16, g=0.5, x_resid=x[:, t].contiguous().to(cuda))
            outs.append(out)
        torch.cuda.synchronize()
        e_ref = orc.bf16_bits_to_f64(oracle_e(spec, tokens, None, w.vocab, table, orc.BF16))
        ref = dense.scalar_gate(x.double().numpy().reshape(B * T, d), dense.project(e_ref, Wm.double().numpy()), 0.5)
        got = np.stack([to_f64(o) for o in outs], axis=1).reshape(B * T, d)
        assert rel_l2(got, ref) <= BF16_TOL, cfg
        assert (state.pos.cpu() == T).all()


@pytest.mark.parametrize("cfg", [2, 4, 5])
def test_decode_lookup_on_the_full_tables(cuda, cfg):
    # the full-size tables (PageGram 200M bf16, PageGram 20B NF4, Engram-27B bf16 with its
    # canonical folding), 4096 sequences per call at staggered positions: sequence b starts
    # lag = b mod 3 steps late (until then it is fed a filler token and restarted after the
    # step, so it stays empty); sampled sequences' e_t are checked bit for bit
    pg = _pg()
    w = W.make_workload(cfg)
    spec = w.tables[0]
    B, T = 4096, 5
    ww = W.shrink(w, B=B, L=T)
    tokens, cmap = W.make_tokens(ww), W.make_canon_map(ww)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    table = W.make_table(w, spec, cuda)
    state = pg.DecodeState(B)
    lag = np.arange(B) % 3
    cm = canon_tensor(cmap, cuda)
    err = torch.empty(1, dtype=torch.int32, device=cuda)
    outs = []
    for step in range(T + 2):
        t_of = step - lag
        tok = np.where((t_of >= 0) & (t_of < T), tokens[np.arange(B), np.clip(t_of, 0, T - 1)], 0).astype(np.int32)
        e = torch.empty(B, spec.e_width, dtype=torch.bfloat16, device=cuda)
        pg.decode_lookup(desc, state, torch.from_numpy(tok).to(cuda), table, e, orc.BF16, canon_map=cm, err_index=err)
        assert err.item() == -1
        idle = np.flatnonzero(t_of < 0).astype(np.int32)
        if idle.size:
            pg.decode_reset(state, torch.from_numpy(idle).to(cuda))
        outs.append(e)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    assert np.array_equal(state.pos.cpu().numpy(), T + 2 - lag)
    rng = np.random.default_rng(cfg)
    sample = np.concatenate([[0, 1, 2, B - 1, B - 2, B - 3], rng.integers(0, B, 42)])
    which = np.array([b * T + t for b in sample for t in range(T)], np.int64)
    ref = oracle_e(spec, tokens, cmap, w.vocab, table, orc.BF16, which=which).reshape(len(sample), T, -1)
    for i, b in enumerate(sample):
        for t in range(T):
            assert np.array_equal(bits16(outs[t + lag[b]][b]), ref[i, t]), (b, t)


@pytest.mark.parametrize("B", [2, 8])
def test_decode_steps_of_the_full_engram_module(cuda, B):
    # the Engram-27B module at full size (5.7 GB table, W 12,800 x 1,280) decoded the way
    # bench.py times it: 2 sequences take the few-rows projection, 8 the tensor-core one
    pg = _pg()
    w = W.make_workload(5)
    spec = w.tables[0]
    T = 5
    ww = W.shrink(w, B=B, L=T)
    tokens, cmap = W.make_tokens(ww), W.make_canon_map(ww)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    table = W.make_table(w, spec, cuda)
    dn = W.make_dense(ww, "cpu")
    d, M, Din = w.d, w.M, spec.e_width
    H = dn["H"].reshape(M, B, T, d)
    Wd, cw = dn["W"].to(cuda), dn["conv_w"].to(cuda)
    g1 = torch.ones(d, device=cuda)
    state = pg.DecodeState(B, d=d, M=M, dtype=pg.BF16)
    ws = torch.empty(pg.workspace_size(B, Din, d, M, pg.BF16, pg.GATE_CONTEXT) // 4 + 4, device=cuda)
    cm = canon_tensor(cmap, cuda)
    vs, als, Hs = [], [], []
    for t in range(T):
        e = torch.empty(B, Din, dtype=torch.bfloat16, device=cuda)
        pg.decode_lookup(desc, state, torch.from_numpy(tokens[:, t].copy()).to(cuda), table, e, orc.BF16, canon_map=cm)
        Ht = H[:, :, t].contiguous().to(cuda)
        v = torch.empty(B, d, dtype=torch.bfloat16, device=cuda)
        alpha = torch.empty(M, B, device=cuda)
        v_ms = torch.empty(B, device=cuda)
        pg.project_gate(e, Wd, d, pg.GATE_CONTEXT, v, pg.BF16, M=M, h=Ht, gamma_h=g1, gamma_k=g1, eps=w.eps,
                        alpha_out=alpha, workspace=ws, v_ms_out=v_ms)
        pg.decode_conv_residual(state, v, alpha, g1, cw, Ht, eps=w.eps, v_ms=v_ms)
        vs.append(v), als.append(alpha), Hs.append(Ht)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    e_ref = orc.bf16_bits_to_f64(oracle_e(spec, tokens, cmap, w.vocab, table, orc.BF16))       # [B*T, Din]
    v_ref, a_ref = dense.engram_gate(e_ref, dn["W"].double().numpy(), H.double().numpy().reshape(M, B * T, d),
                                     np.ones(d), np.ones(d), w.eps, M)
    H_ref = dense.conv_residual(v_ref.reshape(B, T, d), a_ref.reshape(M, B, T), np.ones(d),
                                dn["conv_w"].double().numpy(), w.dilation, w.eps, H.double().numpy())
    v_got = np.stack([to_f64(x) for x in vs], axis=1)
    a_got = np.stack([to_f64(x) for x in als], axis=2)
    H_got = np.stack([to_f64(x) for x in Hs], axis=2)
    assert rel_l2(v_got, v_ref.reshape(B, T, d)) <= BF16_TOL
    assert np.abs(a_got - a_ref.reshape(M, B, T)).max() < 2e-3
    assert rel_l2(H_got, H_ref) <= BF16_TOL
    assert rel_l2(H_got - H.double().numpy(), H_ref - H.double().numpy()) <= 5e-2
