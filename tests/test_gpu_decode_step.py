"""The one-launch decode step (pg_decode_step) against the full-sequence oracle and the
three-call decode step it replaces.

Position t of a sequence decoded one token per call must give what the oracle gives for
position t of the whole sequence: e_t bit for bit (the lookup is the decode lookup's own
code), v, alpha and the conv's update of H within the bf16 tolerance; against the three
calls (pg_decode_lookup, pg_project_gate, pg_decode_conv_residual) the state must advance
identically (pos, the ID ring) and the outputs agree to the rounding of their different
summation orders."""
import numpy as np
import pytest
import torch

from hashed_head_gram_gb300 import workloads as W
from oracle import dense
from oracle import oracle as orc
from tests._helpers import BF16_TOL, bits16, canon_tensor, oracle_e, rel_l2, shrink_table, to_f64

pytestmark = pytest.mark.gpu


def _pg():
    from hashed_head_gram_gb300 import pg
    return pg


def _gen(seed):
    return torch.Generator().manual_seed(seed)


def _workspace(pg, B, d, M, cuda):
    n = pg.decode_step_workspace_size(B, d, M)
    return torch.zeros((n + 3) // 4, dtype=torch.int32, device=cuda)


class Module:
    """The Engram-27B module's dense shapes (d = 2560, M = 4, kernel 4, dilation 3) with
    random gains, over a table spec and tokens [B, T]."""

    def __init__(self, w, spec, B, T, seed, cuda, table=None):
        self.w, self.spec, self.B, self.T = w, spec, B, T
        self.d, self.M, self.Din = w.d, w.M, spec.e_width
        d, M, Din = self.d, self.M, self.Din
        self.tokens = W.make_tokens(W.shrink(w, B=B, L=T))
        self.cmap = W.make_canon_map(W.shrink(w, B=B, L=T))
        self.table = table if table is not None else W.make_table(w, spec, "cpu")
        self.W = (torch.randn((1 + M) * d, Din, generator=_gen(seed)) * 0.02).to(torch.bfloat16)
        self.H = torch.randn(M, B, T, d, generator=_gen(seed + 1)).to(torch.bfloat16)
        self.gh = torch.rand(d, generator=_gen(seed + 2)) + 0.5
        self.gk = torch.rand(d, generator=_gen(seed + 3)) + 0.5
        self.gc = torch.rand(d, generator=_gen(seed + 4)) + 0.5
        self.cw = torch.randn(d, 4, generator=_gen(seed + 5)) * 0.25
        dev = lambda t: t.to(cuda)
        self.dW, self.dgh, self.dgk, self.dgc, self.dcw = map(dev, (self.W, self.gh, self.gk, self.gc, self.cw))
        self.dtab = self.table if self.table.is_cuda else self.table.to(cuda)
        self.dcm = canon_tensor(self.cmap, cuda)

    def oracle(self, which=None):
        B, T, d, M = self.B, self.T, self.d, self.M
        e_bits = oracle_e(self.spec, self.tokens, self.cmap, self.w.vocab, self.table, orc.BF16)
        e_ref = orc.bf16_bits_to_f64(e_bits)
        v_ref, a_ref = dense.engram_gate(e_ref, self.W.double().numpy(), self.H.double().numpy().reshape(M, B * T, d),
                                         self.gh.double().numpy(), self.gk.double().numpy(), self.w.eps, M)
        H_ref = dense.conv_residual(v_ref.reshape(B, T, d), a_ref.reshape(M, B, T), self.gc.double().numpy(),
                                    self.cw.double().numpy(), self.w.dilation, self.w.eps, self.H.double().numpy())
        return e_bits.reshape(B, T, -1), v_ref.reshape(B, T, d), a_ref.reshape(M, B, T), H_ref

    def run_step(self, pg, desc, cuda, graph_steps=0):
        """T one-launch steps; returns e [T, B, Din], v [T, B, d], alpha [T, M, B],
        v_ms [T, B], H [T, M, B, d] (each step's updated branch states) and the state."""
        B, T, d, M = self.B, self.T, self.d, self.M
        state = pg.DecodeState(B, d=d, M=M, dtype=pg.BF16)
        ws = _workspace(pg, B, d, M, cuda)
        tok = torch.from_numpy(np.ascontiguousarray(self.tokens.T)).to(cuda)
        e = torch.empty(T, B, self.Din, dtype=torch.bfloat16, device=cuda)
        v = torch.empty(T, B, d, dtype=torch.bfloat16, device=cuda)
        al = torch.empty(T, M, B, device=cuda)
        ms = torch.empty(T, B, device=cuda)
        H = self.H.permute(2, 0, 1, 3).contiguous().to(cuda)      # [T, M, B, d]
        err = torch.empty(1, dtype=torch.int32, device=cuda)

        def step(t):
            pg.decode_step(desc, state, tok[t], self.dtab, self.dW, d, pg.GATE_CONTEXT, v[t], ws, canon_map=self.dcm,
                           H=H[t], gamma_h=self.dgh, gamma_k=self.dgk, gamma_c=self.dgc, conv_w=self.dcw,
                           eps=self.w.eps, e_out=e[t], alpha_out=al[t], v_ms_out=ms[t],
                           err_index=None if graph_steps else err)
            if not graph_steps:
                assert err.item() == -1

        if graph_steps:
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(device=cuda)
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    for t in range(T):
                        step(t)
            torch.cuda.current_stream().wait_stream(side)
            g.replay()
        else:
            for t in range(T):
                step(t)
        torch.cuda.synchronize()
        assert ws[0].item() & 0x7FFFFFFF == 0              # the grid barrier's counter: only bit 31 flips
        return e, v, al, ms, H, state


@pytest.mark.parametrize("B", [1, 3, 8])
def test_decode_step_of_the_engram_module_matches_the_oracle(cuda, B):
    pg = _pg()
    T = 13                                   # > the ring depth (9) and the ID ring (4)
    w = W.make_workload(5)
    spec = shrink_table(w.tables[0])
    m = Module(w, spec, B, T, 90 + B, cuda)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    pg.device_error(clear=True)
    e, v, al, ms, H, state = m.run_step(pg, desc, cuda)
    assert pg.device_error() == 0
    e_ref, v_ref, a_ref, H_ref = m.oracle()
    for t in range(T):
        assert np.array_equal(bits16(e[t]), np.ascontiguousarray(e_ref[:, t])), t
    assert rel_l2(to_f64(v).transpose(1, 0, 2), v_ref) <= BF16_TOL
    assert np.abs(to_f64(al).transpose(1, 2, 0) - a_ref).max() < 2e-3
    v_got = to_f64(v).transpose(1, 0, 2)
    assert np.allclose(to_f64(ms).T, (v_got ** 2).mean(axis=2), rtol=1e-4, atol=0)
    H_got = to_f64(H).transpose(1, 2, 0, 3)                   # [M, B, T, d]
    H0 = m.H.double().numpy()
    assert rel_l2(H_got, H_ref) <= BF16_TOL
    assert rel_l2(H_got - H0, H_ref - H0) <= 5e-2
    assert (state.pos.cpu() == T).all()
    canon = m.tokens if m.cmap is None else m.cmap[m.tokens].astype(np.int64)
    ids = state.ids.cpu().numpy().view(np.uint32)
    for p in range(T - 4, T):
        assert np.array_equal(ids[:, p % 4], canon[:, p].astype(np.uint32))


def test_decode_step_agrees_with_the_three_call_step(cuda):
    # the same module stepped by pg_decode_lookup + pg_project_gate + pg_decode_conv_residual
    pg = _pg()
    B, T = 3, 12
    w = W.make_workload(5)
    spec = shrink_table(w.tables[0])
    m = Module(w, spec, B, T, 120, cuda)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    e1, v1, al1, ms1, H1, st1 = m.run_step(pg, desc, cuda)
    d, M = m.d, m.M
    st3 = pg.DecodeState(B, d=d, M=M, dtype=pg.BF16)
    ws = torch.empty(pg.workspace_size(B, m.Din, d, M, pg.BF16, pg.GATE_CONTEXT) // 4 + 4, device=cuda)
    tok = torch.from_numpy(np.ascontiguousarray(m.tokens.T)).to(cuda)
    for t in range(T):
        e = torch.empty(B, m.Din, dtype=torch.bfloat16, device=cuda)
        pg.decode_lookup(desc, st3, tok[t], m.dtab, e, orc.BF16, canon_map=m.dcm)
        assert torch.equal(e.view(torch.int16), e1[t].view(torch.int16)), t
        Ht = m.H[:, :, t].contiguous().to(cuda)
        v = torch.empty(B, d, dtype=torch.bfloat16, device=cuda)
        alpha = torch.empty(M, B, device=cuda)
        v_ms = torch.empty(B, device=cuda)
        pg.project_gate(e, m.dW, d, pg.GATE_CONTEXT, v, pg.BF16, M=M, h=Ht, gamma_h=m.dgh, gamma_k=m.dgk,
                        eps=w.eps, alpha_out=alpha, workspace=ws, v_ms_out=v_ms)
        pg.decode_conv_residual(st3, v, alpha, m.dgc, m.dcw, Ht, eps=w.eps, v_ms=v_ms)
        assert rel_l2(to_f64(v1[t]), to_f64(v)) < 1e-2, t
        assert (al1[t] - alpha).abs().max().item() < 1e-4, t
        assert rel_l2(to_f64(H1[t]), to_f64(Ht)) < 1e-2, t
    torch.cuda.synchronize()
    assert torch.equal(st1.pos, st3.pos) and torch.equal(st1.ids, st3.ids)
    assert pg.device_error() == 0


def test_decode_step_in_a_cuda_graph_is_bit_identical_to_eager(cuda):
    pg = _pg()
    B, T = 2, 10
    w = W.make_workload(5)
    spec = shrink_table(w.tables[0])
    m = Module(w, spec, B, T, 140, cuda)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    eager = m.run_step(pg, desc, cuda)
    graph = m.run_step(pg, desc, cuda, graph_steps=T)
    for a, b in zip(eager[:5], graph[:5]):
        assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                           b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16))
    assert torch.equal(eager[5].pos, graph[5].pos)


@pytest.mark.parametrize("cfg,ti,gate", [(2, 0, "scalar"), (4, 0, "scalar"), (3, 0, "none"), (3, 1, "none"),
                                         (2, 0, "none")])
def test_decode_step_scalar_and_no_gate_match_the_oracle(cuda, cfg, ti, gate):
    # PageGram bf16 and NF4 rows, Engram-style and flat rows: x + g W_V e_t (g = 0.5) or W_V e_t
    pg = _pg()
    B, T = 4, 9
    w = W.shrink(W.make_workload(cfg), B=B, L=T)
    spec = shrink_table(w.tables[ti])
    tokens, cmap = W.make_tokens(w), W.make_canon_map(w)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    table = W.make_table(w, spec, "cpu")
    d, Din = 768, spec.e_width
    Wm = (torch.randn(d, Din, generator=_gen(150 + cfg)) * 0.02).to(torch.bfloat16)
    x = torch.randn(B, T, d, generator=_gen(151)).to(torch.bfloat16)
    state = pg.DecodeState(B)
    ws = _workspace(pg, B, d, 0, cuda)
    tab, Wd, cm = table.to(cuda), Wm.to(cuda), canon_tensor(cmap, cuda)
    kind = pg.GATE_SCALAR if gate == "scalar" else pg.GATE_NONE
    outs, es = [], []
    for t in range(T):
        out = torch.empty(B, d, dtype=torch.bfloat16, device=cuda)
        e = torch.empty(B, Din, dtype=torch.bfloat16, device=cuda)
        pg.decode_step(desc, state, torch.from_numpy(tokens[:, t].copy()).to(cuda), tab, Wd, d, kind, out, ws,
                       canon_map=cm, g=0.5, x_resid=x[:, t].contiguous().to(cuda) if gate == "scalar" else None,
                       e_out=e)
        outs.append(out), es.append(e)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    e_bits = oracle_e(spec, tokens, cmap, w.vocab, table, orc.BF16)
    for t in range(T):
        assert np.array_equal(bits16(es[t]), np.ascontiguousarray(e_bits.reshape(B, T, -1)[:, t])), t
    v_ref = dense.project(orc.bf16_bits_to_f64(e_bits), Wm.double().numpy())
    ref = dense.scalar_gate(x.double().numpy().reshape(B * T, d), v_ref, 0.5) if gate == "scalar" else v_ref
    got = np.stack([to_f64(o) for o in outs], axis=1).reshape(B * T, d)
    assert rel_l2(got, ref) <= BF16_TOL
    assert (state.pos.cpu() == T).all()
    assert ws[0].item() & 0x7FFFFFFF == 0


@pytest.mark.parametrize("ks,dil", [(1, 3), (2, 1), (4, 8)])
def test_decode_step_conv_kernel_sizes(cuda, ks, dil):
    # no ring (kernel 1), the shortest ring and the deepest one (3 x 8 + 1 slots)
    pg = _pg()
    B, T = 2, 28 if dil == 8 else 8
    w = W.make_workload(5)
    spec = shrink_table(w.tables[0])
    m = Module(w, spec, B, T, 170 + ks, cuda)
    m.cw = m.cw[:, :ks].contiguous()
    m.dcw = m.cw.to(cuda)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    d, M = m.d, m.M
    state = pg.DecodeState(B, d=d, M=M, dtype=pg.BF16, kernel_size=ks, dilation=dil)
    ws = _workspace(pg, B, d, M, cuda)
    tok = torch.from_numpy(np.ascontiguousarray(m.tokens.T)).to(cuda)
    Hs, vs, als = [], [], []
    for t in range(T):
        Ht = m.H[:, :, t].contiguous().to(cuda)
        v = torch.empty(B, d, dtype=torch.bfloat16, device=cuda)
        al = torch.empty(M, B, device=cuda)
        pg.decode_step(desc, state, tok[t], m.dtab, m.dW, d, pg.GATE_CONTEXT, v, ws, canon_map=m.dcm, H=Ht,
                       gamma_h=m.dgh, gamma_k=m.dgk, gamma_c=m.dgc, conv_w=m.dcw, eps=w.eps, alpha_out=al)
        Hs.append(Ht), vs.append(v), als.append(al)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    e_bits = oracle_e(spec, m.tokens, m.cmap, w.vocab, m.table, orc.BF16)
    v_ref, a_ref = dense.engram_gate(orc.bf16_bits_to_f64(e_bits), m.W.double().numpy(),
                                     m.H.double().numpy().reshape(M, B * T, d), m.gh.double().numpy(),
                                     m.gk.double().numpy(), w.eps, M)
    H_ref = dense.conv_residual(v_ref.reshape(B, T, d), a_ref.reshape(M, B, T), m.gc.double().numpy(),
                                m.cw.double().numpy(), dil, w.eps, m.H.double().numpy())
    H_got = np.stack([to_f64(x) for x in Hs], axis=2)
    H0 = m.H.double().numpy()
    assert rel_l2(H_got, H_ref) <= BF16_TOL
    assert rel_l2(H_got - H0, H_ref - H0) <= 5e-2


def test_decode_step_negative_position_is_reported_and_the_sequence_left_alone(cuda):
    pg = _pg()
    B = 3
    w = W.make_workload(5)
    spec = shrink_table(w.tables[0])
    m = Module(w, spec, B, 1, 190, cuda)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    d, M = m.d, m.M
    state = pg.DecodeState(B, d=d, M=M, dtype=pg.BF16)
    state.pos.copy_(torch.tensor([0, -7, 2], dtype=torch.int32))
    ws = _workspace(pg, B, d, M, cuda)
    Ht = m.H[:, :, 0].contiguous().to(cuda)
    H0 = Ht.clone()
    v = torch.full((B, d), 3.0, dtype=torch.bfloat16, device=cuda)
    e = torch.full((B, m.Din), 3.0, dtype=torch.bfloat16, device=cuda)
    al = torch.full((M, B), 3.0, device=cuda)
    pg.device_error(clear=True)
    pg.decode_step(desc, state, torch.tensor([1, 2, 3], dtype=torch.int32, device=cuda), m.dtab, m.dW, d,
                   pg.GATE_CONTEXT, v, ws, canon_map=m.dcm, H=Ht, gamma_h=m.dgh, gamma_k=m.dgk, gamma_c=m.dgc,
                   conv_w=m.dcw, eps=w.eps, e_out=e, alpha_out=al)
    torch.cuda.synchronize()
    assert pg.device_error(clear=True) == 512
    assert state.pos.cpu().tolist() == [1, -7, 3]
    assert (v[1].float() == 3.0).all() and (e[1].float() == 3.0).all() and (al[:, 1] == 3.0).all()
    assert torch.equal(Ht[:, 1].view(torch.int16), H0[:, 1].view(torch.int16))
    assert not torch.equal(Ht[:, 0].view(torch.int16), H0[:, 0].view(torch.int16))
    assert not (v[0].float() == 3.0).all() and not (v[2].float() == 3.0).all()
    assert ws[0].item() & 0x7FFFFFFF == 0


def test_decode_step_host_checks(cuda):
    pg = _pg()
    w = W.make_workload(5)
    spec = shrink_table(w.tables[0])
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    d, M, Din = w.d, w.M, spec.e_width
    tab = W.make_table(w, spec, "cpu").to(cuda)
    Wd = torch.zeros((1 + M) * d, Din, dtype=torch.bfloat16, device=cuda)
    H = torch.zeros(M, 9, d, dtype=torch.bfloat16, device=cuda)
    g1 = torch.ones(d, device=cuda)
    cw = torch.ones(d, 4, device=cuda)
    v = torch.empty(9, d, dtype=torch.bfloat16, device=cuda)
    tok = torch.zeros(9, dtype=torch.int32, device=cuda)
    kw = dict(H=H, gamma_h=g1, gamma_k=g1, gamma_c=g1, conv_w=cw)
    with pytest.raises(pg.PgError) as ex:         # more sequences than one launch takes
        big = pg.DecodeState(9, d=d, M=M, dtype=pg.BF16)
        pg.decode_step(desc, big, tok, tab, Wd, d, pg.GATE_CONTEXT, v, _workspace(pg, 8, d, M, cuda), **kw)
    assert ex.value.status == 6
    st = pg.DecodeState(2, d=d, M=M, dtype=pg.BF16)
    small = torch.zeros(16, dtype=torch.int32, device=cuda)
    with pytest.raises(pg.PgError) as ex:         # workspace smaller than the size query says
        pg.decode_step(desc, st, tok[:2], tab, Wd, d, pg.GATE_CONTEXT, v[:2], small, **kw)
    assert ex.value.status == 8
    with pytest.raises(pg.PgError) as ex:         # context gate without its gains
        pg.decode_step(desc, st, tok[:2], tab, Wd, d, pg.GATE_CONTEXT, v[:2], _workspace(pg, 2, d, M, cuda), H=H)
    assert ex.value.status == 1
    with pytest.raises(pg.PgError) as ex:         # context gate on a state without a conv part
        pg.decode_step(desc, pg.DecodeState(2), tok[:2], tab, Wd, d, pg.GATE_CONTEXT, v[:2],
                       _workspace(pg, 2, d, M, cuda), **kw)
    assert ex.value.status == 2
    with pytest.raises(pg.PgError) as ex:         # width different from the state's
        pg.decode_step(desc, st, tok[:2], tab, Wd, d - 8, pg.GATE_CONTEXT, v[:2], _workspace(pg, 2, d, M, cuda),
                       **kw)
    assert ex.value.status == 2
    with pytest.raises(pg.PgError) as ex:         # scalar gate without its residual
        pg.decode_step(desc, pg.DecodeState(2), tok[:2], tab, Wd, d, pg.GATE_SCALAR, v[:2],
                       _workspace(pg, 2, d, 0, cuda))
    assert ex.value.status == 1
    torch.cuda.synchronize()
    assert pg.device_error() == 0


@pytest.mark.parametrize("B", [1, 4])
def test_decode_step_of_the_full_engram_module(cuda, B):
    # the full-size Engram-27B module (5.7 GB table, W 12,800 x 1,280, canonical folding),
    # the configuration bench.py times
    pg = _pg()
    w = W.make_workload(5)
    spec = w.tables[0]
    T = 5
    ww = W.shrink(w, B=B, L=T)
    table = W.make_table(w, spec, cuda)
    m = Module(w, spec, B, T, 200 + B, cuda, table=table)
    dn = W.make_dense(ww, "cpu")
    m.W, m.dW = dn["W"], dn["W"].to(cuda)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    e, v, al, ms, H, state = m.run_step(pg, desc, cuda)
    assert pg.device_error() == 0
    e_ref, v_ref, a_ref, H_ref = m.oracle()
    for t in range(T):
        assert np.array_equal(bits16(e[t]), np.ascontiguousarray(e_ref[:, t])), t
    assert rel_l2(to_f64(v).transpose(1, 0, 2), v_ref) <= BF16_TOL
    assert np.abs(to_f64(al).transpose(1, 2, 0) - a_ref).max() < 2e-3
    H_got = to_f64(H).transpose(1, 2, 0, 3)
    H0 = m.H.double().numpy()
    assert rel_l2(H_got, H_ref) <= BF16_TOL
    assert rel_l2(H_got - H0, H_ref - H0) <= 5e-2


def _layout_case(name):
    """Context-gate modules over other table layouts: e_t widths 768 (flat rows: 12 W boxes
    for 16 warps), 1024 (PageGram bf16 and NF4 rows: one box per warp) and 2048 (16 heads:
    two boxes per warp, the second refilling the first's slot)."""
    import dataclasses
    w5 = W.make_workload(5)
    if name == "pagegram_bf16":
        spec = shrink_table(W.make_workload(2).tables[0])
        return dataclasses.replace(w5, tables=[spec], d=512, M=2), spec
    if name == "pagegram_nf4":
        spec = shrink_table(W.make_workload(4).tables[0])
        return dataclasses.replace(w5, tables=[spec], d=768, M=3), spec
    if name == "flat_bf16":
        spec = shrink_table(W.make_workload(3).tables[1])
        return dataclasses.replace(w5, tables=[spec], d=256, M=1), spec
    spec = dataclasses.replace(shrink_table(W.make_workload(2).tables[0]), K=16)   # 2 x 16 heads of 64
    return dataclasses.replace(w5, tables=[spec], d=1024, M=4), spec


@pytest.mark.parametrize("name,B", [("pagegram_bf16", 5), ("pagegram_nf4", 2), ("flat_bf16", 7), ("wide", 3)])
def test_decode_step_context_gate_over_other_layouts(cuda, name, B):
    pg = _pg()
    w, spec = _layout_case(name)
    T = 11
    m = Module(w, spec, B, T, 230 + B, cuda)
    assert m.Din in (768, 1024, 2048)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    pg.device_error(clear=True)
    e, v, al, ms, H, state = m.run_step(pg, desc, cuda)
    assert pg.device_error() == 0
    e_ref, v_ref, a_ref, H_ref = m.oracle()
    for t in range(T):
        assert np.array_equal(bits16(e[t]), np.ascontiguousarray(e_ref[:, t])), t
    assert rel_l2(to_f64(v).transpose(1, 0, 2), v_ref) <= BF16_TOL
    assert np.abs(to_f64(al).transpose(1, 2, 0) - a_ref).max() < 2e-3
    H_got = to_f64(H).transpose(1, 2, 0, 3)
    H0 = m.H.double().numpy()
    assert rel_l2(H_got, H_ref) <= BF16_TOL
    assert rel_l2(H_got - H0, H_ref - H0) <= 5e-2
    assert (state.pos.cpu() == T).all()
