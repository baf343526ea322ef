"""Correlated collisions on the GPU (PageGram report 3.2 and 6.1): pg_collision_counts'
integer pair counts equal the oracle's on the same hashed rows, for PageGram tables of the
report's slot sweep S in {1, 4, 8, 15, 60} at a fixed 200M-parameter budget and for the
Engram-style table of the same budget; at millions of distinct n-grams the mean number of
further shared heads follows (K - 1) / S."""
import numpy as np
import pytest
import torch

from hashed_head_gram_gb300 import workloads as W
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _pg():
    from hashed_head_gram_gb300 import pg
    return pg


def _gpu_rows(pg, desc, spec, grams, cuda):
    """Head rows of every n-gram at its last position: int32 [n * L, O, H] on the GPU."""
    n, L = grams.shape
    O, H = len(spec.orders), orc.heads(spec)
    rows = torch.empty(n * L, O, H, dtype=torch.int32, device=cuda)
    pg.canon_hash(desc, torch.from_numpy(grams).to(cuda), rows)
    return rows


def _order_span(spec, o):
    """[lo, lo + span) holding order o's head-0 rows."""
    if spec.mode == W.MODE_PAGEGRAM:
        lo = sum(p * spec.K * spec.S for p in spec.pages[:o])
        return lo, spec.pages[o] * spec.K * spec.S
    lo = sum(sum(rr) for rr in spec.rows[:o])
    return lo, spec.rows[o][0]


def _gpu_counts(pg, rows, n, L, spec, o, cuda, lo=None, span=None):
    O, H = len(spec.orders), orc.heads(spec)
    lo0, span0 = _order_span(spec, o)
    lo = lo0 if lo is None else lo
    span = span0 if span is None else span
    ws = torch.empty(pg.collision_workspace_size(n, span), dtype=torch.uint8, device=cuda)
    counts = torch.empty(H, dtype=torch.int64, device=cuda)
    view = rows.view(-1)[(L - 1) * O * H + o * H:]
    pg.collision_counts(view, n, H, L * O * H, lo, span, counts, ws)
    torch.cuda.synchronize()
    return counts.cpu().numpy()


def _oracle_counts(spec, grams, vocab, o):
    _, rows, _, bad = orc.index(spec, grams, None, vocab)
    assert bad == -1
    n, L = grams.shape
    last = rows.reshape(n, L, *rows.shape[1:])[:, -1, o, :]
    return orc.collision_counts(last)[1], last


@pytest.mark.parametrize("S", W.SLOT_SWEEP)
@pytest.mark.parametrize("o", [0, 1])
def test_pagegram_counts_match_the_oracle(cuda, S, o):
    pg = _pg()
    spec = W.pagegram_slots(S)
    w = W.make_workload(2)
    n = 300_000
    grams = W.distinct_ngrams(n, spec.orders[o], w.vocab, seed=S)
    desc = pg.table_desc(spec, w.vocab)
    rows = _gpu_rows(pg, desc, spec, grams, cuda)
    pg.device_error(clear=True)
    got = _gpu_counts(pg, rows, n, grams.shape[1], spec, o, cuda)
    assert pg.device_error() == 0
    ref, _ = _oracle_counts(spec, grams, w.vocab, o)
    assert got[0] > 1000
    assert np.array_equal(got, ref)
    if S == 1:
        assert (got == got[0]).all()        # one slot per head: a shared page is every head


def test_engram_counts_match_the_oracle(cuda):
    pg = _pg()
    w = W.make_workload(3)
    spec = w.tables[0]
    n = 400_000
    grams = W.distinct_ngrams(n, 2, w.vocab, seed=7)
    desc = pg.table_desc(spec, w.vocab)
    rows = _gpu_rows(pg, desc, spec, grams, cuda)
    got = _gpu_counts(pg, rows, n, 2, spec, 0, cuda)
    ref, _ = _oracle_counts(spec, grams, w.vocab, 0)
    assert np.array_equal(got, ref)


def test_rows_outside_the_span_are_reported_and_left_out(cuda):
    pg = _pg()
    spec = W.pagegram_slots(4)
    w = W.make_workload(2)
    n = 50_000
    grams = W.distinct_ngrams(n, 2, w.vocab, seed=11)
    desc = pg.table_desc(spec, w.vocab)
    rows = _gpu_rows(pg, desc, spec, grams, cuda)
    lo, span = _order_span(spec, 0)
    cut = span // 2
    pg.device_error(clear=True)
    got = _gpu_counts(pg, rows, n, 2, spec, 0, cuda, lo=lo, span=cut)
    assert pg.device_error(clear=True) == 1024
    _, last = _oracle_counts(spec, grams, w.vocab, 0)
    keep = last[:, 0].astype(np.int64) - lo < cut
    assert np.array_equal(got, orc.collision_counts(last[keep])[1])


def test_empty_and_single_sets(cuda):
    pg = _pg()
    counts = torch.full((8,), 7, dtype=torch.int64, device=cuda)
    ws = torch.empty(pg.collision_workspace_size(1, 100), dtype=torch.uint8, device=cuda)
    rows = torch.zeros(8, dtype=torch.int32, device=cuda)
    pg.collision_counts(rows, 0, 8, 8, 0, 100, counts, ws)
    torch.cuda.synchronize()
    assert (counts.cpu() == 0).all()
    pg.collision_counts(rows, 1, 8, 8, 0, 100, counts, ws)
    torch.cuda.synchronize()
    assert (counts.cpu() == 0).all()


@pytest.mark.parametrize("S", W.SLOT_SWEEP)
def test_extra_shared_heads_follow_k_minus_1_over_s(cuda, S):
    # 4M distinct bigrams: about 4e7 pairs collide on head 0; their mean number of further
    # shared heads is (K - 1) / S (report 3.2; 0.467 measured at S = 15 in 6.1)
    pg = _pg()
    spec = W.pagegram_slots(S)
    w = W.make_workload(2)
    n = 4_000_000
    grams = W.distinct_ngrams(n, 2, w.vocab, seed=100 + S)
    rows = _gpu_rows(pg, pg.table_desc(spec, w.vocab), spec, grams, cuda)
    pg.device_error(clear=True)
    got = _gpu_counts(pg, rows, n, 2, spec, 0, cuda)
    assert pg.device_error() == 0
    pairs0 = got[0]
    head0_rows = spec.pages[0] * spec.S
    assert abs(pairs0 / (n * (n - 1) / 2 / head0_rows) - 1) < 0.02    # about uniform on head 0
    mean = got[1:].sum() / pairs0
    assert abs(mean - 7 / S) <= 0.03 * (7 / S), (S, mean)


@pytest.mark.parametrize("S", W.SLOT_SWEEP)
def test_slot_sweep_lookup_and_one_launch_parity(cuda, S):
    # every table of the sweep at full size (200M parameters) on workload 2's 64 x 1024
    # tokens: the lookup bit for bit at sampled tokens, the one-launch lookup + projection
    # writing the same e_t and the scalar-gated output within the bf16 tolerance
    from oracle import dense
    from tests._helpers import BF16_TOL, bits16, oracle_e, rel_l2, to_f64
    pg = _pg()
    w = W.make_workload(2)
    spec = W.pagegram_slots(S)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    tokens = W.make_tokens(w)
    tok = torch.from_numpy(tokens).to(cuda)
    table = W.make_table(w, spec, cuda)
    dn = W.make_dense(w, cuda)
    e = torch.empty(w.N, spec.e_width, dtype=torch.bfloat16, device=cuda)
    pg.gather_sign_concat(desc, tok, table, e, pg.BF16)
    e1 = torch.empty_like(e)
    out = torch.empty(w.N, w.d, dtype=torch.bfloat16, device=cuda)
    ws = torch.empty(pg.gather_project_workspace_size(w.N, w.d, 0, pg.GATE_SCALAR) // 4 + 1, device=cuda)
    pg.gather_project_gate(desc, tok, table, e1, dn["W"], w.d, pg.GATE_SCALAR, out, ws, g=w.g, x_resid=dn["x"])
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    assert torch.equal(e.view(torch.int16), e1.view(torch.int16))
    rng = np.random.default_rng(S)
    which = np.concatenate([[0, 1, 2, w.L - 1, w.N - 1], rng.integers(0, w.N, 91)]).astype(np.int64)
    ref = oracle_e(spec, tokens, None, w.vocab, table, orc.BF16, which=which)
    idx = torch.from_numpy(which).to(cuda)
    assert np.array_equal(bits16(e[idx]), ref)
    v_ref = dense.project(orc.bf16_bits_to_f64(ref), to_f64(dn["W"]))
    x = to_f64(dn["x"][idx])
    assert rel_l2(to_f64(out[idx]), dense.scalar_gate(x, v_ref, w.g)) <= BF16_TOL


def test_per_head_collision_rate_is_the_same_across_layouts(cuda):
    # PageGram report 3.2: at a fixed budget each head has the same number of rows in both
    # layouts (P_n S for PageGram, M_{n,k} for the Engram-style subtables), so a pair of
    # n-grams collides on a given head equally often; 4M distinct bigrams, head 0
    pg = _pg()
    n = 4_000_000
    rates = {}
    for name, w, spec in (("pagegram", W.make_workload(2), W.pagegram_slots(4)),
                          ("engram", W.make_workload(3), W.make_workload(3).tables[0])):
        grams = W.distinct_ngrams(n, 2, w.vocab, seed=500)
        rows = _gpu_rows(pg, pg.table_desc(spec, w.vocab), spec, grams, cuda)
        got = _gpu_counts(pg, rows, n, 2, spec, 0, cuda)
        head_rows = spec.pages[0] * spec.S if spec.mode == W.MODE_PAGEGRAM else spec.rows[0][0]
        rates[name] = got[0] / (n * (n - 1) / 2) * head_rows     # 1 for an ideal hash
    assert abs(rates["pagegram"] - 1) < 0.02 and abs(rates["engram"] - 1) < 0.02, rates
    assert abs(rates["pagegram"] / rates["engram"] - 1) < 0.02, rates
