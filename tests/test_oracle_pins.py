"""Pins for the CPU oracle: what the pages and the mathematics fix, independent of
the oracle's own formulas. Runs without a GPU (-m "not gpu")."""
import dataclasses
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import dense
from oracle import oracle as orc
from oracle.nf4_levels import derive_levels
from hashed_head_gram_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def _golden_kv(name):
    return {k.strip(): v.strip() for k, v in (r for r in
            (line.split("=") for line in open(os.path.join(GOLDEN, name))
             if "=" in line and not line.startswith("#")))}


def spec(mode, K=8, S=4, r=64, dt=W.DT_F32, pages=(7, 5), rows=None, orders=(2, 3),
         seed=0x1234567, kind=W.HASH_MULXOR):
    return W.TableSpec("t", mode, K=K, S=S, r=r, row_dtype=dt, orders=list(orders),
                       pages=list(pages), rows=rows or [], hash_kind=kind, hash_seed=seed)


def all_bigrams(V):
    a, b = np.meshgrid(np.arange(V), np.arange(V), indexing="ij")
    return np.stack([a.ravel(), b.ravel()], 1).astype(np.int32)  # [V*V, 2]: sequences of length 2


def rows_at_last(sp, toks, vocab):
    _, rows, signs, bad = orc.index(sp, toks, None, vocab)
    L = toks.shape[1]
    rows = rows.reshape(toks.shape[0], L, *rows.shape[1:])[:, -1]
    signs = signs.reshape(toks.shape[0], L, *signs.shape[1:])[:, -1]
    return rows, signs


# ------------------------------------------------------------------ the pages' toy hash

def test_toy_bucket_worked_values():
    for a, b, m, want in _golden_rows("toy_bucket.txt"):
        assert orc.bigram_bucket([int(a), int(b)], int(m)) == int(want)


@pytest.mark.parametrize("tokens,size", [([1], 5), ([1, 2, 3], 5), ([1, 2], 0), ([1, 2], -3),
                                         ([1, 2], 5.0), ([-1, 2], 5), ([1, 2.0], 5), ([1, "2"], 5)])
def test_toy_bucket_rejects_invalid(tokens, size):
    with pytest.raises(ValueError):
        orc.bigram_bucket(tokens, size)


def test_toy_mode_through_the_ngram_window():
    # The sequence 1, 2, 4 holds the explainer's two bigrams (1,2) at t=1 and
    # (2,4) at t=2; the index path must form them from x'_{t-1}, x'_t.
    toks = np.array([[1, 2, 4]], np.int32)
    for m, want in ((5, [0, 0]), (7, [5, 3])):
        sp = spec(W.MODE_FLAT, K=1, S=1, r=64, rows=[[m]], orders=[2], kind=W.HASH_TOY)
        _, rows, _, bad = orc.index(sp, toks, None, 16)
        assert bad == -1
        assert rows[0, 0, 0] == orc.NO_ROW          # no bigram at t = 0
        assert list(rows[1:, 0, 0]) == want


# ------------------------------------------------------------------ mixing function

def test_mix64_matches_splitmix64_reference_outputs():
    g = 0x9E3779B97F4A7C15
    for i, want in _golden_rows("splitmix64.txt"):
        assert orc.lib().orc_mix64((int(i) * g) & (2**64 - 1)) == int(want, 16)


def test_multipliers_odd_and_distinct():
    L = orc.lib()
    ms = {L.orc_multiplier(99, kind, o, k, j) for kind in range(3) for o in range(4)
          for k in range(16) for j in range(4)}
    assert len(ms) == 3 * 4 * 16 * 4
    assert all(m & 1 for m in ms)


# ------------------------------------------------------------------ addressing layouts

@pytest.mark.parametrize("S", [1, 4, 15])
def test_pagegram_heads_share_one_page_and_stay_in_range(S):
    sp = spec(W.MODE_PAGEGRAM, K=8, S=S, pages=(13, 11))
    rng = np.random.default_rng(0)
    toks = rng.integers(0, 500, (4, 300)).astype(np.int32)
    _, rows, _, _ = orc.index(sp, toks, None, 500)
    K, base = 8, [0, 13 * 8 * S]
    for o, P in enumerate(sp.pages):
        rel = rows[:, o, :].astype(np.int64) - base[o]
        assert rel.min() >= 0 and rel.max() < P * K * S          # inside the order's range
        page = rel // (K * S)
        assert (page == page[:, :1]).all()                        # every head in one page
        head_block = (rel % (K * S)) // S
        assert (head_block == np.arange(K)).all()                 # head k in its own S slots


def test_engram_and_flat_rows_inside_their_subtables():
    eng = W.largest_primes(61, 16)
    sp = spec(W.MODE_ENGRAM, K=8, rows=[eng[:8], eng[8:]])
    toks = np.random.default_rng(1).integers(0, 300, (3, 400)).astype(np.int32)
    _, rows, _, _ = orc.index(sp, toks, None, 300)
    base = np.cumsum([0] + eng)[:-1].reshape(2, 8)
    rel = rows.astype(np.int64) - base
    assert (rel >= 0).all() and (rel < np.array(eng).reshape(2, 8)).all()
    assert orc.total_rows(sp) == sum(eng)

    fl = spec(W.MODE_FLAT, K=1, S=1, r=128, rows=[[37], [29]])
    _, rows, _, _ = orc.index(fl, toks, None, 300)
    assert rows[:, 0, 0].max() < 37 and (rows[:, 1, 0] >= 37).all() and rows[:, 1, 0].max() < 66


def test_parameter_budgets_match_the_report():
    g = _golden_kv("layout_arithmetic.txt")
    cfg2, cfg3 = W.make_workload(2), W.make_workload(3)
    pg = cfg2.tables[0]
    assert orc.total_rows(pg) * pg.r == int(g["pagegram_params"])
    flat = cfg3.tables[1]
    assert orc.total_rows(flat) * flat.r == int(g["flat_params"])
    eng = cfg3.tables[0]
    assert abs(orc.total_rows(eng) * eng.r / int(g["flat_params"]) - 1) < 1e-3   # "within 0.1%"


# ------------------------------------------------------------------ hash statistics (brute force)

def test_bucket_loads_are_poisson_like():
    # All 64^2 bigrams into a prime subtable of 61 rows: per-head bucket loads
    # should have variance/mean ~ 1 (PageGram report 6.1). chi^2(60) 99.9% band.
    eng = [61] * 8 + [59] * 8
    sp = spec(W.MODE_ENGRAM, K=8, rows=[eng[:8], eng[8:]], orders=[2, 3])
    rows, _ = rows_at_last(sp, all_bigrams(64), 64)
    for k in range(8):
        counts = np.bincount(rows[:, 0, k].astype(np.int64) - 61 * k, minlength=61)
        stat = ((counts - counts.mean()) ** 2).sum() / counts.mean()
        assert 27.0 < stat < 100.0, (k, stat)   # chi^2(60): 0.05th..99.95th percentile


def _brute_force_pairs(r):
    """Every unordered pair compared directly: [K] counts of pairs equal on head 0 and k."""
    n, K = r.shape
    out = np.zeros(K, np.int64)
    for i in range(n):
        for j in range(i + 1, n):
            if r[i, 0] == r[j, 0]:
                out += (r[i] == r[j]).astype(np.int64)
    return out


@pytest.mark.parametrize("n,K,hi,seed", [(0, 8, 5, 1), (1, 8, 5, 2), (60, 8, 4, 3), (300, 3, 7, 4),
                                         (250, 16, 2, 5), (400, 8, 40, 6)])
def test_collision_counts_equal_brute_force(n, K, hi, seed):
    # small value ranges so that pairs collide often, on head 0 and on the others
    rng = np.random.default_rng(seed)
    r = rng.integers(0, hi, (n, K)).astype(np.uint32)
    r[:, 0] += np.uint32(0xFFFFFF00)              # high bits in use: keys must not alias
    pairs0, shared = orc.collision_counts(r)
    bf = _brute_force_pairs(r)
    assert pairs0 == bf[0] and np.array_equal(shared, bf)


def test_collision_counts_closed_forms():
    n = 37
    same = np.tile(np.arange(8, dtype=np.uint32), (n, 1))
    pairs0, shared = orc.collision_counts(same)
    assert pairs0 == n * (n - 1) // 2 and (shared == pairs0).all()          # all pairs, all heads
    distinct = np.arange(n * 8, dtype=np.uint32).reshape(n, 8)
    assert orc.collision_counts(distinct)[0] == 0
    # two groups on head 0 (sizes 3 and 4); head 1 splits the second group 2 + 2
    r = np.array([[5, 1], [5, 2], [5, 3], [9, 7], [9, 7], [9, 8], [9, 8]], np.uint32)
    pairs0, shared = orc.collision_counts(r)
    assert pairs0 == 3 + 6 and shared[1] == 2


@pytest.mark.parametrize("S", [1, 4, 15])
def test_collision_counts_on_pagegram_rows(S):
    # through the hash: the report's (K - 1) / S law (3.2) and S = 1's full overlap
    sp = spec(W.MODE_PAGEGRAM, K=8, S=S, pages=(3, 3))
    rows, _ = rows_at_last(sp, all_bigrams(96), 96)
    pairs0, shared = orc.collision_counts(rows[:, 0, :])
    if S == 1:
        assert (shared == pairs0).all()
    mean = shared[1:].sum() / pairs0
    assert abs(mean - 7 / S) < 6 * np.sqrt(7 * (1 / S) * (1 - 1 / S) / pairs0) * 3 + 1e-3, (mean, S)


@pytest.mark.parametrize("S,expect", [(4, 7 / 4), (15, 7 / 15)])
def test_pagegram_extra_shared_heads(S, expect):
    # Given two n-grams collide on head 0, the other K-1 heads collide w.p. 1/S
    # each: E[extra shared heads] = (K-1)/S (PageGram report 3.2; 0.467 at S=15, 6.1).
    sp = spec(W.MODE_PAGEGRAM, K=8, S=S, pages=(3, 3))
    rows, _ = rows_at_last(sp, all_bigrams(96), 96)
    r = rows[:, 0, :].astype(np.int64)
    extra, pairs = 0, 0
    order = np.lexsort((r[:, 0],))
    r = r[order]
    starts = np.flatnonzero(np.r_[True, r[1:, 0] != r[:-1, 0]])
    for s, e in zip(starts, np.r_[starts[1:], len(r)]):
        grp = r[s:e]
        if len(grp) < 2:
            continue
        same = (grp[:, None, 1:] == grp[None, :, 1:]).sum(-1)
        iu = np.triu_indices(len(grp), 1)
        extra += same[iu].sum()
        pairs += len(iu[0])
    mean = extra / pairs
    se = np.sqrt(7 * (1 / S) * (1 - 1 / S) / pairs) * 3
    assert abs(mean - expect) < 6 * se + 1e-3, (mean, expect)
    if S == 15:
        g = float(_golden_kv("layout_arithmetic.txt")["extra_shared_heads_S15"])
        assert abs(expect - g) < 5e-4


def test_engram_second_head_recollision_is_about_one_over_M():
    eng = [53] * 16
    sp = spec(W.MODE_ENGRAM, K=8, rows=[eng[:8], eng[8:]])
    rows, _ = rows_at_last(sp, all_bigrams(80), 80)
    r = rows[:, 0, :].astype(np.int64)
    both, head0 = 0, 0
    for v in np.unique(r[:, 0]):
        grp = r[r[:, 0] == v]
        iu = np.triu_indices(len(grp), 1)
        head0 += len(iu[0])
        both += (grp[iu[0], 1] == grp[iu[1], 1]).sum()
    p = both / head0
    assert abs(p - 1 / 53) < 4 * np.sqrt((1 / 53) / head0) + 1e-3, p


def test_sign_bits_are_balanced():
    sp = spec(W.MODE_PAGEGRAM, K=8, S=4, r=80)
    _, signs = rows_at_last(sp, all_bigrams(40), 40)
    bits = np.unpackbits(np.ascontiguousarray(signs).view(np.uint8)).mean()
    assert abs(bits - 0.5) < 0.005


def test_slot_count_extremes():
    # S = 1: n-grams on one page collide on every head (report 3.2, first bullet).
    sp1 = spec(W.MODE_PAGEGRAM, K=8, S=1, pages=(5, 5))
    rows, _ = rows_at_last(sp1, all_bigrams(30), 30)
    r = rows[:, 0, :].astype(np.int64)
    page = r // 8
    same_page = page[:, None, 0] == page[None, :, 0]
    all_heads = (r[:, None, :] == r[None, :, :]).all(-1)
    assert (same_page == all_heads).all()
    # One page per order: heads become independent (second bullet): the
    # conditional head-1 collision rate equals the unconditional 1/S.
    spP = spec(W.MODE_PAGEGRAM, K=8, S=8, pages=(1, 1))
    rows, _ = rows_at_last(spP, all_bigrams(64), 64)
    r = rows[:, 0, :].astype(np.int64)
    c0 = r[:, None, 0] == r[None, :, 0]
    c1 = r[:, None, 1] == r[None, :, 1]
    iu = np.triu_indices(len(r), 1)
    cond = c1[iu][c0[iu]].mean()
    assert abs(cond - 1 / 8) < 0.01, cond


# ------------------------------------------------------------------ n-gram window, canon map

def test_rows_depend_exactly_on_the_suffix_window():
    sp = spec(W.MODE_ENGRAM, K=8, rows=[[101] * 8, [103] * 8])
    rng = np.random.default_rng(3)
    base = rng.integers(0, 1000, (1, 64)).astype(np.int32)
    _, r0, s0, _ = orc.index(sp, base, None, 1000)
    t = 40
    for pos in range(t - 4, t + 2):
        pert = base.copy()
        pert[0, pos] = (pert[0, pos] + 17) % 1000
        _, r1, s1, _ = orc.index(sp, pert, None, 1000)
        for o, n in enumerate([2, 3]):
            inside = t - n + 1 <= pos <= t
            same = (s0[t, o] == s1[t, o]).all()
            assert same != inside, (pos, n)     # sign words track the exact window
    # identical n-grams in other sequences / positions get identical rows
    toks = np.array([[5, 6, 7, 5, 6, 7], [9, 5, 6, 7, 1, 2]], np.int32)
    _, r, _, _ = orc.index(sp, toks, None, 10)
    r = r.reshape(2, 6, 2, 8)
    assert (r[0, 2, 1] == r[0, 5, 1]).all() and (r[0, 2, 1] == r[1, 3, 1]).all()


def test_positions_before_the_start_are_padding_not_a_token():
    # The first positions' n-grams reach back past the start of the sequence, and what
    # stands there is padding: a symbol that is no token. So token x at t = 0 is hashed
    # unlike x after any real token y, and [y, x] at t = 1 unlike [z, y, x] at t = 2 (every
    # y, z of a small vocabulary). Sign words are bijective in the n-gram's 64-bit hash,
    # so they differ exactly when the n-grams do.
    sp = spec(W.MODE_ENGRAM, K=8, rows=[[101] * 8, [103] * 8])
    V = 12
    for x in range(V):
        _, _, s0, _ = orc.index(sp, np.array([[x]], np.int32), None, V)
        pairs = np.array([[y, x] for y in range(V)], np.int32)
        _, _, s1, _ = orc.index(sp, pairs, None, V)
        s1 = s1.reshape(V, 2, *s1.shape[1:])
        for y in range(V):
            assert not np.array_equal(s0[0, 0], s1[y, 1, 0]), (x, y)     # bigram (pad, x) vs (y, x)
            triples = np.array([[z, y, x] for z in range(V)], np.int32)
            _, _, s2, _ = orc.index(sp, triples, None, V)
            s2 = s2.reshape(V, 3, *s2.shape[1:])
            for z in range(V):
                assert not np.array_equal(s1[y, 1, 1], s2[z, 2, 1]), (x, y, z)   # (pad, y, x) vs (z, y, x)


def test_sequences_do_not_leak_into_each_other():
    sp = spec(W.MODE_PAGEGRAM)
    toks = np.random.default_rng(4).integers(0, 50, (3, 10)).astype(np.int32)
    _, r0, _, _ = orc.index(sp, toks, None, 50)
    toks2 = toks.copy()
    toks2[0, -3:] = (toks2[0, -3:] + 1) % 50          # end of sequence 0
    _, r1, _, _ = orc.index(sp, toks2, None, 50)
    assert (r0[10:] == r1[10:]).all()                  # sequences 1 and 2 unchanged


def test_canonical_map_folds_ids_and_is_surjective():
    w = W.make_workload(4)
    cm = W.make_canon_map(w)
    g = _golden_kv("layout_arithmetic.txt")
    assert w.vocab - w.canon_vocab == round(float(g["canon_shrink"]) * w.vocab)
    assert cm.max() < w.canon_vocab and len(np.unique(cm)) == w.canon_vocab
    # two raw IDs with one canonical ID give identical rows
    j = int(np.flatnonzero(np.arange(w.vocab) != cm)[0])
    toks = np.array([[3, 4, j, 8], [3, 4, int(cm[j]), 8]], np.int32)
    sp = spec(W.MODE_PAGEGRAM)
    _, rows, _, _ = orc.index(sp, toks, cm, w.vocab)
    rows = rows.reshape(2, 4, 2, 8)
    assert (rows[0] == rows[1]).all()


def test_out_of_range_ids_are_reported():
    sp = spec(W.MODE_PAGEGRAM)
    toks = np.array([[1, 2, 3], [4, 70, 6]], np.int32)
    _, _, _, bad = orc.index(sp, toks, None, 50)
    assert bad == 4
    # several: the smallest flat position is the one reported (IDs >= V and negative IDs)
    toks = np.array([[1, 2, 3], [4, 70, 6], [50, 2, -1]], np.int32)
    assert orc.index(sp, toks, None, 50)[3] == 4
    toks[0, 2] = -7
    assert orc.index(sp, toks, None, 50)[3] == 2
    with pytest.raises(ValueError):
        orc.lookup(sp, toks, None, 50, np.zeros((orc.total_rows(sp), 256), np.uint8), orc.F32)


# ------------------------------------------------------------------ assembly: sign, concat, flat, NF4

def _marker_table(sp):
    R = orc.total_rows(sp)
    t = (np.arange(R)[:, None] + 1 + np.arange(sp.r)[None, :] / 128.0).astype(np.float32)
    return t


def test_concat_order_and_sign_flip():
    sp = spec(W.MODE_PAGEGRAM, K=8, S=4, r=64, pages=(11, 7))
    toks = np.random.default_rng(5).integers(0, 200, (2, 50)).astype(np.int32)
    table = _marker_table(sp)
    e = orc.lookup(sp, toks, None, 200, table.view(np.uint8), orc.F32)
    _, rows, signs, _ = orc.index(sp, toks, None, 200)
    e = e.reshape(-1, 2, 8, 64)
    row_of_block = np.floor(np.abs(e[..., 0])).astype(np.int64) - 1
    assert (row_of_block == rows).all()                          # block (o,k) holds row (o,k)
    assert (np.abs(e) == table[rows.astype(np.int64)]).all()    # only the sign can differ
    bits = (signs[..., 0][..., None] >> np.arange(64, dtype=np.uint64)) & np.uint64(1)
    assert ((e < 0) == (bits == 1)).all()


def test_flat_sum_of_two_signed_rows():
    sp = spec(W.MODE_FLAT, K=1, S=1, r=128, rows=[[31], [17]])
    toks = np.random.default_rng(6).integers(0, 100, (1, 40)).astype(np.int32)
    table = np.zeros((48, 128), np.float32)
    table[31:] = 1.0                                  # order-3 rows: ones; order-2: zeros
    e = orc.lookup(sp, toks, None, 100, table.view(np.uint8), orc.F32)
    _, rows, signs, _ = orc.index(sp, toks, None, 100)
    bits = (signs[:, 1, 0][:, :, None] >> np.arange(64, dtype=np.uint64)).reshape(-1, 128) & 1
    assert (np.abs(e) == 1).all() and ((e < 0) == (bits == 1)).all()


def test_bf16_sign_flip_is_exact():
    sp = spec(W.MODE_ENGRAM, K=4, r=80, dt=W.DT_BF16, rows=[[13] * 4, [11] * 4])
    R = orc.total_rows(sp)
    vals = torch.randn(R, 80).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    toks = np.random.default_rng(7).integers(0, 60, (2, 20)).astype(np.int32)
    e = orc.lookup(sp, toks, None, 60, vals.view(np.uint8).reshape(R, -1), orc.BF16)
    _, rows, _, _ = orc.index(sp, toks, None, 60)
    src = vals[rows.reshape(-1).astype(np.int64)].reshape(e.shape)
    assert ((e ^ src) & 0x7FFF == 0).all()


def test_nf4_format_arithmetic_and_levels():
    g = _golden_kv("layout_arithmetic.txt")
    assert 64 * 4 // 8 + 2 == int(g["nf4_row_bytes"])
    assert 4096 // int(g["nf4_row_bytes"]) == int(g["nf4_rows_per_4k"])
    assert 8 * 15 * 34 == int(g["page_bytes_S15"]) and 8 * 4 * 34 == int(g["page_bytes_S4"])
    lv = orc.nf4_levels()
    assert (np.diff(lv) > 0).all() and lv[0] == -1 and lv[7] == 0 and lv[15] == 1


def test_nf4_levels_are_qlora_published_table():
    # the 16 NF4 values printed in the QLoRA paper (Appendix E), each to the precision it is
    # printed with: the oracle's fp32 levels are those values rounded to fp32, bit for bit
    pub = np.array([float(r[0]) for r in _golden_rows("nf4_levels_qlora.txt")])
    assert pub.shape == (16,)
    lv = orc.nf4_levels()
    assert (lv.view(np.uint32) == pub.astype(np.float32).view(np.uint32)).all()
    # and a plain restatement of the construction (normal quantiles, exact fp64 outer
    # probability) lands within 2 fp32 ulps of them: a wrong outer probability, a wrong
    # 7/8 split or a missing normalisation would move a level by >= 1e-3
    d = derive_levels().astype(np.float64)
    assert np.abs(d - pub).max() <= 2e-7
    # symmetric-type control: the same quantiles with an 8/8 split (no exact zero) differ
    # from the table by far more than the tolerance above
    from scipy.stats import norm
    delta = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0)
    sym = norm.ppf(np.linspace(1 - delta, delta, 16))
    assert np.abs(sym / sym.max() - pub).max() > 1e-2


def test_nf4_decode_special_rows():
    sp = spec(W.MODE_PAGEGRAM, K=2, S=1, r=64, dt=W.DT_NF4, pages=(1, 1))
    table = np.zeros((4, 34), np.uint8)
    table[0, :32] = 0x77                      # all codes = level 0.0, scale 1.5
    table[0, 32:] = np.array([0x3E00], np.uint16).view(np.uint8)
    table[1, :32] = (np.arange(32) * 37 % 256).astype(np.uint8)   # varied codes, scale 1.0
    table[1, 32:] = np.array([0x3C00], np.uint16).view(np.uint8)
    table[2, :32] = 0xF0                      # codes 0 / 15 alternating, scale 0
    table[3, :32] = 0xAB
    table[3, 32:] = np.array([0x4000], np.uint16).view(np.uint8)  # scale 2
    rows = np.array([[[0, 1], [2, 3]]], np.uint32)
    signs = np.zeros((1, 2, 2, 1), np.uint64)
    e = orc.assemble(sp, rows, orc.fetch_rows(table, rows), signs, orc.F32).reshape(4, 64)
    lv = orc.nf4_levels()
    assert (e[0] == 0).all() and not np.signbit(e[0]).any()    # zero row stays exactly zero
    codes = np.stack([table[1, :32] & 15, table[1, :32] >> 4], 1).reshape(-1)
    assert (e[1] == lv[codes]).all()                           # scale 1 returns the level
    assert (e[2] == 0).all()
    assert (e[3] == np.tile(np.float32([lv[0xB] * 2, lv[0xA] * 2]), 32)).all()


def test_number_conversions_against_libraries():
    L = orc.lib()
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.standard_normal(3000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 3000),
                        np.float32([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 3.3895314e38, 1e-40])])
    x = x.astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.f32_to_bf16_bits(x)
    assert (got == want).all()
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float32)
    ours = np.array([L.orc_f16_to_f32(int(v)) for v in h], np.float32)
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all() and (ours[~nan].view(np.uint32) == ref[~nan].view(np.uint32)).all()


# ------------------------------------------------------------------ dense half vs torch (fp64)

def _dense_case(seed=9, B=2, L=23, d=64, M=3, Din=96):
    g = torch.Generator().manual_seed(seed)
    return dict(e=torch.randn(B * L, Din, generator=g, dtype=torch.float64),
                W=torch.randn((1 + M) * d, Din, generator=g, dtype=torch.float64) * 0.1,
                h=torch.randn(M, B * L, d, generator=g, dtype=torch.float64),
                gh=torch.rand(d, generator=g, dtype=torch.float64) + 0.5,
                gk=torch.rand(d, generator=g, dtype=torch.float64) + 0.5,
                gc=torch.rand(d, generator=g, dtype=torch.float64) + 0.5,
                w=torch.randn(d, 4, generator=g, dtype=torch.float64) * 0.3,
                H=torch.randn(M, B, L, d, generator=g, dtype=torch.float64),
                B=B, L=L, d=d, M=M)


def test_projection_and_gate_against_torch():
    c = _dense_case()
    d, M, eps = c["d"], c["M"], 1e-6
    v, alpha = dense.engram_gate(c["e"].numpy(), c["W"].numpy(), c["h"].numpy(),
                                 c["gh"].numpy(), c["gk"].numpy(), eps, M)
    vk = c["e"] @ c["W"].T
    assert np.allclose(v, vk[:, :d].numpy(), rtol=1e-12, atol=1e-12)
    for m in range(M):
        k = vk[:, (1 + m) * d:(2 + m) * d]
        s = (F.rms_norm(c["h"][m], (d,), c["gh"], eps) * F.rms_norm(k, (d,), c["gk"], eps)).sum(-1)
        ref = torch.sigmoid(s / d ** 0.5)
        assert np.allclose(alpha[m], ref.numpy(), rtol=1e-12, atol=1e-14)
    x = torch.randn(c["e"].shape[0], d, dtype=torch.float64)
    assert np.allclose(dense.scalar_gate(x.numpy(), v, 0.5), (x + 0.5 * vk[:, :d]).numpy())


# kernel 4, dilation 3 is the Engram notes' conv; the others cover one tap, dilation 1 and
# windows that reach past the start of the 23-position sequences (3 * 8 = 24 back)
@pytest.mark.parametrize("ks,dil", [(4, 3), (1, 1), (2, 1), (3, 2), (2, 5), (4, 8), (3, 7)])
def test_conv_residual_against_torch_conv1d(ks, dil):
    c = _dense_case()
    B, L, d, M, eps = c["B"], c["L"], c["d"], c["M"], 1e-6
    v = torch.randn(B, L, d, dtype=torch.float64)
    alpha = torch.rand(M, B, L, dtype=torch.float64)
    w = c["w"][:, :ks]
    got = dense.conv_residual(v.numpy(), alpha.numpy(), c["gc"].numpy(), w.numpy(), dil, eps, c["H"].numpy())
    pad = (ks - 1) * dil
    for m in range(M):
        u = alpha[m][..., None] * v
        z = F.rms_norm(u, (d,), c["gc"], eps)
        # torch conv1d is a cross-correlation: tap i of the left-padded input reads
        # position t - dil * (ks - 1 - i), so our tap j = ks - 1 - i.
        wt = w.flip(1)[:, None, :]
        conv = F.conv1d(F.pad(z.transpose(1, 2), (pad, 0)), wt, groups=d, dilation=dil).transpose(1, 2)
        ref = c["H"][m] + F.silu(conv) + u
        assert np.allclose(got[m], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_zero_table_leaves_the_residual_stream_unchanged():
    c = _dense_case()
    n, d, M = c["B"] * c["L"], c["d"], c["M"]
    e = np.zeros((n, c["e"].shape[1]))
    v, alpha = dense.engram_gate(e, c["W"].numpy(), c["h"].numpy(), c["gh"].numpy(),
                                 c["gk"].numpy(), 1e-6, M)
    assert (v == 0).all() and (alpha == 0.5).all()
    H = c["H"].numpy()
    out = dense.conv_residual(v.reshape(c["B"], c["L"], d), alpha.reshape(M, c["B"], c["L"]),
                              c["gc"].numpy(), c["w"].numpy(), 3, 1e-6, H)
    assert (out == H).all()


def test_zero_conv_weights_give_the_identity_path():
    c = _dense_case()
    v = np.random.default_rng(1).standard_normal((c["B"], c["L"], c["d"]))
    alpha = np.random.default_rng(2).random((c["M"], c["B"], c["L"]))
    H = np.zeros_like(c["H"].numpy())
    out = dense.conv_residual(v, alpha, c["gc"].numpy(), np.zeros((c["d"], 4)), 3, 1e-6, H)
    assert (out == alpha[..., None] * v[None]).all()


def test_causality_of_the_whole_path():
    # Changing later tokens never changes earlier reads or outputs (explainer,
    # "怎么验证确实值得加？"; conv must be causal, section "一次 lookup").
    sp = spec(W.MODE_ENGRAM, K=4, r=16, rows=[[37] * 4, [41] * 4])
    rng = np.random.default_rng(11)
    B, L, d, M = 2, 30, 32, 2
    toks = rng.integers(0, 90, (B, L)).astype(np.int32)
    table = (rng.integers(-128, 128, (orc.total_rows(sp), 16)) / 64).astype(np.float32)
    Wm = rng.standard_normal(((1 + M) * d, 2 * 4 * 16)) * 0.05
    h = rng.standard_normal((M, B * L, d))
    w = rng.standard_normal((d, 4)) * 0.3
    ones = np.ones(d)

    def run(tk):
        e = orc.lookup(sp, tk, None, 90, table.view(np.uint8), orc.F32).astype(np.float64)
        v, alpha = dense.engram_gate(e, Wm, h, ones, ones, 1e-6, M)
        H = dense.conv_residual(v.reshape(B, L, d), alpha.reshape(M, B, L), ones, w, 3, 1e-6,
                                h.reshape(M, B, L, d))
        return e.reshape(B, L, -1), H

    e0, H0 = run(toks)
    t = 17
    pert = toks.copy()
    pert[0, t + 1:] = (pert[0, t + 1:] + 5) % 90
    e1, H1 = run(pert)
    assert (e0[0, :t + 1] == e1[0, :t + 1]).all() and (H0[:, 0, :t + 1] == H1[:, 0, :t + 1]).all()
    assert (e0[1] == e1[1]).all() and (H0[:, 1] == H1[:, 1]).all()
    assert not (H0[:, 0, t + 1:] == H1[:, 0, t + 1:]).all()


def test_hash_version_1_regression_values():
    # Stored by tests/golden/make_hash_golden.py from the oracle itself: guards
    # hash_version 1 against silent drift (not an external pin).
    import importlib.util
    p = os.path.join(GOLDEN, "make_hash_golden.py")
    spec_ = importlib.util.spec_from_file_location("mkg", p)
    mkg = importlib.util.module_from_spec(spec_)
    spec_.loader.exec_module(mkg)
    stored = {}
    for row in _golden_rows("hash_v1.txt"):
        cfg, name, i, o, k, r, s = row
        stored[(int(cfg), name, int(i), int(o), int(k))] = (int(r), int(s, 16))
    seen = 0
    for cfg in range(1, 6):
        w = W.make_workload(cfg)
        for sp in w.tables:
            _, rows, signs, _ = orc.index(sp, mkg.TOKENS, None, 50304)
            for (i, o, k), r in np.ndenumerate(rows):
                assert stored[(cfg, sp.name, i, o, k)] == (int(r), int(signs[i, o, k, 0]))
                seen += 1
    assert seen == len(stored)
