"""GPU parity of pg_canon_hash and pg_gather_sign_concat against the CPU oracle:
indices, sign words and gathered rows must match bit for bit."""
import dataclasses

import numpy as np
import pytest
import torch

from hashed_head_gram_gb300 import workloads as W
from oracle import oracle as orc
from tests._helpers import bits16, canon_tensor, oracle_e, shrink_table

pytestmark = pytest.mark.gpu

CASES = [(cfg, i) for cfg in range(1, 6) for i in range(len(W.make_workload(cfg).tables))]


def _pg():
    from hashed_head_gram_gb300 import pg
    return pg


def _inputs(cfg, ti, B=3, L=517, small=True):
    w = W.shrink(W.make_workload(cfg), B=B, L=L)
    spec = w.tables[ti]
    if small:
        spec = shrink_table(spec)
    return w, spec, W.make_tokens(w), W.make_canon_map(w)


@pytest.mark.parametrize("cfg,ti", CASES)
def test_canon_hash_matches_oracle(cuda, cfg, ti):
    pg = _pg()
    w, spec, tokens, cmap = _inputs(cfg, ti, small=False)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    O, H, Wd = len(spec.orders), orc.heads(spec), orc.sign_words(spec)
    tok = torch.from_numpy(tokens).to(cuda)
    rows = torch.empty(w.N, O, H, dtype=torch.int32, device=cuda)
    signs = torch.empty(w.N, O, H, Wd, dtype=torch.int64, device=cuda)
    canon = torch.empty(w.N, dtype=torch.int32, device=cuda)
    err = torch.empty(1, dtype=torch.int32, device=cuda)
    pg.canon_hash(desc, tok, rows, canon_map=canon_tensor(cmap, cuda), canon_out=canon, sign_out=signs,
                  err_index=err)
    torch.cuda.synchronize()
    c_ref, r_ref, s_ref, bad = orc.index(spec, tokens, cmap, w.vocab)
    assert bad == -1 and err.item() == -1
    assert np.array_equal(canon.cpu().numpy().view(np.uint32), c_ref)
    assert np.array_equal(rows.cpu().numpy().view(np.uint32), r_ref)
    assert np.array_equal(signs.cpu().numpy().view(np.uint64), s_ref)


@pytest.mark.parametrize("cfg,ti", CASES)
def test_gather_matches_oracle(cuda, cfg, ti):
    pg = _pg()
    w, spec, tokens, cmap = _inputs(cfg, ti)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    table = W.make_table(w, spec, "cpu")
    out_dtype = orc.F32 if spec.row_dtype == orc.F32 else orc.BF16
    ref = oracle_e(spec, tokens, cmap, w.vocab, table, out_dtype)
    e = torch.empty(w.N, spec.e_width, dtype=torch.float32 if out_dtype == orc.F32 else torch.bfloat16,
                    device=cuda)
    err = torch.empty(1, dtype=torch.int32, device=cuda)
    pg.gather_sign_concat(desc, torch.from_numpy(tokens).to(cuda), table.to(cuda), e, out_dtype,
                          canon_map=canon_tensor(cmap, cuda), err_index=err)
    torch.cuda.synchronize()
    assert err.item() == -1
    got = e.cpu().numpy() if out_dtype == orc.F32 else bits16(e)
    if out_dtype == orc.F32:
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    else:
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("cfg,ti", [(2, 0), (4, 0), (3, 1)])
def test_gather_f32_output_of_narrow_rows(cuda, cfg, ti):
    # bf16 and NF4 rows written widened to fp32 (same values, exact).
    pg = _pg()
    w, spec, tokens, cmap = _inputs(cfg, ti, B=2, L=300)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    table = W.make_table(w, spec, "cpu")
    ref = oracle_e(spec, tokens, cmap, w.vocab, table, orc.F32)
    e = torch.empty(w.N, spec.e_width, dtype=torch.float32, device=cuda)
    pg.gather_sign_concat(desc, torch.from_numpy(tokens).to(cuda), table.to(cuda), e, orc.F32,
                          canon_map=canon_tensor(cmap, cuda))
    assert np.array_equal(e.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_toy_hash_on_the_gpu(cuda):
    pg = _pg()
    toks = np.array([[1, 2, 4, 9, 0, 3]], np.int32)
    for m in (5, 7, 1000003):
        spec = W.TableSpec("toy", W.MODE_FLAT, K=1, S=1, r=64, row_dtype=W.DT_BF16, orders=[2],
                           rows=[[m]], hash_kind=W.HASH_TOY)
        desc = pg.table_desc(spec, 16)
        rows = torch.empty(1, 6, 1, 1, dtype=torch.int32, device=cuda)
        pg.canon_hash(desc, torch.from_numpy(toks).to(cuda), rows)
        _, ref, _, _ = orc.index(spec, toks, None, 16)
        assert np.array_equal(rows.cpu().numpy().view(np.uint32).reshape(-1), ref.reshape(-1))
    if True:  # the explainer's worked values, through the GPU path
        spec = W.TableSpec("toy", W.MODE_FLAT, K=1, S=1, r=64, row_dtype=W.DT_BF16, orders=[2],
                           rows=[[7]], hash_kind=W.HASH_TOY)
        rows = torch.empty(3, dtype=torch.int32, device=cuda)
        pg.canon_hash(pg.table_desc(spec, 16), torch.tensor([[1, 2, 4]], dtype=torch.int32, device=cuda), rows)
        assert rows.cpu().numpy().view(np.uint32)[1:].tolist() == [5, 3]


@pytest.mark.parametrize("cfg", [2, 5, 4])  # two-token batches, one-token batches, NF4 rows
def test_out_of_range_tokens_are_reported_and_clamped(cuda, cfg):
    pg = _pg()
    w, spec, tokens, cmap = _inputs(cfg, 0, B=4, L=100)
    tokens = tokens.copy()
    tokens[2, 50] = w.vocab + 5
    tokens[3, 7] = -1
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    table = W.make_table(w, spec, "cpu")
    e = torch.empty(w.N, spec.e_width, dtype=torch.bfloat16, device=cuda)
    err = torch.empty(1, dtype=torch.int32, device=cuda)
    pg.gather_sign_concat(desc, torch.from_numpy(tokens).to(cuda), table.to(cuda), e, orc.BF16,
                          canon_map=canon_tensor(cmap, cuda), err_index=err)
    torch.cuda.synchronize()
    assert err.item() == 2 * 100 + 50
    # tokens whose windows avoid the bad IDs still match the oracle
    good = np.array([i for i in range(w.N) if not (250 <= i <= 252 or 307 <= i <= 309)])
    ref = oracle_e(spec, tokens.clip(0, w.vocab - 1), cmap, w.vocab, table, orc.BF16, which=good)
    assert np.array_equal(bits16(e)[good], ref)


def test_empty_batch_is_a_no_op(cuda):
    pg = _pg()
    w, spec, _, _ = _inputs(2, 0, B=1, L=10)
    desc = pg.table_desc(spec, w.vocab)
    table = W.make_table(w, spec, "cpu").to(cuda)
    e = torch.full((1, spec.e_width), 7.0, dtype=torch.bfloat16, device=cuda)
    before = pg.launch_count()
    pg.gather_sign_concat(desc, torch.empty(0, 10, dtype=torch.int32, device=cuda), table, e, orc.BF16)
    assert pg.launch_count() == before and (e == 7.0).all()


def test_host_rejects_bad_arguments(cuda):
    pg = _pg()
    w, spec, tokens, _ = _inputs(2, 0, B=1, L=16)
    table = W.make_table(w, spec, "cpu").to(cuda)
    tok = torch.from_numpy(tokens).to(cuda)
    e = torch.empty(w.N, spec.e_width, dtype=torch.bfloat16, device=cuda)
    desc = pg.table_desc(spec, w.vocab)
    with pytest.raises(pg.PgError) as ex:
        pg.gather_sign_concat(desc, tok, table[:-1], e, orc.BF16)      # table too small
    assert ex.value.status == 4
    bad = pg.table_desc(spec, w.vocab)
    bad.hash_version = 2
    with pytest.raises(pg.PgError) as ex:
        pg.gather_sign_concat(bad, tok, table, e, orc.BF16)
    assert ex.value.status == 7
    with pytest.raises(pg.PgError) as ex:
        pg.gather_sign_concat(desc, tok, table, e, orc.NF4)
    assert ex.value.status == 3


def test_gather_is_causal(cuda):
    pg = _pg()
    w, spec, tokens, cmap = _inputs(5, 0, B=2, L=200)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    table = W.make_table(w, spec, "cpu").to(cuda)
    cm = canon_tensor(cmap, cuda)
    outs = []
    for pert in (False, True):
        tk = tokens.copy()
        if pert:
            tk[0, 120:] = (tk[0, 120:] + 11) % w.vocab
        e = torch.empty(w.N, spec.e_width, dtype=torch.bfloat16, device=cuda)
        pg.gather_sign_concat(desc, torch.from_numpy(tk).to(cuda), table, e, orc.BF16, canon_map=cm)
        outs.append(bits16(e).reshape(2, 200, -1))
    assert np.array_equal(outs[0][0, :120], outs[1][0, :120])
    assert np.array_equal(outs[0][1], outs[1][1])
    assert not np.array_equal(outs[0][0, 120:], outs[1][0, 120:])


# Layouts other than the workloads' (so the runtime-geometry gather runs): head counts,
# widths, slots, order sets and dtypes the compile-time variants do not cover.
OTHER_LAYOUTS = [
    dict(mode=W.MODE_PAGEGRAM, K=4, S=2, r=32, dt=W.DT_BF16, orders=[2, 3], pages=[37, 31]),
    dict(mode=W.MODE_PAGEGRAM, K=16, S=1, r=64, dt=W.DT_BF16, orders=[2, 3], pages=[11, 13]),
    dict(mode=W.MODE_ENGRAM, K=3, S=1, r=128, dt=W.DT_BF16, orders=[1, 2, 4], rows=None),
    dict(mode=W.MODE_ENGRAM, K=8, S=1, r=64, dt=W.DT_F32, orders=[2], rows=None),
    dict(mode=W.MODE_PAGEGRAM, K=4, S=15, r=64, dt=W.DT_NF4, orders=[2, 3, 4], pages=[7, 5, 3]),
    dict(mode=W.MODE_FLAT, K=1, S=1, r=512, dt=W.DT_BF16, orders=[2, 3, 4], rows=[[211], [199], [197]]),
    dict(mode=W.MODE_FLAT, K=1, S=1, r=128, dt=W.DT_F32, orders=[3], rows=[[101]]),
    dict(mode=W.MODE_ENGRAM, K=2, S=1, r=1024, dt=W.DT_BF16, orders=[2, 3], rows=None),
    # degenerate addressing: one page per order (every n-gram in page 0), one row per order
    dict(mode=W.MODE_PAGEGRAM, K=8, S=4, r=64, dt=W.DT_BF16, orders=[2, 3], pages=[1, 1]),
    dict(mode=W.MODE_FLAT, K=1, S=1, r=64, dt=W.DT_BF16, orders=[2, 3], rows=[[1], [1]]),
]


@pytest.mark.parametrize("lay", range(len(OTHER_LAYOUTS)))
def test_gather_other_layouts(cuda, lay):
    pg = _pg()
    d = dict(OTHER_LAYOUTS[lay])
    rows = d.pop("rows", None)
    if d["mode"] == W.MODE_ENGRAM:
        pr = W.largest_primes(997, len(d["orders"]) * d["K"])
        rows = [pr[i * d["K"]:(i + 1) * d["K"]] for i in range(len(d["orders"]))]
    spec = W.TableSpec("t", d["mode"], K=d["K"], S=d["S"], r=d["r"], row_dtype=d["dt"], orders=d["orders"],
                       pages=d.get("pages", []), rows=rows or [], hash_seed=0xC0FFEE + lay)
    w = W.shrink(W.make_workload(2), B=3, L=211)
    tokens = W.make_tokens(w)
    table = torch.randint(-128, 128, (spec.table_rows, spec.r), dtype=torch.int8,
                          generator=torch.Generator().manual_seed(lay))
    if spec.row_dtype == W.DT_NF4:
        table = torch.randint(0, 256, (spec.table_rows, 34), dtype=torch.uint8,
                              generator=torch.Generator().manual_seed(lay))
        table[:, 33] = 0x3C     # scale 1.0 .. 1.99: keeps the fp16 scale finite
    else:
        table = (table.float() / 64).to(torch.float32 if spec.row_dtype == W.DT_F32 else torch.bfloat16)
    out_dtypes = [orc.F32] if spec.row_dtype == W.DT_F32 else [orc.BF16, orc.F32]
    desc = pg.table_desc(spec, w.vocab)
    for od in out_dtypes:
        ref = oracle_e(spec, tokens, None, w.vocab, table, od)
        e = torch.empty(w.N, spec.e_width, dtype=torch.float32 if od == orc.F32 else torch.bfloat16, device=cuda)
        pg.gather_sign_concat(desc, torch.from_numpy(tokens).to(cuda), table.to(cuda), e, od)
        got = e.cpu().numpy().view(np.uint32) if od == orc.F32 else bits16(e)
        assert np.array_equal(got, ref.view(np.uint32) if od == orc.F32 else ref), (lay, od)


def test_nf4_levels_on_the_gpu_match_the_oracle(cuda):
    # One row per code value with scale 1.0: the GPU's level table, read back through the
    # gather, equals the oracle's (each side holds its own copy of the NF4 levels).
    pg = _pg()
    spec = W.TableSpec("t", W.MODE_PAGEGRAM, K=1, S=1, r=64, row_dtype=W.DT_NF4, orders=[1], pages=[1],
                       hash_seed=3)
    tab = torch.zeros(1, 34, dtype=torch.uint8)
    tab[0, :32] = torch.tensor([(2 * i % 16) | (((2 * i + 1) % 16) << 4) for i in range(32)], dtype=torch.uint8)
    tab[0, 32:] = torch.tensor([0x00, 0x3C], dtype=torch.uint8)   # fp16 1.0, little-endian
    tokens = np.array([[5]], np.int32)
    e = torch.empty(1, 64, dtype=torch.float32, device=cuda)
    pg.gather_sign_concat(pg.table_desc(spec, 16), torch.from_numpy(tokens).to(cuda), tab.to(cuda), e, orc.F32)
    _, _, signs, _ = orc.index(spec, tokens, None, 16)
    lv = orc.nf4_levels()
    bits = (signs[0, 0, 0, 0] >> np.arange(64, dtype=np.uint64)) & np.uint64(1)
    want = np.where(bits == 1, -1.0, 1.0).astype(np.float32) * lv[np.arange(64) % 16]
    assert np.array_equal(np.abs(e.cpu().numpy()[0]), np.abs(want))
    assert np.array_equal(e.cpu().numpy()[0].view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("row_bytes,out_row", [(128, 0), (160, 0), (34, 0), (34, 128), (256, 0), (16, 0), (16, 48)])
def test_row_copy_moves_each_rows_window(cuda, row_bytes, out_row):
    # The diagnostic row copy: output row i = the aligned 16-byte window holding row
    # rows[i], zero-padded to the output row; chunks past the table's end (a row index
    # beyond it, or the table's ragged tail) are zeros. Checked byte for byte on the host.
    pg = _pg()
    g = torch.Generator().manual_seed(row_bytes + out_row)
    R, n = 1001, 3000
    table = torch.randint(0, 256, (R * row_bytes + 5,), dtype=torch.uint8, generator=g)
    rows = torch.randint(0, R, (n,), dtype=torch.int32, generator=g)
    rows[7] = R + 50
    rows[8] = R - 1
    wb = pg.row_copy_window(row_bytes)
    ob = out_row or wb
    out = torch.full((n, ob), 7, dtype=torch.uint8, device=cuda)
    pg.row_copy(table.to(cuda), row_bytes, rows.to(cuda), out, out_row)
    tb = table.numpy()
    want = np.zeros((n, ob), np.uint8)
    for i, r in enumerate(rows.numpy().astype(np.int64)):
        start = (r * row_bytes) & ~15
        for c in range(wb // 16):
            a = start + 16 * c
            if a + 16 <= tb.size:
                want[i, 16 * c:16 * c + 16] = tb[a:a + 16]
    assert np.array_equal(out.cpu().numpy(), want)
    for i, r in enumerate(rows.numpy()[:64].astype(np.int64)):  # the window holds the row
        s = r * row_bytes
        if s + row_bytes <= (tb.size // 16) * 16:
            assert np.array_equal(want[i, s % 16:s % 16 + row_bytes], tb[s:s + row_bytes])
