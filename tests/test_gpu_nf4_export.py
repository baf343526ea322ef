"""pg_nf4_quantize (NF4 export, PageGram report 3.3 / 9.4 check 5): the 34-byte rows are
bit-identical to the oracle's, and an exported table reads back through the NF4 gather
exactly as the oracle assembles it."""
import numpy as np
import pytest
import torch

from hashed_head_gram_gb300 import workloads as W
from oracle import oracle as orc
from tests._helpers import bits16, oracle_e, shrink_table

pytestmark = pytest.mark.gpu


def _pg():
    from hashed_head_gram_gb300 import pg
    return pg


def _rows(kind, n, rng):
    x = {"normal": rng.standard_normal((n, 64)),
         "heavy": rng.standard_t(1.5, (n, 64)),
         "tiny": rng.standard_normal((n, 64)) * 1e-7,          # scales in the fp16 subnormal range
         "huge": rng.standard_normal((n, 64)) * 3e4,           # scales past 65504 saturate
         "sparse": rng.standard_normal((n, 64)) * (rng.random((n, 64)) < 0.05),
         "zero": np.zeros((n, 64))}[kind].astype(np.float32)
    if kind == "normal":
        lv = orc.nf4_levels()                                  # rows of exact levels, ties included
        codes = rng.integers(0, 16, (n // 4, 64))
        codes[:, 0] = 15
        x[: n // 4] = lv[codes] * np.float32(0.5)
        mid = ((lv[:-1] + lv[1:]) / 2).astype(np.float32)      # midpoints between adjacent levels
        x[n // 4: n // 4 + 1, :15] = mid
        x[n // 4, 15] = 1.0
    return x


@pytest.mark.parametrize("kind", ["normal", "heavy", "tiny", "huge", "sparse", "zero"])
@pytest.mark.parametrize("n", [1, 37, 10007])
def test_export_matches_the_oracle_bit_for_bit(cuda, kind, n):
    pg = _pg()
    x = _rows(kind, n, np.random.default_rng(n + len(kind)))
    out = torch.full((n, 34), 0xAB, dtype=torch.uint8, device=cuda)
    pg.nf4_quantize(torch.from_numpy(x).to(cuda), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), orc.nf4_quantize(x))


def test_exported_table_reads_back_through_the_nf4_gather(cuda):
    # the 20B-parameter workload's NF4 layout at a small size: fp32 rows exported on the GPU,
    # then gathered, signed and concatenated; compared with the oracle on the same bytes
    pg = _pg()
    w = W.shrink(W.make_workload(4), B=2, L=300)
    spec = shrink_table(w.tables[0])
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((spec.table_rows, 64)) * rng.uniform(0.01, 10, (spec.table_rows, 1))).astype(np.float32)
    table = torch.empty(spec.table_rows, 34, dtype=torch.uint8, device=cuda)
    pg.nf4_quantize(torch.from_numpy(x).to(cuda), table)
    tokens = W.make_tokens(w)
    cmap = W.make_canon_map(w)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    e = torch.empty(w.N, spec.e_width, dtype=torch.bfloat16, device=cuda)
    cm = None if cmap is None else torch.from_numpy(cmap.view(np.int32)).to(cuda)
    pg.gather_sign_concat(desc, torch.from_numpy(tokens).to(cuda), table, e, orc.BF16, canon_map=cm)
    torch.cuda.synchronize()
    ref = oracle_e(spec, tokens, cmap, w.vocab, table.cpu(), orc.BF16)
    assert np.array_equal(bits16(e), ref)


def test_export_rejects_what_it_does_not_cover(cuda):
    pg = _pg()
    x = torch.zeros(8, 64, device=cuda)
    out = torch.empty(8, 34, dtype=torch.uint8, device=cuda)
    with pytest.raises(pg.PgError) as ex:
        pg.nf4_quantize(torch.zeros(8, 80, device=cuda), torch.empty(8, 34, dtype=torch.uint8, device=cuda))
    assert ex.value.status == 6
    with pytest.raises(pg.PgError) as ex:
        pg.nf4_quantize(x.view(-1)[1:1 + 7 * 64].view(7, 64), out)     # 4-byte aligned only
    assert ex.value.status == 5
    pg.nf4_quantize(x[:0], out[:0])                                     # nothing to do
