"""Shared test helpers: seeded inputs, oracle calls, comparisons."""
import dataclasses

import numpy as np
import torch

from hashed_head_gram_gb300 import workloads as W
from oracle import oracle as orc

BF16_TOL = 2e-2   # rel-L2 for bf16 outputs against the fp64 oracle
F32_TOL = 1e-5    # rel-L2 for fp32 outputs against the fp64 oracle


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def table_bytes_view(table: torch.Tensor, spec) -> torch.Tensor:
    """uint8 [rows, row_bytes] view of a table tensor (any device)."""
    return table.contiguous().view(torch.uint8).reshape(spec.table_rows, spec.row_bytes)


def oracle_e(spec, tokens: np.ndarray, cmap, vocab: int, table: torch.Tensor, out_dtype: int,
             which=None) -> np.ndarray:
    """Oracle e_t for the listed flat token indices (all when None). Rows are fetched
    from the table tensor by index (torch indexing on the input), so tables of any
    size work."""
    canon, rows, signs, bad = orc.index(spec, tokens, cmap, vocab, which)
    assert bad == -1
    tb = table_bytes_view(table, spec)
    flat = torch.from_numpy(rows.reshape(-1).astype(np.int64)).to(tb.device)
    rowdata = tb[flat].cpu().numpy().reshape(rows.shape + (spec.row_bytes,))
    return orc.assemble(spec, rows, rowdata, signs, out_dtype)


def small_engram(spec, primes_target=1100):
    """The same Engram-style table with small prime subtables (oracle-sized)."""
    p = W.largest_primes(primes_target, len(spec.orders) * spec.K)
    return dataclasses.replace(spec, rows=[p[i * spec.K:(i + 1) * spec.K] for i in range(len(spec.orders))])


def small_pagegram(spec, pages=(61, 59)):
    return dataclasses.replace(spec, pages=list(pages[:len(spec.orders)]))


def small_flat(spec, rows=(997, 991)):
    return dataclasses.replace(spec, rows=[[r] for r in rows[:len(spec.orders)]])


def shrink_table(spec):
    if spec.mode == W.MODE_ENGRAM:
        return small_engram(spec)
    if spec.mode == W.MODE_PAGEGRAM:
        return small_pagegram(spec)
    return small_flat(spec)


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def canon_tensor(cmap, dev):
    return None if cmap is None else torch.from_numpy(cmap.view(np.int32)).to(dev)
