"""Seeded synthetic workloads for the hashed multi-head N-gram lookup.

This module holds configuration data (sizes, prime row counts) and seeded input
generators only. It contains none of the lookup's own arithmetic (no hashing, no
addressing, no gather, no projection): the CUDA path and the CPU oracle each
implement that independently and both receive these inputs.

Five workloads, shaped after the pages' own settings:

1. tiny, fp32, uniform IDs (vocab 1024, 4096 tokens); PageGram K=8 S=4 P_n=64
   r=64, plus flat (2 x 512 rows of width 256) and Engram-style (16 primes
   <= 2048) tables over the same tokens; W_V 256x1024.
2. PageGram 200M-parameter table in bf16 (PageGram tech report, section 4,
   "external table configuration": P_n = 48,823 / 48,821 prime pages at S=4);
   Zipf(1.1) IDs over vocab 50,304, batch 64x1024; W_V to d=768; scalar gate.
3. Engram-style (16 primes <= 195,312, r=64) and flat (2 x 130,208 rows of width
   768) tables at the same 200M budget, same tokens as 2.
4. 20B-parameter PageGram table in NF4 (34-byte rows; PageGram tech report,
   section 3.3): P_n = 4,882,811 / 4,882,789; vocab 128,000 folded to 98,010
   canonical IDs (23.43% smaller, Engram notes section 3.2); Zipf(1.05), 16x4096.
5. Engram-27B-shaped module (Engram notes section 3.7: d=2560, max order 3,
   8 heads, memory width 1280 -> r=80; mHC with M=4 branches, section 3.4):
   16 primes <= 2,226,562, bf16, Zipf(1.05) over 128k with canonical folding,
   batch 8x4096.

Synthetic stand-ins: the pages train on private corpora and trained tables; none
are available, so token streams are i.i.d. Zipf (rank = ID) or uniform, tables
hold int8/64 values (exact in bf16 and fp32) or random NF4 codes with an fp16
scale in [1, 2), and dense weights are N(0, 0.02).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np
import torch

MODE_FLAT, MODE_ENGRAM, MODE_PAGEGRAM = 0, 1, 2
HASH_MULXOR, HASH_TOY = 0, 1
DT_F32, DT_BF16, DT_NF4 = 0, 1, 2
GATE_NONE, GATE_SCALAR, GATE_CONTEXT = 0, 1, 2

NF4_ROW_BYTES = 34  # 64 four-bit codes + one fp16 scale
BASE_SEED = 20261202


def largest_primes(target: int, count: int) -> List[int]:
    """The `count` largest distinct primes <= target, in descending order
    (plain trial division; the configs need at most 16 primes)."""
    out: List[int] = []
    x = target
    while len(out) < count and x >= 2:
        if x < 4:
            prime = x >= 2
        elif x % 2 == 0:
            prime = False
        else:
            prime = True
            f = 3
            while f * f <= x:
                if x % f == 0:
                    prime = False
                    break
                f += 2
        if prime:
            out.append(x)
        x -= 1
    if len(out) < count:
        raise ValueError(f"fewer than {count} primes <= {target}")
    return out


@dataclasses.dataclass
class TableSpec:
    """One hashed table; fields map one-to-one onto the C-ABI table descriptor."""
    name: str
    mode: int
    K: int
    S: int
    r: int                       # head width (flat: row width = d)
    row_dtype: int
    orders: List[int] = dataclasses.field(default_factory=lambda: [2, 3])
    pages: List[int] = dataclasses.field(default_factory=list)          # PageGram P_n
    rows: List[List[int]] = dataclasses.field(default_factory=list)     # Engram M_{n,k}; flat [[R_n]]
    hash_kind: int = HASH_MULXOR
    hash_seed: int = 0

    @property
    def num_orders(self) -> int:
        return len(self.orders)

    @property
    def table_rows(self) -> int:
        """Number of stored rows (the table's first dimension)."""
        if self.mode == MODE_PAGEGRAM:
            return sum(p * self.K * self.S for p in self.pages)
        return sum(sum(rr) for rr in self.rows)

    @property
    def row_bytes(self) -> int:
        if self.row_dtype == DT_NF4:
            return NF4_ROW_BYTES
        return self.r * (4 if self.row_dtype == DT_F32 else 2)

    @property
    def table_bytes(self) -> int:
        return self.table_rows * self.row_bytes

    @property
    def e_width(self) -> int:
        """Width of e_t: concat of O*K heads of width r, or d for the flat sum."""
        if self.mode == MODE_FLAT:
            return self.r
        return self.num_orders * self.K * self.r


@dataclasses.dataclass
class Workload:
    cfg_id: int
    name: str
    B: int
    L: int
    vocab: int
    canon_vocab: Optional[int]   # None: identity canonical map
    zipf_s: Optional[float]      # None: uniform IDs
    tables: List[TableSpec]
    d: int
    dtype: int                   # dense dtype: DT_F32 or DT_BF16
    gate: int
    M: int = 0                   # branches (context gate)
    g: float = 0.5               # scalar gate value (its initial value in the PageGram report)
    eps: float = 1e-6
    dilation: int = 3
    conv_kernel: int = 4

    @property
    def N(self) -> int:
        return self.B * self.L


def _seed64(ss: np.random.SeedSequence) -> int:
    return int(ss.generate_state(1, np.uint64)[0]) & 0x7FFFFFFFFFFFFFFF


def _children(cfg_id: int) -> Dict[str, np.random.SeedSequence]:
    names = ["tokens", "canon", "dense", "table", "hash"]
    kids = np.random.SeedSequence(BASE_SEED + cfg_id).spawn(len(names))
    return dict(zip(names, kids))


def make_workload(cfg_id: int) -> Workload:
    hs = _seed64(_children(cfg_id)["hash"])
    if cfg_id == 1:
        eng = largest_primes(2048, 16)
        tables = [
            TableSpec("pagegram", MODE_PAGEGRAM, K=8, S=4, r=64, row_dtype=DT_F32,
                      pages=[64, 64], hash_seed=hs),
            TableSpec("flat", MODE_FLAT, K=1, S=1, r=256, row_dtype=DT_F32,
                      rows=[[512], [512]], hash_seed=hs),
            TableSpec("engram", MODE_ENGRAM, K=8, S=1, r=64, row_dtype=DT_F32,
                      rows=[eng[:8], eng[8:]], hash_seed=hs),
        ]
        return Workload(1, "tiny-fp32", B=1, L=4096, vocab=1024, canon_vocab=None,
                        zipf_s=None, tables=tables, d=256, dtype=DT_F32, gate=GATE_NONE)
    if cfg_id == 2:
        tables = [TableSpec("pagegram", MODE_PAGEGRAM, K=8, S=4, r=64, row_dtype=DT_BF16,
                            pages=[48823, 48821], hash_seed=hs)]
        return Workload(2, "pagegram-200M-bf16", B=64, L=1024, vocab=50304, canon_vocab=None,
                        zipf_s=1.1, tables=tables, d=768, dtype=DT_BF16, gate=GATE_SCALAR)
    if cfg_id == 3:
        hs2 = _seed64(_children(2)["hash"])  # same hash family as workload 2
        eng = largest_primes(195312, 16)
        tables = [
            TableSpec("engram", MODE_ENGRAM, K=8, S=1, r=64, row_dtype=DT_BF16,
                      rows=[eng[:8], eng[8:]], hash_seed=hs2),
            TableSpec("flat", MODE_FLAT, K=1, S=1, r=768, row_dtype=DT_BF16,
                      rows=[[130208], [130208]], hash_seed=hs2),
        ]
        return Workload(3, "engram-vs-flat-200M-bf16", B=64, L=1024, vocab=50304,
                        canon_vocab=None, zipf_s=1.1, tables=tables, d=768, dtype=DT_BF16,
                        gate=GATE_SCALAR)
    if cfg_id == 4:
        tables = [TableSpec("pagegram-nf4", MODE_PAGEGRAM, K=8, S=4, r=64, row_dtype=DT_NF4,
                            pages=largest_primes(4882812, 2), hash_seed=hs)]
        return Workload(4, "pagegram-20B-nf4", B=16, L=4096, vocab=128000,
                        canon_vocab=128000 - round(0.2343 * 128000), zipf_s=1.05,
                        tables=tables, d=1024, dtype=DT_BF16, gate=GATE_NONE)
    if cfg_id == 5:
        eng = largest_primes(2226562, 16)
        tables = [TableSpec("engram-27B", MODE_ENGRAM, K=8, S=1, r=80, row_dtype=DT_BF16,
                            rows=[eng[:8], eng[8:]], hash_seed=hs)]
        return Workload(5, "engram27b-module-bf16", B=8, L=4096, vocab=128000,
                        canon_vocab=128000 - round(0.2343 * 128000), zipf_s=1.05,
                        tables=tables, d=2560, dtype=DT_BF16, gate=GATE_CONTEXT, M=4)
    raise ValueError(f"unknown workload {cfg_id}")


# PageGram report section 4 evaluates S in {1, 4, 8, 15, 60} at a fixed table size.
SLOT_SWEEP = (1, 4, 8, 15, 60)


def pagegram_slots(S: int) -> TableSpec:
    """Workload 2's 200M-parameter PageGram table with S slots per head and page. The
    budget P_n K S r stays that of S = 4 (48,823 and 48,821 pages, report section 4): P_n
    are the two largest primes <= 48,823 * 4 / S, which for S = 4 are the report's."""
    base = make_workload(2).tables[0]
    return dataclasses.replace(base, S=S, pages=largest_primes((48823 * 4) // S, 2))


def distinct_ngrams(n: int, order: int, vocab: int, seed: int) -> np.ndarray:
    """n distinct n-grams, int32 [n, order]: the first n points of the base-m grid over
    `order` digits (m = the least integer with m ** order >= n), digit j mapped through
    its own seeded injection of [0, m) into [0, vocab)."""
    m = max(1, int(round(n ** (1.0 / order))))
    while m ** order < n:
        m += 1
    if m > vocab:
        raise ValueError("vocabulary too small for that many distinct n-grams")
    rng = np.random.default_rng(np.random.SeedSequence([BASE_SEED, 0x5EED, n, order, seed]))
    i = np.arange(n, dtype=np.int64)
    out = np.empty((n, order), np.int32)
    for j in range(order):
        digit = (i // m ** (order - 1 - j)) % m
        out[:, j] = rng.choice(vocab, size=m, replace=False)[digit]
    return out


def shrink(w: Workload, B: int, L: int) -> Workload:
    """Same tables and weights shape, fewer tokens (for oracle-sized tests)."""
    return dataclasses.replace(w, B=B, L=L)


# ----------------------------------------------------------------- generators

def zipf_ids(rng: np.random.Generator, V: int, s: float, n: int) -> np.ndarray:
    """i.i.d. IDs with P(id = i) proportional to (i+1)^-s, by inverse CDF."""
    p = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(p)
    cdf /= cdf[-1]
    u = rng.random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), V - 1).astype(np.int32)


def make_tokens(w: Workload, rank: int = 0, uniform: bool = False) -> np.ndarray:
    """int32 [B, L] token IDs. `rank` offsets the stream for data-parallel shards;
    `uniform` draws i.i.d. uniform IDs instead of the workload's Zipf stream (the
    no-reuse control: almost every row of the batch distinct)."""
    ss = _children(w.cfg_id)["tokens"]
    if rank:
        ss = np.random.SeedSequence([ss.entropy, 7919 * rank])
    if uniform:
        ss = np.random.SeedSequence([ss.entropy, 0x0C0FFEE])
    rng = np.random.Generator(np.random.PCG64(ss))
    n = w.B * w.L
    if w.zipf_s is None or uniform:
        ids = rng.integers(0, w.vocab, n, dtype=np.int64).astype(np.int32)
    else:
        ids = zipf_ids(rng, w.vocab, w.zipf_s, n)
    return ids.reshape(w.B, w.L)


def make_canon_map(w: Workload) -> Optional[np.ndarray]:
    """uint32 [V] surjection V -> V'. IDs < V' keep their value, the rest map
    uniformly at random into [0, V'); None for the identity map."""
    if w.canon_vocab is None:
        return None
    rng = np.random.Generator(np.random.PCG64(_children(w.cfg_id)["canon"]))
    m = np.arange(w.vocab, dtype=np.uint32)
    extra = w.vocab - w.canon_vocab
    m[w.canon_vocab:] = rng.integers(0, w.canon_vocab, extra, dtype=np.int64).astype(np.uint32)
    return m


def _torch_gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_table(w: Workload, spec: TableSpec, device="cpu") -> torch.Tensor:
    """The table contents. f32/bf16: [rows, r] with values int8/64 (exact in both
    types). NF4: uint8 [rows, 34] = 32 bytes of random codes + an fp16 scale
    1 + k/1024 (k uniform in [0, 1024)), little-endian."""
    idx = [t.name for t in w.tables].index(spec.name)
    ss = np.random.SeedSequence([_children(w.cfg_id)["table"].entropy, idx])
    gen = _torch_gen(_seed64(ss), device)
    R = spec.table_rows
    if spec.row_dtype == DT_NF4:
        codes = torch.randint(0, 256, (R, 32), dtype=torch.uint8, device=device, generator=gen)
        k = torch.randint(0, 1024, (R,), dtype=torch.int32, device=device, generator=gen)
        scale = (1.0 + k.to(torch.float32) / 1024.0).to(torch.float16)
        del k
        sb = scale.view(torch.uint8).view(R, 2)
        out = torch.cat([codes, sb], dim=1).contiguous()
        return out
    q = torch.randint(-128, 128, (R, spec.r), dtype=torch.int8, device=device, generator=gen)
    dt = torch.float32 if spec.row_dtype == DT_F32 else torch.bfloat16
    t = q.to(dt)
    del q
    t.div_(64.0)
    return t


def make_dense(w: Workload, device="cpu", zero_conv: bool = False) -> Dict[str, torch.Tensor]:
    """Dense weights and hidden states.

    W: [(1+M)*d, Din] (W_V rows then W_K^(1..M) rows), N(0, 0.02), where Din is
       the e_t width of the first table.
    x: [N, d] residual stream for the scalar gate, N(0, 1).
    H: [M, N, d] branch hidden states, N(0, 1); the context gate reads them as
       h^(m) and the conv residual adds Y into them.
    gamma_h, gamma_k, gamma_c: [d] ones (fp32). conv_w: [d, 4] N(0, 0.25) fp32.
    """
    ss = _children(w.cfg_id)["dense"]
    gen = _torch_gen(_seed64(ss), device)
    dt = torch.float32 if w.dtype == DT_F32 else torch.bfloat16
    din = w.tables[0].e_width
    rows = (1 + w.M) * w.d
    out: Dict[str, torch.Tensor] = {}
    out["W"] = (torch.randn(rows, din, generator=gen, device=device) * 0.02).to(dt)
    if w.gate == GATE_SCALAR:
        out["x"] = torch.randn(w.N, w.d, generator=gen, device=device).to(dt)
    if w.gate == GATE_CONTEXT:
        out["H"] = torch.randn(w.M, w.N, w.d, generator=gen, device=device).to(dt)
        out["gamma_h"] = torch.ones(w.d, device=device)
        out["gamma_k"] = torch.ones(w.d, device=device)
        out["gamma_c"] = torch.ones(w.d, device=device)
        if zero_conv:
            out["conv_w"] = torch.zeros(w.d, w.conv_kernel, device=device)
        else:
            out["conv_w"] = torch.randn(w.d, w.conv_kernel, generator=gen, device=device) * 0.25
    return out
