"""ctypes wrapper around the C oracle (oracle/pg_oracle.c) -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU legs may use this module.

Functions take a table spec with the attributes mode, hash_kind, orders, K, S, r,
pages, rows, row_dtype and hash_seed (hashed_head_gram_gb300.workloads.TableSpec
has them) and plain numpy arrays. Nothing here calls the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pg_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

PAD = 0xFFFFFFFF
NO_ROW = 0xFFFFFFFF
F32, BF16, NF4 = 0, 1, 2
FLAT, ENGRAM, PAGEGRAM = 0, 1, 2
HASH_MULXOR, HASH_TOY = 0, 1


class OrcDesc(ctypes.Structure):
    _fields_ = [
        ("mode", ctypes.c_int32),
        ("hash_kind", ctypes.c_int32),
        ("num_orders", ctypes.c_int32),
        ("orders", ctypes.c_int32 * 4),
        ("K", ctypes.c_int32),
        ("S", ctypes.c_int32),
        ("r", ctypes.c_int32),
        ("pages", ctypes.c_uint32 * 4),
        ("rows", (ctypes.c_uint32 * 16) * 4),
        ("row_dtype", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
        ("seed", ctypes.c_uint64),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math, no FP contraction)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c99", "-fno-fast-math", "-ffp-contract=off",
                                   "-fPIC", "-shared", "-o", tmp, _SRC])
            os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u64, u32, i64, i32, vp = (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64,
                                  ctypes.c_int32, ctypes.c_void_p)
        L.orc_mix64.restype = u64; L.orc_mix64.argtypes = [u64]
        L.orc_multiplier.restype = u64
        L.orc_multiplier.argtypes = [u64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.orc_hash64.restype = u64
        L.orc_hash64.argtypes = [u64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp]
        L.orc_fold32.restype = u32; L.orc_fold32.argtypes = [u64]
        L.orc_sign_word.restype = u64; L.orc_sign_word.argtypes = [u64, ctypes.c_int]
        L.orc_toy_bucket.restype = u32; L.orc_toy_bucket.argtypes = [u32, u32, u32]
        L.orc_nf4_level.restype = ctypes.c_float; L.orc_nf4_level.argtypes = [ctypes.c_int]
        L.orc_f16_to_f32.restype = ctypes.c_float; L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16; L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        L.orc_bf16_to_f32.restype = ctypes.c_float; L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_f32_to_f16_sat.restype = ctypes.c_uint16; L.orc_f32_to_f16_sat.argtypes = [ctypes.c_float]
        L.orc_nf4_quantize.restype = None; L.orc_nf4_quantize.argtypes = [vp, i64, vp]
        L.orc_f32_to_e4m3_sat.restype = ctypes.c_uint8; L.orc_f32_to_e4m3_sat.argtypes = [ctypes.c_float]
        L.orc_e4m3_to_f32.restype = ctypes.c_float; L.orc_e4m3_to_f32.argtypes = [ctypes.c_uint8]
        L.orc_fp8_quantize.restype = None; L.orc_fp8_quantize.argtypes = [vp, i64, i64, vp, vp]
        L.orc_total_rows.restype = u64; L.orc_total_rows.argtypes = [ctypes.POINTER(OrcDesc)]
        L.orc_sign_words.restype = ctypes.c_int; L.orc_sign_words.argtypes = [ctypes.POINTER(OrcDesc)]
        L.orc_heads.restype = ctypes.c_int; L.orc_heads.argtypes = [ctypes.POINTER(OrcDesc)]
        L.orc_index.restype = i64
        L.orc_index.argtypes = [ctypes.POINTER(OrcDesc), vp, i64, i64, vp, u32, vp, i64, vp, vp, vp]
        L.orc_assemble.restype = ctypes.c_int
        L.orc_assemble.argtypes = [ctypes.POINTER(OrcDesc), i64, vp, vp, vp, ctypes.c_int, vp]
        _lib = L
    return _lib


def desc_of(spec) -> OrcDesc:
    d = OrcDesc()
    d.mode = spec.mode
    d.hash_kind = spec.hash_kind
    d.num_orders = len(spec.orders)
    for i, n in enumerate(spec.orders):
        d.orders[i] = n
    d.K, d.S, d.r = spec.K, spec.S, spec.r
    for i, p in enumerate(spec.pages):
        d.pages[i] = p
    for i, rr in enumerate(spec.rows):
        for k, m in enumerate(rr):
            d.rows[i][k] = m
    d.row_dtype = spec.row_dtype
    d.seed = spec.hash_seed & 0xFFFFFFFFFFFFFFFF
    return d


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def heads(spec) -> int:
    return 1 if spec.mode == FLAT else spec.K


def sign_words(spec) -> int:
    return (spec.r + 63) // 64


def row_bytes(spec) -> int:
    return 34 if spec.row_dtype == NF4 else spec.r * (4 if spec.row_dtype == F32 else 2)


def total_rows(spec) -> int:
    d = desc_of(spec)
    return int(lib().orc_total_rows(ctypes.byref(d)))


# ------------------------------------------------------------------ the pages' toy hash

def bigram_bucket(tokens: Sequence[int], table_size: int) -> int:
    """The Engram explainer's teaching bucket (section "Hash 冲突是什么样？"):
    (3a + b) mod m for exactly two non-negative integer IDs and a positive
    integer table size; anything else raises ValueError."""
    if len(tokens) != 2 or type(table_size) is not int or table_size <= 0:
        raise ValueError("need exactly two IDs and a positive integer table size")
    for tok in tokens:
        if type(tok) is not int or tok < 0:
            raise ValueError("token IDs must be non-negative integers")
    return int(lib().orc_toy_bucket(tokens[0], tokens[1], table_size))


# ------------------------------------------------------------------ lookup stages

def index(spec, tokens: np.ndarray, canon_map: Optional[np.ndarray], vocab: int,
          which: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray, np.ndarray, int]:
    """Canonical IDs, rows [n, O, H] (uint32) and sign words [n, O, H, W] (uint64)
    for all tokens of the [B, L] array, or for the listed flat indices. Returns
    (canon, rows, signs, first_bad_index_or_-1)."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    B, L = tokens.shape
    cm = None if canon_map is None else np.ascontiguousarray(canon_map, dtype=np.uint32)
    wh = None if which is None else np.ascontiguousarray(which, dtype=np.int64)
    n = B * L if wh is None else len(wh)
    O, H, W = len(spec.orders), heads(spec), sign_words(spec)
    canon = np.zeros(n, np.uint32)
    rows = np.zeros((n, O, H), np.uint32)
    signs = np.zeros((n, O, H, W), np.uint64)
    d = desc_of(spec)
    bad = lib().orc_index(ctypes.byref(d), _ptr(tokens), B, L, _ptr(cm), vocab, _ptr(wh),
                          0 if wh is None else len(wh), _ptr(canon), _ptr(rows), _ptr(signs))
    return canon, rows, signs, int(bad)


def fetch_rows(table_bytes: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """Stored bytes of each addressed row: table_bytes is uint8 [R, row_bytes];
    ORC NO_ROW entries fetch zeros."""
    flat = rows.reshape(-1)
    out = np.zeros((flat.size, table_bytes.shape[1]), np.uint8)
    ok = flat != NO_ROW
    out[ok] = table_bytes[flat[ok].astype(np.int64)]
    return out.reshape(rows.shape + (table_bytes.shape[1],))


def assemble(spec, rows: np.ndarray, rowdata: np.ndarray, signs: np.ndarray,
             out_dtype: int) -> np.ndarray:
    """e_t from fetched rows: float32 [n, width], or bf16 bits as uint16 [n, width]."""
    n = rows.shape[0]
    width = spec.r if spec.mode == FLAT else len(spec.orders) * heads(spec) * spec.r
    out = np.zeros((n, width), np.float32 if out_dtype == F32 else np.uint16)
    d = desc_of(spec)
    rc = lib().orc_assemble(ctypes.byref(d), n, _ptr(np.ascontiguousarray(rows)),
                            _ptr(np.ascontiguousarray(rowdata)),
                            _ptr(np.ascontiguousarray(signs)), out_dtype, _ptr(out))
    if rc != 0:
        raise ValueError("unsupported row/output dtype combination")
    return out


def lookup(spec, tokens: np.ndarray, canon_map: Optional[np.ndarray], vocab: int,
           table_bytes: np.ndarray, out_dtype: int, which: Optional[np.ndarray] = None):
    """Full lookup e_t (index -> fetch -> assemble); raises ValueError on a token
    ID outside [0, vocab), as the explainer's bucket function does."""
    canon, rows, signs, bad = index(spec, tokens, canon_map, vocab, which)
    if bad >= 0:
        raise ValueError(f"token ID out of range at flat index {bad}")
    return assemble(spec, rows, fetch_rows(table_bytes, rows), signs, out_dtype)


# ------------------------------------------------------------------ number helpers

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    f = lib().orc_f32_to_bf16
    flat = np.ascontiguousarray(x, np.float32).reshape(-1)
    return np.array([f(float(v)) for v in flat], np.uint16).reshape(np.shape(x))


def nf4_levels() -> np.ndarray:
    return np.array([lib().orc_nf4_level(c) for c in range(16)], np.float32)


def f32_to_f16_sat(x: float) -> int:
    """fp16 bits of x: round to nearest, ties to even, saturating at +-65504 (R15)."""
    return int(lib().orc_f32_to_f16_sat(float(x)))


def nf4_quantize(x: np.ndarray) -> np.ndarray:
    """NF4 export (PageGram report 3.3; QLoRA's absmax quantisation, reading R15):
    x [n, 64] fp32 -> [n, 34] uint8 rows in the R6 layout."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.ndim == 2 and x.shape[1] == 64
    out = np.zeros((x.shape[0], 34), np.uint8)
    lib().orc_nf4_quantize(x.ctypes.data, x.shape[0], out.ctypes.data)
    return out


def nf4_dequantize(rows: np.ndarray) -> np.ndarray:
    """[n, 34] NF4 rows -> [n, 64] fp32 values level[code] * float(scale) (R6)."""
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    lv = nf4_levels()
    codes = np.empty((rows.shape[0], 64), np.int64)
    codes[:, 0::2] = rows[:, :32] & 15
    codes[:, 1::2] = rows[:, :32] >> 4
    sbits = rows[:, 32].astype(np.uint16) | (rows[:, 33].astype(np.uint16) << 8)
    scale = np.array([lib().orc_f16_to_f32(int(b)) for b in sbits], np.float32)
    return (lv[codes] * scale[:, None]).astype(np.float32)


def f32_to_e4m3_sat(x: float) -> int:
    """OCP FP8 E4M3 bits of x: round to nearest, ties to even, saturating at +-448 (R16)."""
    return int(lib().orc_f32_to_e4m3_sat(float(x)))


def e4m3_to_f32(b: np.ndarray) -> np.ndarray:
    """Values of E4M3 bytes (exact in fp32)."""
    table = np.array([lib().orc_e4m3_to_f32(i) for i in range(256)], np.float32)
    return table[np.asarray(b, np.uint8)]


def fp8_quantize(x: np.ndarray):
    """FP8 projection operand (reading R16, Engram notes 3.4): rows of x [n, cols] fp32 ->
    (E4M3 bytes [n, cols], fp32 scales [n]) with value ~= e4m3(q) * scale."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n, cols = x.shape
    q = np.zeros((n, cols), np.uint8)
    s = np.zeros(n, np.float32)
    lib().orc_fp8_quantize(x.ctypes.data, n, cols, q.ctypes.data, s.ctypes.data)
    return q, s


def fp8_dequantize(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """fp64 values e4m3(q) * scale of FP8 rows (both factors exact in fp64)."""
    return e4m3_to_f32(q).astype(np.float64) * np.asarray(s, np.float64)[:, None]


# ------------------------------------------------------------------ correlated collisions

def collision_counts(rows: np.ndarray) -> Tuple[int, np.ndarray]:
    """Head-collision counts over a set of distinct n-grams of one order (PageGram report
    3.2, measured in 6.1): rows [n, K] holds each n-gram's K head rows. Over all unordered
    pairs {i, j}: shared[k] = #pairs whose head-0 rows are equal and whose head-k rows are
    equal; shared[0] = pairs0 = #pairs colliding on head 0. The mean number of further
    heads a head-0 collision shares is sum(shared[1:]) / pairs0, which the report derives
    as (K - 1) / S for PageGram and which is about (K - 1) / M_{n,k} for independent
    Engram-style subtables. Definition written out: for each head k, count the equal
    (row_0, row_k) keys and add C(c, 2) for every key seen c times."""
    r = np.asarray(rows).astype(np.uint64)
    n, K = r.shape
    shared = np.zeros(K, np.int64)
    for k in range(K):
        key = (r[:, 0] << np.uint64(32)) | r[:, k]
        _, c = np.unique(key, return_counts=True)
        c = c.astype(np.int64)
        shared[k] = int((c * (c - 1) // 2).sum())
    return int(shared[0]), shared
