"""Thin Python binding of libpg.so (include/pg.h): argument marshalling only.

Every function takes torch tensors that live on the current CUDA device, passes
their data pointers and sizes through the C ABI, and raises PgError on a non-zero
status. All computation happens in the library's CUDA kernels; nothing here
computes or falls back to anything. When libpg.so is missing the import fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpg.so")

PG_ABI_VERSION = 1
PG_HASH_VERSION = 1
PG_MAX_ORDERS = 4
PG_MAX_HEADS = 16
PG_NO_ROW = 0xFFFFFFFF
FLAT, ENGRAM, PAGEGRAM = 0, 1, 2
HASH_MULXOR, HASH_TOY = 0, 1
F32, BF16, NF4 = 0, 1, 2
GATE_NONE, GATE_SCALAR, GATE_CONTEXT = 0, 1, 2

STATUS = {0: "PG_OK", 1: "PG_ERR_NULL", 2: "PG_ERR_SHAPE", 3: "PG_ERR_DTYPE", 4: "PG_ERR_RANGE",
          5: "PG_ERR_ALIGN", 6: "PG_ERR_UNSUPPORTED", 7: "PG_ERR_VERSION", 8: "PG_ERR_WORKSPACE",
          9: "PG_ERR_CUDA", 10: "PG_ERR_DEVICE", 11: "PG_ERR_SCRATCH_LIMIT"}


class PgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.pg_status_str(status).decode() if _lib is not None else ""
        extra = f", cuda error {_lib.pg_last_cuda_error()}" if status == 9 and _lib is not None else ""
        super().__init__(f"{where}: {STATUS.get(status, status)} ({msg}{extra})")


class TableDesc(ctypes.Structure):
    _fields_ = [
        ("abi_version", ctypes.c_uint32),
        ("hash_version", ctypes.c_uint32),
        ("mode", ctypes.c_int32),
        ("hash_kind", ctypes.c_int32),
        ("num_orders", ctypes.c_int32),
        ("orders", ctypes.c_int32 * PG_MAX_ORDERS),
        ("K", ctypes.c_int32),
        ("S", ctypes.c_int32),
        ("r", ctypes.c_int32),
        ("pages", ctypes.c_uint32 * PG_MAX_ORDERS),
        ("rows", (ctypes.c_uint32 * PG_MAX_HEADS) * PG_MAX_ORDERS),
        ("row_dtype", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("hash_seed", ctypes.c_uint64),
        ("vocab", ctypes.c_uint32),
        ("canon_vocab", ctypes.c_uint32),
    ]


class DecodeStateC(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("M", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("kernel_size", ctypes.c_int32),
        ("dilation", ctypes.c_int32),
        ("depth", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("pos", ctypes.c_void_p),
        ("ids", ctypes.c_void_p),
        ("ring_v", ctypes.c_void_p),
        ("ring_alpha", ctypes.c_void_p),
        ("ring_ms", ctypes.c_void_p),
    ]



class DecodeStepArgsC(ctypes.Structure):
    _fields_ = [
        ("W", ctypes.c_void_p),
        ("d", ctypes.c_int32),
        ("gate_kind", ctypes.c_int32),
        ("g", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("x_resid", ctypes.c_void_p),
        ("H", ctypes.c_void_p),
        ("gamma_h", ctypes.c_void_p),
        ("gamma_k", ctypes.c_void_p),
        ("gamma_c", ctypes.c_void_p),
        ("conv_w", ctypes.c_void_p),
        ("e_out", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("alpha_out", ctypes.c_void_p),
        ("v_ms_out", ctypes.c_void_p),
    ]

def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libpg.so is not built ({_LIB_PATH}); run `python -m hashed_head_gram_gb300.build`")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i32, u32, u64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint64,
                                  ctypes.c_float, ctypes.c_size_t)
    dp = ctypes.POINTER(TableDesc)
    L.pg_status_str.restype = ctypes.c_char_p
    L.pg_status_str.argtypes = [ctypes.c_int]
    L.pg_abi_version.restype = u32
    L.pg_last_cuda_error.restype = i32
    L.pg_launch_count.restype = u64
    L.pg_device_error.restype = ctypes.c_int
    L.pg_device_error.argtypes = [ctypes.POINTER(i32), i32]
    L.pg_table_geometry.restype = ctypes.c_int
    L.pg_table_geometry.argtypes = [dp, ctypes.POINTER(u64), ctypes.POINTER(u32), ctypes.POINTER(u32)]
    L.pg_canon_hash.restype = ctypes.c_int
    L.pg_canon_hash.argtypes = [dp, vp, i32, i32, vp, vp, vp, vp, vp, vp]
    L.pg_gather_sign_concat.restype = ctypes.c_int
    L.pg_gather_sign_concat.argtypes = [dp, vp, i32, i32, vp, vp, u64, vp, i32, vp, vp]
    L.pg_project_gate_workspace_size.restype = ctypes.c_int
    L.pg_project_gate_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(sz)]
    L.pg_project_gate.restype = ctypes.c_int
    L.pg_project_gate.argtypes = [i32, i32, i32, i32, i32, vp, vp, i32, f32, vp, vp, vp, vp, f32, vp, vp,
                                  vp, vp, sz, vp]
    L.pg_lookup_project_gate.restype = ctypes.c_int
    L.pg_lookup_project_gate.argtypes = [dp, vp, i32, i32, vp, vp, u64, i32, i32, vp, i32, f32, vp, vp, vp, vp,
                                         f32, vp, vp, vp, sz, vp, vp]
    L.pg_gather_project_gate.restype = ctypes.c_int
    L.pg_gather_project_gate.argtypes = [dp, vp, i32, i32, vp, vp, u64, vp, i32, i32, vp, i32, f32, vp, vp, vp,
                                         vp, f32, vp, vp, vp, vp, sz, vp, vp]
    L.pg_gather_project_gate_workspace_size.restype = ctypes.c_int
    L.pg_gather_project_gate_workspace_size.argtypes = [i32, i32, i32, i32, ctypes.POINTER(sz)]
    L.pg_gather_sign_concat_e4m3.restype = ctypes.c_int
    L.pg_gather_sign_concat_e4m3.argtypes = [dp, vp, i32, i32, vp, vp, u64, vp, vp, vp, vp]
    L.pg_project_gate_conv_workspace_size.restype = ctypes.c_int
    L.pg_project_gate_conv_workspace_size.argtypes = [i32, i32, i32, ctypes.POINTER(sz)]
    L.pg_project_gate_conv.restype = ctypes.c_int
    L.pg_project_gate_conv.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, i32, i32, f32, vp, vp, vp,
                                       vp, sz, vp]
    L.pg_fp8_quantize.restype = ctypes.c_int
    L.pg_fp8_quantize.argtypes = [vp, i32, ctypes.c_int64, ctypes.c_int64, vp, vp, vp]
    L.pg_project_gate_fp8.restype = ctypes.c_int
    L.pg_project_gate_fp8.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, i32, f32, vp, vp, vp, vp, f32, vp, vp,
                                      vp, vp, sz, vp]
    L.pg_nf4_quantize.restype = ctypes.c_int
    L.pg_nf4_quantize.argtypes = [vp, ctypes.c_int64, i32, vp, vp]
    L.pg_project_gate_context_noalloc.restype = ctypes.c_int
    L.pg_project_gate_context_noalloc.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, f32, vp, vp, vp]
    sp = ctypes.POINTER(DecodeStateC)
    L.pg_decode_state_size.restype = ctypes.c_int
    L.pg_decode_state_size.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(u64)]
    L.pg_decode_state_init.restype = ctypes.c_int
    L.pg_decode_state_init.argtypes = [sp, vp, u64, i32, i32, i32, i32, i32, i32, vp]
    L.pg_decode_reset.restype = ctypes.c_int
    L.pg_decode_reset.argtypes = [sp, vp, i32, vp]
    L.pg_decode_lookup.restype = ctypes.c_int
    L.pg_decode_lookup.argtypes = [dp, sp, vp, vp, vp, u64, vp, i32, vp, vp]
    L.pg_decode_conv_residual.restype = ctypes.c_int
    L.pg_decode_conv_residual.argtypes = [sp, vp, vp, vp, vp, vp, f32, vp, vp]
    L.pg_decode_step_workspace_size.restype = ctypes.c_int
    L.pg_decode_step_workspace_size.argtypes = [i32, i32, i32, ctypes.POINTER(u64)]
    L.pg_decode_step.restype = ctypes.c_int
    L.pg_decode_step.argtypes = [dp, sp, vp, vp, vp, u64, ctypes.POINTER(DecodeStepArgsC), vp, u64, vp, vp]
    L.pg_collision_counts_workspace_size.restype = ctypes.c_int
    L.pg_collision_counts_workspace_size.argtypes = [ctypes.c_int64, u32, ctypes.POINTER(sz)]
    L.pg_collision_counts.restype = ctypes.c_int
    L.pg_collision_counts.argtypes = [vp, ctypes.c_int64, i32, ctypes.c_int64, u32, u32, vp, vp, sz, vp]
    L.pg_conv_residual.restype = ctypes.c_int
    L.pg_conv_residual.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, i32, i32, f32, vp, vp]
    L.pg_selftest_bounded_waits.restype = ctypes.c_int
    L.pg_selftest_bounded_waits.argtypes = [vp, vp]
    L.pg_row_copy_window.restype = ctypes.c_int
    L.pg_row_copy_window.argtypes = [u32, ctypes.POINTER(u32)]
    L.pg_row_copy.restype = ctypes.c_int
    L.pg_row_copy.argtypes = [vp, u64, u32, vp, ctypes.c_int64, vp, u32, vp]
    return L


_lib = _load()


def lib():
    return _lib


def _check(status: int, where: str):
    if status != 0:
        raise PgError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def table_desc(spec, vocab: int, canon_vocab: Optional[int] = None) -> TableDesc:
    """Descriptor for a workloads.TableSpec (or any object with its fields)."""
    d = TableDesc()
    d.abi_version = PG_ABI_VERSION
    d.hash_version = PG_HASH_VERSION
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
    d.hash_seed = spec.hash_seed & 0xFFFFFFFFFFFFFFFF
    d.vocab = vocab
    d.canon_vocab = canon_vocab if canon_vocab is not None else vocab
    return d


def table_geometry(desc: TableDesc):
    rows, rb, ew = ctypes.c_uint64(), ctypes.c_uint32(), ctypes.c_uint32()
    _check(_lib.pg_table_geometry(ctypes.byref(desc), ctypes.byref(rows), ctypes.byref(rb), ctypes.byref(ew)),
           "pg_table_geometry")
    return rows.value, rb.value, ew.value


def canon_hash(desc: TableDesc, tokens: torch.Tensor, rows_out: torch.Tensor,
               canon_map: Optional[torch.Tensor] = None, canon_out: Optional[torch.Tensor] = None,
               sign_out: Optional[torch.Tensor] = None, err_index: Optional[torch.Tensor] = None,
               stream=None):
    B, L = tokens.shape
    _check(_lib.pg_canon_hash(ctypes.byref(desc), _ptr(tokens), B, L, _ptr(canon_map), _ptr(canon_out),
                              _ptr(rows_out), _ptr(sign_out), _ptr(err_index), _stream(stream)),
           "pg_canon_hash")


def gather_sign_concat(desc: TableDesc, tokens: torch.Tensor, table: torch.Tensor, e_out: torch.Tensor,
                       out_dtype: int, canon_map: Optional[torch.Tensor] = None,
                       err_index: Optional[torch.Tensor] = None, stream=None):
    B, L = tokens.shape
    nbytes = table.numel() * table.element_size()
    _check(_lib.pg_gather_sign_concat(ctypes.byref(desc), _ptr(tokens), B, L, _ptr(canon_map), _ptr(table),
                                      nbytes, _ptr(e_out), out_dtype, _ptr(err_index), _stream(stream)),
           "pg_gather_sign_concat")


def project_gate_conv_workspace_size(N: int, d: int, M: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.pg_project_gate_conv_workspace_size(N, d, M, ctypes.byref(n)), "pg_project_gate_conv_workspace_size")
    return n.value


def project_gate_conv(B: int, L: int, e: torch.Tensor, W: torch.Tensor, d: int, M: int, H: torch.Tensor,
                      gamma_h: torch.Tensor, gamma_k: torch.Tensor, gamma_c: torch.Tensor, conv_w: torch.Tensor,
                      v_out: torch.Tensor, alpha_out: torch.Tensor, workspace: torch.Tensor, dilation: int = 3,
                      eps: float = 1e-6, v_ms_out: Optional[torch.Tensor] = None, stream=None):
    """Context-gated projection + causal conv + residual in one launch; H [M, B*L, d] updated
    in place (it is also the gate's h)."""
    ks = conv_w.shape[1]
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.pg_project_gate_conv(B, L, e.shape[1], d, M, _ptr(e), _ptr(W), _ptr(H), _ptr(gamma_h), _ptr(gamma_k),
                                     _ptr(gamma_c), _ptr(conv_w), ks, dilation, eps, _ptr(v_out), _ptr(alpha_out),
                                     _ptr(v_ms_out), _ptr(workspace), ws_bytes, _stream(stream)),
           "pg_project_gate_conv")


def gather_sign_concat_e4m3(desc: TableDesc, tokens: torch.Tensor, table: torch.Tensor, q_out: torch.Tensor,
                            scale_out: torch.Tensor, canon_map: Optional[torch.Tensor] = None,
                            err_index: Optional[torch.Tensor] = None, stream=None):
    """q_out: uint8 [B*L, e_width] E4M3 codes; scale_out: fp32 [B*L]."""
    B, L = tokens.shape
    nbytes = table.numel() * table.element_size()
    _check(_lib.pg_gather_sign_concat_e4m3(ctypes.byref(desc), _ptr(tokens), B, L, _ptr(canon_map), _ptr(table),
                                           nbytes, _ptr(q_out), _ptr(scale_out), _ptr(err_index), _stream(stream)),
           "pg_gather_sign_concat_e4m3")


def workspace_size(N: int, Din: int, d: int, M: int, dtype: int, gate_kind: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.pg_project_gate_workspace_size(N, Din, d, M, dtype, gate_kind, ctypes.byref(n)),
           "pg_project_gate_workspace_size")
    return n.value


def project_gate(e: torch.Tensor, W: Optional[torch.Tensor], d: int, gate_kind: int, v_out: torch.Tensor,
                 dtype: int, M: int = 0, g: float = 0.0, x_resid: Optional[torch.Tensor] = None,
                 h: Optional[torch.Tensor] = None, gamma_h: Optional[torch.Tensor] = None,
                 gamma_k: Optional[torch.Tensor] = None, eps: float = 1e-6,
                 alpha_out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 v_ms_out: Optional[torch.Tensor] = None, stream=None):
    N, Din = e.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.pg_project_gate(N, Din, d, M, dtype, _ptr(e), _ptr(W), gate_kind, g, _ptr(x_resid), _ptr(h),
                                _ptr(gamma_h), _ptr(gamma_k), eps, _ptr(v_out), _ptr(alpha_out),
                                _ptr(v_ms_out), _ptr(workspace), ws_bytes, _stream(stream)),
           "pg_project_gate")


def lookup_project_gate(desc: TableDesc, tokens: torch.Tensor, table: torch.Tensor, W: torch.Tensor, d: int,
                        gate_kind: int, v_out: torch.Tensor, canon_map: Optional[torch.Tensor] = None, M: int = 0,
                        g: float = 0.0, x_resid: Optional[torch.Tensor] = None, h: Optional[torch.Tensor] = None,
                        gamma_h: Optional[torch.Tensor] = None, gamma_k: Optional[torch.Tensor] = None,
                        eps: float = 1e-6, alpha_out: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, err_index: Optional[torch.Tensor] = None,
                        stream=None):
    """gather_sign_concat + project_gate in one kernel (e_t never leaves shared memory)."""
    B, L = tokens.shape
    nbytes = table.numel() * table.element_size()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.pg_lookup_project_gate(ctypes.byref(desc), _ptr(tokens), B, L, _ptr(canon_map), _ptr(table),
                                       nbytes, d, M, _ptr(W), gate_kind, g, _ptr(x_resid), _ptr(h), _ptr(gamma_h),
                                       _ptr(gamma_k), eps, _ptr(v_out), _ptr(alpha_out), _ptr(workspace),
                                       ws_bytes, _ptr(err_index), _stream(stream)),
           "pg_lookup_project_gate")


def gather_project_workspace_size(N: int, d: int, M: int, gate_kind: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.pg_gather_project_gate_workspace_size(N, d, M, gate_kind, ctypes.byref(n)),
           "pg_gather_project_gate_workspace_size")
    return n.value


def gather_project_gate(desc: TableDesc, tokens: torch.Tensor, table: torch.Tensor, e_out: torch.Tensor,
                        W: torch.Tensor, d: int, gate_kind: int, v_out: torch.Tensor, workspace: torch.Tensor,
                        canon_map: Optional[torch.Tensor] = None, M: int = 0, g: float = 0.0,
                        x_resid: Optional[torch.Tensor] = None, h: Optional[torch.Tensor] = None,
                        gamma_h: Optional[torch.Tensor] = None, gamma_k: Optional[torch.Tensor] = None,
                        eps: float = 1e-6, alpha_out: Optional[torch.Tensor] = None,
                        v_ms_out: Optional[torch.Tensor] = None, err_index: Optional[torch.Tensor] = None,
                        stream=None):
    """gather_sign_concat (into e_out) + project_gate in one launch, the lookup overlapped
    with the tensor-core work."""
    B, L = tokens.shape
    nbytes = table.numel() * table.element_size()
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.pg_gather_project_gate(ctypes.byref(desc), _ptr(tokens), B, L, _ptr(canon_map), _ptr(table),
                                       nbytes, _ptr(e_out), d, M, _ptr(W), gate_kind, g, _ptr(x_resid), _ptr(h),
                                       _ptr(gamma_h), _ptr(gamma_k), eps, _ptr(v_out), _ptr(alpha_out),
                                       _ptr(v_ms_out), _ptr(workspace), ws_bytes, _ptr(err_index),
                                       _stream(stream)),
           "pg_gather_project_gate")


def fp8_quantize(x: torch.Tensor, q: torch.Tensor, scale: torch.Tensor, stream=None):
    """E4M3 rows with absmax/448 scales: x [rows, cols] fp32 or bf16 -> q uint8, scale fp32 [rows]."""
    rows, cols = x.shape
    _check(_lib.pg_fp8_quantize(_ptr(x), dtype_code(x.dtype), rows, cols, _ptr(q), _ptr(scale), _stream(stream)),
           "pg_fp8_quantize")


def project_gate_fp8(e_q: torch.Tensor, e_scale: torch.Tensor, W_q: torch.Tensor, W_scale: torch.Tensor, d: int,
                     gate_kind: int, v_out: torch.Tensor, M: int = 0, g: float = 0.0,
                     x_resid: Optional[torch.Tensor] = None, h: Optional[torch.Tensor] = None,
                     gamma_h: Optional[torch.Tensor] = None, gamma_k: Optional[torch.Tensor] = None,
                     eps: float = 1e-6, alpha_out: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, v_ms_out: Optional[torch.Tensor] = None,
                     stream=None):
    """project_gate on E4M3 operands (pg_fp8_quantize's output)."""
    N, Din = e_q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.pg_project_gate_fp8(N, Din, d, M, _ptr(e_q), _ptr(e_scale), _ptr(W_q), _ptr(W_scale), gate_kind, g,
                                    _ptr(x_resid), _ptr(h), _ptr(gamma_h), _ptr(gamma_k), eps, _ptr(v_out),
                                    _ptr(alpha_out), _ptr(v_ms_out), _ptr(workspace), ws_bytes, _stream(stream)),
           "pg_project_gate_fp8")


def nf4_quantize(x: torch.Tensor, out: torch.Tensor, stream=None):
    """NF4 export: x fp32 [n, 64] -> out uint8 [n, 34] (the PG_NF4 row layout)."""
    n, r = x.shape
    _check(_lib.pg_nf4_quantize(_ptr(x), n, r, _ptr(out), _stream(stream)), "pg_nf4_quantize")


def project_gate_context_noalloc(e: torch.Tensor, W: torch.Tensor, d: int, M: int, h: torch.Tensor,
                                 gamma_h: torch.Tensor, gamma_k: torch.Tensor, v_out: torch.Tensor,
                                 alpha_out: torch.Tensor, eps: float = 1e-6, stream=None):
    """Context-gate projection with the library's static scratch (no workspace, no
    allocation); for callers that cannot allocate device memory."""
    N, Din = e.shape
    _check(_lib.pg_project_gate_context_noalloc(N, Din, d, M, _ptr(e), _ptr(W), _ptr(h), _ptr(gamma_h),
                                                _ptr(gamma_k), eps, _ptr(v_out), _ptr(alpha_out),
                                                _stream(stream)),
           "pg_project_gate_context_noalloc")


def conv_residual(B: int, L: int, d: int, M: int, dtype: int, v: torch.Tensor, alpha: torch.Tensor,
                  gamma_c: torch.Tensor, conv_w: torch.Tensor, H: torch.Tensor, dilation: int = 3,
                  eps: float = 1e-6, v_ms: Optional[torch.Tensor] = None, stream=None):
    ks = conv_w.shape[1]
    _check(_lib.pg_conv_residual(B, L, d, M, dtype, _ptr(v), _ptr(alpha), _ptr(v_ms), _ptr(gamma_c), _ptr(conv_w),
                                 ks, dilation, eps, _ptr(H), _stream(stream)),
           "pg_conv_residual")


def decode_state_size(B: int, d: int = 0, M: int = 0, dtype: int = BF16, kernel_size: int = 4,
                      dilation: int = 3) -> int:
    n = ctypes.c_uint64()
    _check(_lib.pg_decode_state_size(B, d, M, dtype, kernel_size, dilation, ctypes.byref(n)),
           "pg_decode_state_size")
    return n.value


class DecodeState:
    """A decode state and the device buffer it lives in (pg_decode_state_init zeroes it:
    B empty sequences). `pos`, `ids`, `ring_v`, `ring_alpha` and `ring_ms` are views of the
    buffer's parts, for inspection and for restarting sequences by hand."""

    def __init__(self, B: int, d: int = 0, M: int = 0, dtype: int = BF16, kernel_size: int = 4,
                 dilation: int = 3, device=None, stream=None):
        nbytes = decode_state_size(B, d, M, dtype, kernel_size, dilation)
        self.buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=device or torch.device("cuda"))
        base = (-self.buf.data_ptr()) % 256
        self.mem = self.buf[base:base + nbytes]
        self.c = DecodeStateC()
        _check(_lib.pg_decode_state_init(ctypes.byref(self.c), _ptr(self.mem), nbytes, B, d, M, dtype, kernel_size,
                                         dilation, _stream(stream)), "pg_decode_state_init")

    def _part(self, ptr, count, dtype):
        if not ptr or count == 0:
            return None
        off = ptr - self.mem.data_ptr()
        nbytes = count * torch.empty(0, dtype=dtype).element_size()
        return self.mem[off:off + nbytes].view(dtype)

    @property
    def pos(self):
        return self._part(self.c.pos, self.c.B, torch.int32)

    @property
    def ids(self):
        return self._part(self.c.ids, self.c.B * 4, torch.int32).view(self.c.B, 4)

    @property
    def ring_v(self):
        t = self._part(self.c.ring_v, self.c.B * self.c.depth * self.c.d,
                       torch.float32 if self.c.dtype == F32 else torch.bfloat16)
        return None if t is None else t.view(self.c.B, self.c.depth, self.c.d)

    @property
    def ring_alpha(self):
        t = self._part(self.c.ring_alpha, self.c.B * self.c.depth * self.c.M, torch.float32)
        return None if t is None else t.view(self.c.B, self.c.depth, self.c.M)

    @property
    def ring_ms(self):
        t = self._part(self.c.ring_ms, self.c.B * self.c.depth, torch.float32)
        return None if t is None else t.view(self.c.B, self.c.depth)


def decode_reset(state: DecodeState, slots: torch.Tensor, stream=None):
    _check(_lib.pg_decode_reset(ctypes.byref(state.c), _ptr(slots), slots.numel(), _stream(stream)),
           "pg_decode_reset")


def decode_lookup(desc: TableDesc, state: DecodeState, tokens: torch.Tensor, table: torch.Tensor,
                  e_out: torch.Tensor, out_dtype: int, canon_map: Optional[torch.Tensor] = None,
                  err_index: Optional[torch.Tensor] = None, stream=None):
    nbytes = table.numel() * table.element_size()
    _check(_lib.pg_decode_lookup(ctypes.byref(desc), ctypes.byref(state.c), _ptr(tokens), _ptr(canon_map),
                                 _ptr(table), nbytes, _ptr(e_out), out_dtype, _ptr(err_index), _stream(stream)),
           "pg_decode_lookup")


def decode_conv_residual(state: DecodeState, v: torch.Tensor, alpha: torch.Tensor, gamma_c: torch.Tensor,
                         conv_w: torch.Tensor, H: torch.Tensor, eps: float = 1e-6,
                         v_ms: Optional[torch.Tensor] = None, stream=None):
    _check(_lib.pg_decode_conv_residual(ctypes.byref(state.c), _ptr(v), _ptr(alpha), _ptr(v_ms), _ptr(gamma_c),
                                        _ptr(conv_w), eps, _ptr(H), _stream(stream)),
           "pg_decode_conv_residual")



def decode_step_workspace_size(B: int, d: int, M: int = 0) -> int:
    b = ctypes.c_uint64()
    _check(_lib.pg_decode_step_workspace_size(B, d, M, ctypes.byref(b)), "pg_decode_step_workspace_size")
    return b.value


def decode_step(desc: TableDesc, state: DecodeState, tokens: torch.Tensor, table: torch.Tensor, W: torch.Tensor,
                d: int, gate_kind: int, out: torch.Tensor, workspace: torch.Tensor, canon_map: Optional[torch.Tensor] = None,
                g: float = 1.0, x_resid: Optional[torch.Tensor] = None, H: Optional[torch.Tensor] = None,
                gamma_h: Optional[torch.Tensor] = None, gamma_k: Optional[torch.Tensor] = None,
                gamma_c: Optional[torch.Tensor] = None, conv_w: Optional[torch.Tensor] = None, eps: float = 1e-6,
                e_out: Optional[torch.Tensor] = None, alpha_out: Optional[torch.Tensor] = None,
                v_ms_out: Optional[torch.Tensor] = None, err_index: Optional[torch.Tensor] = None, stream=None):
    """pg_decode_step: one decode step (lookup, projection, gate and, for the context gate,
    the conv) in one launch. `workspace` must be zero before its first use."""
    a = DecodeStepArgsC(_ptr(W), d, gate_kind, g, eps, _ptr(x_resid), _ptr(H), _ptr(gamma_h), _ptr(gamma_k),
                        _ptr(gamma_c), _ptr(conv_w), _ptr(e_out), _ptr(out), _ptr(alpha_out), _ptr(v_ms_out))
    nbytes = table.numel() * table.element_size()
    wbytes = workspace.numel() * workspace.element_size()
    _check(_lib.pg_decode_step(ctypes.byref(desc), ctypes.byref(state.c), _ptr(tokens), _ptr(canon_map), _ptr(table),
                               nbytes, ctypes.byref(a), _ptr(workspace), wbytes, _ptr(err_index), _stream(stream)),
           "pg_decode_step")

def collision_workspace_size(n: int, row0_span: int) -> int:
    b = ctypes.c_size_t()
    _check(_lib.pg_collision_counts_workspace_size(n, row0_span, ctypes.byref(b)),
           "pg_collision_counts_workspace_size")
    return b.value


def collision_counts(rows: torch.Tensor, n: int, K: int, stride: int, row0_lo: int, row0_span: int,
                     counts_out: torch.Tensor, workspace: torch.Tensor, stream=None):
    """rows: int32 view of the uint32 head rows (n-gram i, head k at i * stride + k);
    counts_out: int64 [K] (uint64 counts); workspace: >= collision_workspace_size bytes."""
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.pg_collision_counts(_ptr(rows), n, K, stride, row0_lo, row0_span, _ptr(counts_out),
                                    _ptr(workspace), ws_bytes, _stream(stream)), "pg_collision_counts")


def launch_count() -> int:
    return int(_lib.pg_launch_count())


def device_error(clear: bool = False) -> int:
    code = ctypes.c_int32()
    _check(_lib.pg_device_error(ctypes.byref(code), 1 if clear else 0), "pg_device_error")
    return code.value


def selftest_bounded_waits(zero_word: torch.Tensor, stream=None):
    """zero_word: a 4-byte device tensor (set to 0 by the call). Afterwards (about 2 s on
    the device) the device error word holds 2048 | 4096 when both waits gave up as they
    should."""
    _check(_lib.pg_selftest_bounded_waits(_ptr(zero_word), _stream(stream)), "pg_selftest_bounded_waits")


def row_copy_window(row_bytes: int) -> int:
    w = ctypes.c_uint32()
    _check(_lib.pg_row_copy_window(row_bytes, ctypes.byref(w)), "pg_row_copy_window")
    return w.value


def row_copy(table: torch.Tensor, row_bytes: int, rows: torch.Tensor, out: torch.Tensor, out_row_bytes: int = 0,
             stream=None):
    """Diagnostic: out [n, out_row_bytes or row_copy_window(row_bytes)] bytes = the windows of
    the table rows `rows` (int32 view of uint32 indices, n = rows.numel()), zero-padded."""
    nbytes = table.numel() * table.element_size()
    _check(_lib.pg_row_copy(_ptr(table), nbytes, row_bytes, _ptr(rows), rows.numel(), _ptr(out), out_row_bytes,
                            _stream(stream)), "pg_row_copy")


def dtype_code(t: torch.dtype) -> int:
    return {torch.float32: F32, torch.bfloat16: BF16}[t]


__all__ = ["PgError", "TableDesc", "table_desc", "table_geometry", "canon_hash", "gather_sign_concat",
           "gather_sign_concat_e4m3", "project_gate_conv", "project_gate_conv_workspace_size",
           "workspace_size", "project_gate", "lookup_project_gate", "gather_project_workspace_size",
           "gather_project_gate", "nf4_quantize", "fp8_quantize", "project_gate_fp8", "project_gate_context_noalloc", "conv_residual",
           "decode_state_size", "DecodeState", "decode_reset", "decode_lookup", "decode_conv_residual",
           "collision_workspace_size", "collision_counts", "launch_count", "device_error", "selftest_bounded_waits",
           "row_copy_window", "row_copy", "lib",
           "FLAT", "ENGRAM", "PAGEGRAM", "F32", "BF16", "NF4", "GATE_NONE", "GATE_SCALAR", "GATE_CONTEXT",
           "HASH_MULXOR", "HASH_TOY", "PG_NO_ROW"]
