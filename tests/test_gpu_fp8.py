"""FP8 projection (Engram notes 3.4; reading R16): pg_fp8_quantize's codes and scales are
bit-identical to the oracle's, and pg_project_gate_fp8 matches the fp64 oracle computed on
the same E4M3 operands (products exact, fp32 sums, bf16 output) for every gate."""
import numpy as np
import pytest
import torch

from oracle import dense
from oracle import oracle as orc
from tests._helpers import BF16_TOL, rel_l2, to_f64

pytestmark = pytest.mark.gpu

FP8_OPERAND_TOL = 4e-3   # the bf16 rounding of the output (~1e-3 rel-L2) plus fp32 sums


def _pg():
    from hashed_head_gram_gb300 import pg
    return pg


def _gen(seed):
    return torch.Generator().manual_seed(seed)


def _quantize_gpu(pg, x, cuda):
    q = torch.empty(x.shape, dtype=torch.uint8, device=cuda)
    s = torch.empty(x.shape[0], device=cuda)
    pg.fp8_quantize(x.to(cuda), q, s)
    torch.cuda.synchronize()
    return q, s


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,cols", [(1, 8), (37, 1280), (1000, 1024), (3, 12800)])
def test_quantize_matches_the_oracle_bit_for_bit(cuda, dtype, rows, cols):
    pg = _pg()
    g = _gen(rows + cols)
    x = torch.randn(rows, cols, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 4)
    x[0, : cols // 2] = 0
    if rows > 2:
        x[1] = 0                                       # a zero row: scale 0, zero codes
        x[2] *= 1e-35                                  # scales far below E4M3's subnormals
    x = x.to(dtype)
    q, s = _quantize_gpu(pg, x, cuda)
    q_ref, s_ref = orc.fp8_quantize(x.float().numpy())
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


def _operands(pg, cuda, N, Din, Dcols, seed):
    e = (torch.randint(-128, 128, (N, Din), generator=_gen(seed)).float() / 64).to(torch.bfloat16)
    Wm = (torch.randn(Dcols, Din, generator=_gen(seed + 1)) * 0.02).to(torch.bfloat16)
    qe, se = _quantize_gpu(pg, e, cuda)
    qw, sw = _quantize_gpu(pg, Wm, cuda)
    qe_ref, se_ref = orc.fp8_quantize(e.float().numpy())
    qw_ref, sw_ref = orc.fp8_quantize(Wm.float().numpy())
    assert np.array_equal(qe.cpu().numpy(), qe_ref) and np.array_equal(qw.cpu().numpy(), qw_ref)
    return e, Wm, (qe, se, qw, sw), (orc.fp8_dequantize(qe_ref, se_ref), orc.fp8_dequantize(qw_ref, sw_ref))


# N = 429 and 1000 end in a ragged second half of a CTA pair; N = 640 has a pair whose
# second CTA holds no rows
@pytest.mark.parametrize("N,Din,d", [(429, 1024, 768), (1000, 1280, 256), (640, 256, 512)])
def test_fp8_projection_scalar_and_none_gates(cuda, N, Din, d):
    pg = _pg()
    e, Wm, (qe, se, qw, sw), (de, dw) = _operands(pg, cuda, N, Din, d, 40)
    ref = dense.project(de, dw)
    v = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    pg.project_gate_fp8(qe, se, qw, sw, d, pg.GATE_NONE, v)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    assert rel_l2(to_f64(v), ref) <= FP8_OPERAND_TOL
    x = torch.randn(N, d, generator=_gen(42)).to(torch.bfloat16)
    out = torch.empty_like(v)
    pg.project_gate_fp8(qe, se, qw, sw, d, pg.GATE_SCALAR, out, g=0.5, x_resid=x.to(cuda))
    assert rel_l2(to_f64(out), dense.scalar_gate(x.double().numpy(), ref, 0.5)) <= FP8_OPERAND_TOL
    # what FP8 costs against the unquantised operands (E4M3's 3 mantissa bits)
    exact = dense.project(e.double().numpy(), Wm.double().numpy())
    assert rel_l2(to_f64(v), exact) <= 0.06


@pytest.mark.parametrize("N,Din,d,M", [(300, 1280, 2560, 4), (129, 256, 256, 2)])
def test_fp8_projection_context_gate(cuda, N, Din, d, M):
    pg = _pg()
    e, Wm, (qe, se, qw, sw), (de, dw) = _operands(pg, cuda, N, Din, (1 + M) * d, 50)
    h = torch.randn(M, N, d, generator=_gen(52)).to(torch.bfloat16)
    gh = torch.rand(d, generator=_gen(53)) + 0.5
    gk = torch.rand(d, generator=_gen(54)) + 0.5
    v = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    alpha = torch.empty(M, N, device=cuda)
    v_ms = torch.empty(N, device=cuda)
    ws = torch.empty(pg.workspace_size(N, Din, d, M, pg.BF16, pg.GATE_CONTEXT) // 4, device=cuda)
    pg.project_gate_fp8(qe, se, qw, sw, d, pg.GATE_CONTEXT, v, M=M, h=h.to(cuda), gamma_h=gh.to(cuda),
                        gamma_k=gk.to(cuda), eps=1e-6, alpha_out=alpha, workspace=ws, v_ms_out=v_ms)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    v_ref, a_ref = dense.engram_gate(de, dw, h.double().numpy(), gh.double().numpy(), gk.double().numpy(), 1e-6, M)
    assert rel_l2(to_f64(v), v_ref) <= FP8_OPERAND_TOL
    assert rel_l2(to_f64(alpha), a_ref) <= BF16_TOL
    assert np.abs(to_f64(alpha) - a_ref).max() < 1e-3
    ms_stored = (to_f64(v) ** 2).mean(axis=1)
    assert np.abs(to_f64(v_ms) - ms_stored).max() <= 1e-5 * ms_stored.max()


def test_fp8_rejects_what_it_does_not_cover(cuda):
    pg = _pg()
    q = torch.zeros(64, 192, dtype=torch.uint8, device=cuda)
    s = torch.ones(64, device=cuda)
    v = torch.empty(64, 256, dtype=torch.bfloat16, device=cuda)
    with pytest.raises(pg.PgError) as ex:                         # Din % 256 != 0
        pg.project_gate_fp8(q, s, torch.zeros(256, 192, dtype=torch.uint8, device=cuda), torch.ones(256, device=cuda),
                            256, pg.GATE_NONE, v)
    assert ex.value.status == 6
    with pytest.raises(pg.PgError) as ex:                         # cols % 8 != 0
        pg.fp8_quantize(torch.zeros(4, 12, device=cuda), torch.empty(4, 12, dtype=torch.uint8, device=cuda),
                        torch.empty(4, device=cuda))
    assert ex.value.status == 6


# ---- E4M3 e_t straight from the gather (pg_gather_sign_concat_e4m3)

def _e4m3_case(cfg, B, L, small=True):
    from tests._helpers import shrink_table
    from hashed_head_gram_gb300 import workloads as W
    w = W.shrink(W.make_workload(cfg), B=B, L=L)
    spec = shrink_table(w.tables[0]) if small else w.tables[0]
    return w, spec, W.make_tokens(w), W.make_canon_map(w)


@pytest.mark.parametrize("cfg,B,L", [(2, 3, 517), (3, 2, 301), (5, 3, 517), (5, 1, 1), (2, 1, 3)])
def test_gather_e4m3_matches_oracle_and_the_two_calls(cuda, cfg, B, L):
    from tests._helpers import canon_tensor, oracle_e
    from hashed_head_gram_gb300 import workloads as W
    pg = _pg()
    w, spec, tokens, cmap = _e4m3_case(cfg, B, L)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    table = W.make_table(w, spec, "cpu")
    N, D = w.N, spec.e_width
    # the oracle: e_t in bf16, then E4M3 codes and scales of each row
    e_ref = oracle_e(spec, tokens, cmap, w.vocab, table, orc.BF16)
    q_ref, s_ref = orc.fp8_quantize(orc.bf16_bits_to_f64(e_ref).astype(np.float32))
    tok = torch.from_numpy(tokens).to(cuda)
    cm = canon_tensor(cmap, cuda)
    td = table.to(cuda)
    q = torch.full((N, D), 0xA5, dtype=torch.uint8, device=cuda)
    s = torch.full((N,), float("nan"), device=cuda)
    err = torch.empty(1, dtype=torch.int32, device=cuda)
    pg.gather_sign_concat_e4m3(desc, tok, td, q, s, canon_map=cm, err_index=err)
    torch.cuda.synchronize()
    assert err.item() == -1 and pg.device_error() == 0
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    # and the same bytes as pg_gather_sign_concat (bf16) followed by pg_fp8_quantize
    e = torch.empty(N, D, dtype=torch.bfloat16, device=cuda)
    pg.gather_sign_concat(desc, tok, td, e, orc.BF16, canon_map=cm)
    q2, s2 = _quantize_gpu(pg, e, cuda)
    assert torch.equal(q, q2) and torch.equal(s.view(torch.int32), s2.view(torch.int32))


def test_gather_e4m3_zero_rows_and_rejections(cuda):
    from hashed_head_gram_gb300 import workloads as W
    pg = _pg()
    w, spec, tokens, cmap = _e4m3_case(5, 2, 40)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    table = torch.zeros(spec.table_rows, spec.r, dtype=torch.bfloat16)   # e_t = 0: scale 0, codes 0
    q = torch.full((w.N, spec.e_width), 7, dtype=torch.uint8, device=cuda)
    s = torch.full((w.N,), 1.0, device=cuda)
    pg.gather_sign_concat_e4m3(desc, torch.from_numpy(tokens).to(cuda), table.to(cuda), q, s,
                               canon_map=None if cmap is None else torch.from_numpy(cmap.view(np.int32)).to(cuda))
    torch.cuda.synchronize()
    assert int(q.max().item()) == 0 and float(s.abs().max().item()) == 0.0
    # NF4 rows and the tiny fp32 table are outside this entry point
    w4, spec4, tok4, _ = _e4m3_case(4, 1, 8)
    with pytest.raises(pg.PgError, match="DTYPE"):
        pg.gather_sign_concat_e4m3(pg.table_desc(spec4, w4.vocab, w4.canon_vocab), torch.from_numpy(tok4).to(cuda),
                                   torch.zeros(spec4.table_rows, 34, dtype=torch.uint8, device=cuda),
                                   torch.empty(8, spec4.e_width, dtype=torch.uint8, device=cuda),
                                   torch.empty(8, device=cuda))


@pytest.mark.parametrize("scale_exp", [-130, -120, -100, -90, -80, -60, 0, 60, 120])
def test_gather_e4m3_extreme_magnitudes(cuda, scale_exp):
    # rows of very different magnitudes, up to scales whose reciprocal leaves the normal
    # range (the kernel then divides plainly); codes and scales still equal the oracle's
    from tests._helpers import canon_tensor, oracle_e
    pg = _pg()
    w, spec, tokens, cmap = _e4m3_case(5, 2, 77)
    desc = pg.table_desc(spec, w.vocab, w.canon_vocab)
    g = _gen(900 + scale_exp)
    vals = torch.randn(spec.table_rows, spec.r, generator=g) * torch.exp(torch.randn(spec.table_rows, 1, generator=g))
    table = (vals * (2.0 ** scale_exp)).to(torch.bfloat16)
    e_ref = oracle_e(spec, tokens, cmap, w.vocab, table, orc.BF16)
    q_ref, s_ref = orc.fp8_quantize(orc.bf16_bits_to_f64(e_ref).astype(np.float32))
    q = torch.empty(w.N, spec.e_width, dtype=torch.uint8, device=cuda)
    s = torch.empty(w.N, device=cuda)
    pg.gather_sign_concat_e4m3(desc, torch.from_numpy(tokens).to(cuda), table.to(cuda), q, s,
                               canon_map=canon_tensor(cmap, cuda))
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)
