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
