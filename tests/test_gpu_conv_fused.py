"""pg_project_gate_conv: the context-gated projection and the causal conv + residual in one
launch (Engram notes 3.3, 3.4, 3.1). Its v, alpha, mean(v^2) and updated H must equal
pg_project_gate followed by pg_conv_residual bit for bit (same arithmetic, one launch), and
the fp64 oracle within the bf16 tolerance."""
import numpy as np
import pytest
import torch

from oracle import dense
from tests._helpers import BF16_TOL, rel_l2, to_f64

pytestmark = pytest.mark.gpu


def _pg():
    from hashed_head_gram_gb300 import pg
    return pg


def _case(B, L, Din, d, M, ks, seed, zero_e=False):
    g = torch.Generator().manual_seed(seed)
    N = B * L
    e = (torch.randint(-128, 128, (N, Din), generator=g).float() / 64).to(torch.bfloat16)
    if zero_e:
        e.zero_()
    W = (torch.randn((1 + M) * d, Din, generator=g) * 0.02).to(torch.bfloat16)
    H = torch.randn(M, N, d, generator=g).to(torch.bfloat16)
    gh = torch.rand(d, generator=g) + 0.5
    gk = torch.rand(d, generator=g) + 0.5
    gc = torch.rand(d, generator=g) + 0.5
    cw = torch.randn(d, ks, generator=g) * 0.25
    return e, W, H, gh, gk, gc, cw


def _two_calls(pg, cuda, B, L, d, M, e, W, H, gh, gk, gc, cw, dil):
    N = B * L
    v = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    a = torch.empty(M, N, device=cuda)
    ms = torch.empty(N, device=cuda)
    ws = torch.empty(pg.workspace_size(N, e.shape[1], d, M, pg.BF16, pg.GATE_CONTEXT) // 4 + 4, device=cuda)
    Hd = H.to(cuda)
    pg.project_gate(e.to(cuda), W.to(cuda), d, pg.GATE_CONTEXT, v, pg.BF16, M=M, h=Hd, gamma_h=gh.to(cuda),
                    gamma_k=gk.to(cuda), eps=1e-6, alpha_out=a, workspace=ws, v_ms_out=ms)
    pg.conv_residual(B, L, d, M, pg.BF16, v, a, gc.to(cuda), cw.to(cuda), Hd, dilation=dil, eps=1e-6, v_ms=ms)
    return v, a, ms, Hd


def _fused(pg, cuda, B, L, d, M, e, W, H, gh, gk, gc, cw, dil, with_ms=True):
    N = B * L
    v = torch.full((N, d), float("nan"), dtype=torch.bfloat16, device=cuda)
    a = torch.full((M, N), float("nan"), device=cuda)
    ms = torch.full((N,), float("nan"), device=cuda) if with_ms else None
    ws = torch.full((pg.project_gate_conv_workspace_size(N, d, M) // 4 + 4,), 7.0, device=cuda)   # dirty
    Hd = H.to(cuda)
    pg.project_gate_conv(B, L, e.to(cuda), W.to(cuda), d, M, Hd, gh.to(cuda), gk.to(cuda), gc.to(cuda), cw.to(cuda),
                         v, a, ws, dilation=dil, eps=1e-6, v_ms_out=ms)
    return v, a, ms, Hd


# ragged m-blocks (N % 256 != 0, a CTA with no rows), sequences shorter than an m-block,
# several kernel sizes and dilations (halo 0 .. 24), the Engram-27B module's widths
CASES = [(2, 300, 256, 512, 2, 4, 3), (1, 1000, 128, 256, 1, 4, 3), (3, 517, 192, 768, 3, 3, 2),
         (4, 64, 256, 256, 4, 4, 3), (2, 200, 64, 256, 2, 1, 1), (1, 700, 128, 512, 2, 4, 8),
         (2, 1024, 1280, 2560, 4, 4, 3)]


@pytest.mark.parametrize("B,L,Din,d,M,ks,dil", CASES)
def test_fused_equals_the_two_calls_bit_for_bit(cuda, B, L, Din, d, M, ks, dil):
    pg = _pg()
    pg.device_error(clear=True)
    args = _case(B, L, Din, d, M, ks, 40 + d + ks)
    ref = _two_calls(pg, cuda, B, L, d, M, *args, dil)
    got = _fused(pg, cuda, B, L, d, M, *args, dil)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    for r, o, name in zip(ref, got, ["v", "alpha", "v_ms", "H"]):
        view = torch.int16 if r.dtype == torch.bfloat16 else torch.int32
        assert torch.equal(r.view(view), o.view(view)), name


def test_fused_matches_the_oracle(cuda):
    pg = _pg()
    B, L, Din, d, M, ks, dil = 2, 384, 256, 512, 2, 4, 3
    e, W, H, gh, gk, gc, cw = _case(B, L, Din, d, M, ks, 77)
    v, a, ms, Hn = _fused(pg, cuda, B, L, d, M, e, W, H, gh, gk, gc, cw, dil)
    torch.cuda.synchronize()
    N = B * L
    v_ref, a_ref = dense.engram_gate(e.double().numpy(), W.double().numpy(), H.double().numpy(), gh.double().numpy(),
                                     gk.double().numpy(), 1e-6, M)
    assert rel_l2(to_f64(v), v_ref) <= BF16_TOL
    assert rel_l2(to_f64(a), a_ref) <= BF16_TOL
    H_ref = dense.conv_residual(to_f64(v).reshape(B, L, d), to_f64(a).reshape(M, B, L), gc.double().numpy(),
                                cw.double().numpy(), dil, 1e-6, H.double().numpy().reshape(M, B, L, d))
    assert rel_l2(to_f64(Hn).reshape(M, B, L, d), H_ref) <= BF16_TOL
    assert np.allclose(to_f64(ms), (to_f64(v) ** 2).mean(axis=1), rtol=1e-5, atol=1e-7)


def test_fused_zero_table_leaves_H_unchanged(cuda):
    # e = 0 -> v = 0, alpha = 1/2 exactly, Y = 0: H bit-identical (PageGram report 9.4 check 3)
    pg = _pg()
    B, L, Din, d, M, ks, dil = 2, 300, 128, 256, 2, 4, 3
    e, W, H, gh, gk, gc, cw = _case(B, L, Din, d, M, ks, 78, zero_e=True)
    v, a, ms, Hn = _fused(pg, cuda, B, L, d, M, e, W, H, gh, gk, gc, cw, dil, with_ms=False)
    torch.cuda.synchronize()
    assert (to_f64(v) == 0).all() and (a.cpu() == 0.5).all()
    assert torch.equal(Hn.cpu().view(torch.int16), H.view(torch.int16))


def test_fused_rejections(cuda):
    pg = _pg()
    B, L, Din, d, M, ks = 1, 300, 128, 384, 2, 4          # d % 256 != 0
    e, W, H, gh, gk, gc, cw = _case(B, L, Din, d, M, ks, 79)
    with pytest.raises(pg.PgError, match="UNSUPPORTED"):
        _fused(pg, cuda, B, L, d, M, e, W, H, gh, gk, gc, cw, 3)
    d = 256
    e, W, H, gh, gk, gc, cw = _case(B, L, Din, d, M, ks, 80)
    small = torch.empty(16, device=cuda)
    with pytest.raises(pg.PgError, match="WORKSPACE"):
        pg.project_gate_conv(B, L, e.to(cuda), W.to(cuda), d, M, H.to(cuda), gh.to(cuda), gk.to(cuda), gc.to(cuda),
                             cw.to(cuda), torch.empty(300, d, dtype=torch.bfloat16, device=cuda),
                             torch.empty(M, 300, device=cuda), small)
    with pytest.raises(pg.PgError, match="SHAPE"):   # halo 3 * 9 > 24 (dilation out of range)
        _fused(pg, cuda, B, L, d, M, e, W, H, gh, gk, gc, cw, 9)
