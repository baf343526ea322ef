"""GPU parity of pg_project_gate (SIMT fp32 and tcgen05 bf16 paths) and
pg_conv_residual against the fp64 oracle, within the stated rel-L2 tolerances."""
import numpy as np
import pytest
import torch

from hashed_head_gram_gb300 import workloads as W
from oracle import dense
from tests._helpers import BF16_TOL, F32_TOL, rel_l2, to_f64

pytestmark = pytest.mark.gpu


def _pg():
    from hashed_head_gram_gb300 import pg
    return pg


def _gen(seed):
    return torch.Generator().manual_seed(seed)


def _e_bf16(N, Din, seed):
    # e_t-like values: int8/64 with random signs (exact in bf16)
    return (torch.randint(-128, 128, (N, Din), generator=_gen(seed)).float() / 64).to(torch.bfloat16)


def test_simt_fp32_projection_config1(cuda):
    pg = _pg()
    N, Din, d = 4096, 1024, 256                   # the tiny workload's full size
    e = torch.randint(-128, 128, (N, Din), generator=_gen(1)).float() / 64
    Wv = torch.randn(d, Din, generator=_gen(2)) * 0.02
    v = torch.empty(N, d, device=cuda)
    pg.project_gate(e.to(cuda), Wv.to(cuda), d, pg.GATE_NONE, v, pg.F32)
    ref = dense.project(e.double().numpy(), Wv.double().numpy())
    assert rel_l2(to_f64(v), ref) <= F32_TOL
    x = torch.randn(N, d, generator=_gen(3))
    out = torch.empty(N, d, device=cuda)
    pg.project_gate(e.to(cuda), Wv.to(cuda), d, pg.GATE_SCALAR, out, pg.F32, g=0.5, x_resid=x.to(cuda))
    assert rel_l2(to_f64(out), dense.scalar_gate(x.double().numpy(), ref, 0.5)) <= F32_TOL


# fp32 SIMT shapes: split K over clusters of 4 and 2 CTAs and none, K not a multiple of the
# 32-deep k-tile, ragged rows and columns; Din % 4 != 0 and a W offset by 4 bytes take the
# kernel with 4-byte loads.
@pytest.mark.parametrize("N,Din,d,shift", [(1000, 1280, 256, 0), (77, 192, 384, 0), (65, 100, 72, 0),
                                           (640, 64, 64, 0), (33, 99, 40, 0), (300, 512, 128, 1)])
def test_simt_fp32_projection_shapes(cuda, N, Din, d, shift):
    pg = _pg()
    e = torch.randint(-128, 128, (N, Din), generator=_gen(6)).float() / 64
    Wv = torch.randn(d, Din, generator=_gen(7)) * 0.02
    x = torch.randn(N, d, generator=_gen(8))
    ref = dense.project(e.double().numpy(), Wv.double().numpy())
    buf = torch.empty(d * Din + shift, device=cuda)
    wd = buf[shift:].view(d, Din)
    wd.copy_(Wv.to(cuda))
    for gate in (pg.GATE_NONE, pg.GATE_SCALAR):
        out = torch.empty(N, d, device=cuda)
        pg.project_gate(e.to(cuda), wd, d, gate, out, pg.F32, g=0.5, x_resid=x.to(cuda))
        want = ref if gate == pg.GATE_NONE else dense.scalar_gate(x.double().numpy(), ref, 0.5)
        assert rel_l2(to_f64(out), want) <= F32_TOL, gate


# d % 256 == 0 runs 256 x 256 tiles on CTA pairs: N = 429 and 1000 end in a ragged second
# half, N = 640 in a pair whose second CTA has no rows at all; d = 128 / 384 run single CTAs.
@pytest.mark.parametrize("N,Din,d", [(429, 1024, 768), (128, 64, 128), (1000, 1280, 256), (77, 192, 384),
                                     (640, 512, 512)])
def test_tcgen05_projection(cuda, N, Din, d):
    pg = _pg()
    e = _e_bf16(N, Din, 4)
    Wv = (torch.randn(d, Din, generator=_gen(5)) * 0.02).to(torch.bfloat16)
    v = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    pg.project_gate(e.to(cuda), Wv.to(cuda), d, pg.GATE_NONE, v, pg.BF16)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    ref = dense.project(e.double().numpy(), Wv.double().numpy())
    err = rel_l2(to_f64(v), ref)
    assert err <= BF16_TOL
    assert err <= 4e-3        # bf16 output rounding dominates; fp32 accumulation
    x = torch.randn(N, d, generator=_gen(6)).to(torch.bfloat16)
    out = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    pg.project_gate(e.to(cuda), Wv.to(cuda), d, pg.GATE_SCALAR, out, pg.BF16, g=0.5, x_resid=x.to(cuda))
    torch.cuda.synchronize()
    assert rel_l2(to_f64(out), dense.scalar_gate(x.double().numpy(), ref, 0.5)) <= BF16_TOL


@pytest.mark.parametrize("N,Din,d,M", [(300, 1280, 2560, 4), (129, 128, 256, 2), (64, 64, 384, 1),
                                       (384, 256, 512, 2)])
def test_tcgen05_context_gate(cuda, N, Din, d, M):
    pg = _pg()
    e = _e_bf16(N, Din, 7)
    Wm = (torch.randn((1 + M) * d, Din, generator=_gen(8)) * 0.02).to(torch.bfloat16)
    h = torch.randn(M, N, d, generator=_gen(9)).to(torch.bfloat16)
    gh = torch.rand(d, generator=_gen(10)) + 0.5
    gk = torch.rand(d, generator=_gen(11)) + 0.5
    v = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    alpha = torch.empty(M, N, device=cuda)
    v_ms = torch.empty(N, device=cuda)
    ws = torch.empty(pg.workspace_size(N, Din, d, M, pg.BF16, pg.GATE_CONTEXT) // 4, device=cuda)
    pg.project_gate(e.to(cuda), Wm.to(cuda), d, pg.GATE_CONTEXT, v, pg.BF16, M=M, h=h.to(cuda),
                    gamma_h=gh.to(cuda), gamma_k=gk.to(cuda), eps=1e-6, alpha_out=alpha, workspace=ws,
                    v_ms_out=v_ms)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    v_ref, a_ref = dense.engram_gate(e.double().numpy(), Wm.double().numpy(), h.double().numpy(),
                                     gh.double().numpy(), gk.double().numpy(), 1e-6, M)
    assert rel_l2(to_f64(v), v_ref) <= BF16_TOL
    assert rel_l2(to_f64(alpha), a_ref) <= BF16_TOL
    assert np.abs(to_f64(alpha) - a_ref).max() < 1e-3
    # mean(v^2) of the stored (bf16) v: fp32 sums of exact squares, so ~1e-6 relative
    ms_stored = (to_f64(v) ** 2).mean(axis=1)
    assert np.abs(to_f64(v_ms) - ms_stored).max() <= 1e-5 * ms_stored.max()
    assert rel_l2(to_f64(v_ms), (v_ref ** 2).mean(axis=1)) <= BF16_TOL
    # the same call without v_ms_out needs no room for it
    need = M * (d // (256 if d % 256 == 0 else 128)) * 3 * N * 4
    alpha2 = torch.empty_like(alpha)
    pg.project_gate(e.to(cuda), Wm.to(cuda), d, pg.GATE_CONTEXT, v, pg.BF16, M=M, h=h.to(cuda),
                    gamma_h=gh.to(cuda), gamma_k=gk.to(cuda), eps=1e-6, alpha_out=alpha2,
                    workspace=ws[:need // 4])
    torch.cuda.synchronize()
    assert torch.equal(alpha, alpha2)


def test_context_gate_rejects_small_workspace(cuda):
    pg = _pg()
    N, Din, d, M = 64, 64, 256, 2
    e = torch.zeros(N, Din, dtype=torch.bfloat16, device=cuda)
    Wm = torch.zeros((1 + M) * d, Din, dtype=torch.bfloat16, device=cuda)
    h = torch.zeros(M, N, d, dtype=torch.bfloat16, device=cuda)
    g1 = torch.ones(d, device=cuda)
    need = pg.workspace_size(N, Din, d, M, pg.BF16, pg.GATE_CONTEXT)   # includes the v_ms_out room
    base = M * (d // 256) * 3 * N * 4
    assert need == base + (d // 256) * N * 4
    v = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    a = torch.empty(M, N, device=cuda)
    for nbytes, v_ms in ((base - 4, None), (need - 4, torch.empty(N, device=cuda))):
        with pytest.raises(pg.PgError) as ex:
            pg.project_gate(e, Wm, d, pg.GATE_CONTEXT, v, pg.BF16, M=M, h=h, gamma_h=g1, gamma_k=g1, alpha_out=a,
                            workspace=torch.empty(nbytes // 4, device=cuda), v_ms_out=v_ms)
        assert ex.value.status == 8


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_identity_projection_for_flat_tables(cuda, dtype):
    pg = _pg()
    N, d = 333, 768
    e = (torch.randint(-128, 128, (N, d), generator=_gen(12)).float() / 64).to(dtype)
    x = torch.randn(N, d, generator=_gen(13)).to(dtype)
    out = torch.empty(N, d, dtype=dtype, device=cuda)
    pg.project_gate(e.to(cuda), None, d, pg.GATE_SCALAR, out, pg.dtype_code(dtype), g=0.5, x_resid=x.to(cuda))
    ref = dense.scalar_gate(x.double().numpy(), e.double().numpy(), 0.5)
    assert rel_l2(to_f64(out), ref) <= (BF16_TOL if dtype == torch.bfloat16 else F32_TOL)


def _conv_case(B, L, d, M, seed, zero_w=False, dtype=torch.bfloat16):
    g = _gen(seed)
    v = torch.randn(B * L, d, generator=g).to(dtype)
    alpha = torch.rand(M, B * L, generator=g)
    gc = torch.rand(d, generator=g) + 0.5
    w = torch.zeros(d, 4) if zero_w else torch.randn(d, 4, generator=g) * 0.25
    H = torch.randn(M, B * L, d, generator=g).to(dtype)
    return v, alpha, gc, w, H


# d <= 3072 runs 4 channels per thread, larger d 8 (d = 8192: 1024 threads); M = 3 takes the
# runtime-branch-count kernel
@pytest.mark.parametrize("B,L,d,M,dtype", [(2, 75, 2560, 4, torch.bfloat16), (3, 16, 64, 2, torch.bfloat16),
                                           (1, 40, 256, 3, torch.float32), (2, 9, 512, 1, torch.bfloat16),
                                           (1, 37, 4608, 2, torch.bfloat16), (1, 20, 8192, 1, torch.float32)])
@pytest.mark.parametrize("given_ms", [False, True])
def test_conv_residual(cuda, B, L, d, M, dtype, given_ms):
    pg = _pg()
    v, alpha, gc, w, H = _conv_case(B, L, d, M, 14, dtype=dtype)
    Hd = H.to(cuda)
    # given_ms: mean(v^2) supplied (as pg_project_gate's v_ms_out would), else computed inside
    v_ms = (v.double() ** 2).mean(dim=1).float().to(cuda) if given_ms else None
    pg.conv_residual(B, L, d, M, pg.dtype_code(dtype), v.to(cuda), alpha.to(cuda), gc.to(cuda), w.to(cuda), Hd,
                     dilation=3, eps=1e-6, v_ms=v_ms)
    ref = dense.conv_residual(v.double().numpy().reshape(B, L, d), alpha.double().numpy().reshape(M, B, L),
                              gc.double().numpy(), w.double().numpy(), 3, 1e-6,
                              H.double().numpy().reshape(M, B, L, d))
    tol = BF16_TOL if dtype == torch.bfloat16 else F32_TOL
    assert rel_l2(to_f64(Hd).reshape(M, B, L, d), ref) <= tol
    # the update itself (H_new - H) is also close: a stricter view of the same output
    upd = to_f64(Hd).reshape(M, B, L, d) - H.double().numpy().reshape(M, B, L, d)
    assert rel_l2(upd, ref - H.double().numpy().reshape(M, B, L, d)) <= (5e-2 if dtype == torch.bfloat16 else F32_TOL)


# sequences of several 32-position runs with a ragged tail, every kernel size and a spread of
# dilations: the causal window crosses run boundaries (up to 3 * 8 = 24 positions back),
# M = 8 and M = 3 take the runtime-branch-count kernel
@pytest.mark.parametrize("ks,dil,B,L,d,M,dtype", [
    (4, 8, 2, 100, 512, 2, torch.bfloat16),
    (4, 8, 1, 70, 256, 8, torch.float32),
    (1, 1, 2, 65, 512, 4, torch.bfloat16),
    (2, 1, 1, 97, 2560, 4, torch.bfloat16),
    (3, 2, 3, 33, 128, 3, torch.bfloat16),
    (2, 5, 2, 64, 768, 1, torch.float32),
    (3, 7, 1, 150, 1024, 4, torch.bfloat16),
])
@pytest.mark.parametrize("given_ms", [False, True])
def test_conv_residual_kernel_sizes_and_dilations(cuda, ks, dil, B, L, d, M, dtype, given_ms):
    pg = _pg()
    v, alpha, gc, w, H = _conv_case(B, L, d, M, 40 + ks * 10 + dil, dtype=dtype)
    w = w[:, :ks].contiguous()
    Hd = H.to(cuda)
    v_ms = (v.double() ** 2).mean(dim=1).float().to(cuda) if given_ms else None
    pg.conv_residual(B, L, d, M, pg.dtype_code(dtype), v.to(cuda), alpha.to(cuda), gc.to(cuda), w.to(cuda), Hd,
                     dilation=dil, eps=1e-6, v_ms=v_ms)
    ref = dense.conv_residual(v.double().numpy().reshape(B, L, d), alpha.double().numpy().reshape(M, B, L),
                              gc.double().numpy(), w.double().numpy(), dil, 1e-6,
                              H.double().numpy().reshape(M, B, L, d))
    assert rel_l2(to_f64(Hd).reshape(M, B, L, d), ref) <= (BF16_TOL if dtype == torch.bfloat16 else F32_TOL)
    # the first positions of every sequence see only the taps that reach back into it
    upd = to_f64(Hd).reshape(M, B, L, d) - H.double().numpy().reshape(M, B, L, d)
    ref_upd = ref - H.double().numpy().reshape(M, B, L, d)
    head = min(L, (ks - 1) * dil + 1)
    assert rel_l2(upd[:, :, :head], ref_upd[:, :, :head]) <= (5e-2 if dtype == torch.bfloat16 else F32_TOL)


def test_zero_table_leaves_H_bit_identical(cuda):
    # e = 0 -> v = 0, alpha = 1/2 exactly, Y = 0: H is unchanged bit for bit
    # (PageGram report appendix D/E check 3).
    pg = _pg()
    N, Din, d, M, B, L = 96, 128, 256, 2, 2, 48
    e = torch.zeros(N, Din, dtype=torch.bfloat16, device=cuda)
    Wm = (torch.randn((1 + M) * d, Din, generator=_gen(15)) * 0.02).to(torch.bfloat16).to(cuda)
    H = torch.randn(M, N, d, generator=_gen(16)).to(torch.bfloat16).to(cuda)
    H0 = H.clone()
    g1 = torch.ones(d, device=cuda)
    v = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    alpha = torch.empty(M, N, device=cuda)
    ws = torch.empty(pg.workspace_size(N, Din, d, M, pg.BF16, pg.GATE_CONTEXT) // 4, device=cuda)
    pg.project_gate(e, Wm, d, pg.GATE_CONTEXT, v, pg.BF16, M=M, h=H, gamma_h=g1, gamma_k=g1, alpha_out=alpha,
                    workspace=ws)
    pg.conv_residual(B, L, d, M, pg.BF16, v, alpha, g1, torch.randn(d, 4, device=cuda), H)
    torch.cuda.synchronize()
    assert (v.float() == 0).all() and (alpha == 0.5).all()
    assert torch.equal(H.view(torch.int16), H0.view(torch.int16))


def test_zero_conv_is_the_identity_path(cuda):
    pg = _pg()
    B, L, d, M = 2, 30, 128, 2
    v, alpha, gc, w, H = _conv_case(B, L, d, M, 17, zero_w=True, dtype=torch.float32)
    Hd = torch.zeros_like(H).to(cuda)
    pg.conv_residual(B, L, d, M, pg.F32, v.to(cuda), alpha.to(cuda), gc.to(cuda), w.to(cuda), Hd)
    ref = alpha.double().numpy()[..., None] * v.double().numpy()[None]
    assert np.array_equal(to_f64(Hd), (alpha[..., None] * v[None]).double().numpy())  # fp32 u = alpha * v
    assert rel_l2(to_f64(Hd), ref) <= 1e-7


# ------------------------------------------------------------------ few rows (decode batches)

@pytest.mark.parametrize("N", [1, 2, 3, 5, 8, 13, 16])
@pytest.mark.parametrize("Din,d", [(1024, 768), (1280, 2560), (256, 128)])
def test_few_rows_scalar_and_none_gates(cuda, N, Din, d):
    # up to 4 rows take the W-streaming SIMT kernel, more the tensor-core path: both sides
    pg = _pg()
    e = _e_bf16(N, Din, 90 + N)
    Wm = (torch.randn(d, Din, generator=_gen(91)) * 0.02).to(torch.bfloat16)
    x = torch.randn(N, d, generator=_gen(92)).to(torch.bfloat16)
    ref = dense.project(e.double().numpy(), Wm.double().numpy())
    v = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    pg.project_gate(e.to(cuda), Wm.to(cuda), d, pg.GATE_NONE, v, pg.BF16)
    out = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    pg.project_gate(e.to(cuda), Wm.to(cuda), d, pg.GATE_SCALAR, out, pg.BF16, g=0.5, x_resid=x.to(cuda))
    torch.cuda.synchronize()
    assert rel_l2(to_f64(v), ref) <= BF16_TOL
    assert rel_l2(to_f64(out), dense.scalar_gate(x.double().numpy(), ref, 0.5)) <= BF16_TOL
    # each output is one fp32 dot product (error <= Din 2^-24 sum |e W|) rounded once to bf16
    # (relative error <= 2^-8)
    s_abs = dense.project(np.abs(e.double().numpy()), np.abs(Wm.double().numpy()))
    bound = 2.0 ** -8 * np.abs(ref) + 1.01 * Din * 2.0 ** -24 * s_abs * (1 + 2.0 ** -8)
    assert np.all(np.abs(to_f64(v) - ref) <= bound)


@pytest.mark.parametrize("N", [1, 3, 8, 16])
@pytest.mark.parametrize("Din,d,M", [(1280, 2560, 4), (256, 256, 2), (512, 128, 1)])
def test_few_rows_context_gate(cuda, N, Din, d, M):
    pg = _pg()
    e = _e_bf16(N, Din, 95 + N)
    Wm = (torch.randn((1 + M) * d, Din, generator=_gen(96)) * 0.02).to(torch.bfloat16)
    h = torch.randn(M, N, d, generator=_gen(97)).to(torch.bfloat16)
    gh = torch.rand(d, generator=_gen(98)) + 0.5
    gk = torch.rand(d, generator=_gen(99)) + 0.5
    v = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    alpha = torch.empty(M, N, device=cuda)
    v_ms = torch.empty(N, device=cuda)
    ws = torch.empty(pg.workspace_size(N, Din, d, M, pg.BF16, pg.GATE_CONTEXT) // 4, device=cuda)
    pg.project_gate(e.to(cuda), Wm.to(cuda), d, pg.GATE_CONTEXT, v, pg.BF16, M=M, h=h.to(cuda), gamma_h=gh.to(cuda),
                    gamma_k=gk.to(cuda), eps=1e-6, alpha_out=alpha, workspace=ws, v_ms_out=v_ms)
    torch.cuda.synchronize()
    assert pg.device_error() == 0
    v_ref, a_ref = dense.engram_gate(e.double().numpy(), Wm.double().numpy(), h.double().numpy(),
                                     gh.double().numpy(), gk.double().numpy(), 1e-6, M)
    assert rel_l2(to_f64(v), v_ref) <= BF16_TOL
    assert np.abs(to_f64(alpha) - a_ref).max() < 1e-3
    ms_stored = (to_f64(v) ** 2).mean(axis=1)
    assert np.abs(to_f64(v_ms) - ms_stored).max() <= 1e-5 * ms_stored.max()
    # a workspace of the 256-column size sends the call to the tensor-core path: same values
    # within the tolerance (other accumulation order)
    small_ws = torch.empty(M * (d // (256 if d % 256 == 0 else 128)) * 3 * N + 4, device=cuda)
    v2 = torch.empty_like(v)
    alpha2 = torch.empty_like(alpha)
    pg.project_gate(e.to(cuda), Wm.to(cuda), d, pg.GATE_CONTEXT, v2, pg.BF16, M=M, h=h.to(cuda), gamma_h=gh.to(cuda),
                    gamma_k=gk.to(cuda), eps=1e-6, alpha_out=alpha2, workspace=small_ws)
    torch.cuda.synchronize()
    assert rel_l2(to_f64(v2), v_ref) <= BF16_TOL
    assert np.abs(to_f64(alpha2) - a_ref).max() < 1e-3

