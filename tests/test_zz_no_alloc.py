"""pg_project_gate_context_noalloc: the context-gate projection for callers that
cannot allocate device memory (a runtime that owns all device memory through its
own pool, or a plug-in without an allocator). It must give what pg_project_gate
gives with a caller-provided workspace, call after call, and refuse requests larger
than its static scratch. This file is collected last on purpose."""
import ctypes

import pytest
import torch

from tests._helpers import BF16_TOL, rel_l2, to_f64

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _case(N, Din, d, M, seed, dev):
    g = torch.Generator().manual_seed(seed)
    e = (torch.randint(-128, 128, (N, Din), generator=g).float() / 64).to(torch.bfloat16)
    W = (torch.randn((1 + M) * d, Din, generator=g) * 0.02).to(torch.bfloat16)
    h = torch.randn(M, N, d, generator=g).to(torch.bfloat16)
    gh = torch.rand(d, generator=g) + 0.5
    gk = torch.rand(d, generator=g) + 0.5
    return [t.to(dev) for t in (e, W, h, gh, gk)]


def test_noalloc_matches_the_workspace_entry_point_on_consecutive_calls(cuda):
    from hashed_head_gram_gb300 import pg
    lib = pg.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # the larger call first: the later calls must not see its leftovers. N <= 4 runs the
    # few-rows kernel (64-column partial sums) through the same scratch.
    for N, Din, d, M, seed in [(700, 1280, 2560, 4, 21), (129, 256, 384, 2, 22), (1, 1280, 2560, 4, 23),
                               (4, 1280, 2560, 4, 24), (3, 256, 384, 2, 25)]:
        e, W, h, gh, gk = _case(N, Din, d, M, seed, cuda)
        v_ref = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
        a_ref = torch.empty(M, N, device=cuda)
        ws = torch.empty(pg.workspace_size(N, Din, d, M, pg.BF16, pg.GATE_CONTEXT) // 4, device=cuda)
        pg.project_gate(e, W, d, pg.GATE_CONTEXT, v_ref, pg.BF16, M=M, h=h, gamma_h=gh, gamma_k=gk, eps=1e-6,
                        alpha_out=a_ref, workspace=ws)
        v = torch.full((N, d), float("nan"), dtype=torch.bfloat16, device=cuda)
        a = torch.full((M, N), float("nan"), device=cuda)
        status = lib.pg_project_gate_context_noalloc(N, Din, d, M, _p(e), _p(W), _p(h), _p(gh), _p(gk), 1e-6,
                                                     _p(v), _p(a), stream)
        assert status == 0, pg.STATUS.get(status, status)
        torch.cuda.synchronize()
        assert pg.device_error() == 0
        assert rel_l2(to_f64(v), to_f64(v_ref)) <= BF16_TOL
        assert rel_l2(to_f64(a), to_f64(a_ref)) <= BF16_TOL
        # same kernels, deterministic reductions: identical results
        assert torch.equal(v.view(torch.int16), v_ref.view(torch.int16)) and torch.equal(a, a_ref)


def test_noalloc_refuses_requests_beyond_its_scratch(cuda):
    from hashed_head_gram_gb300 import pg
    lib = pg.lib()
    N, Din, d, M = 40000, 1280, 2560, 4          # needs 4 * 10 * 3 * 40000 * 4 B > 16 MiB
    e = torch.empty(N, Din, dtype=torch.bfloat16, device=cuda)
    W = torch.empty((1 + M) * d, Din, dtype=torch.bfloat16, device=cuda)
    h = torch.empty(M, N, d, dtype=torch.bfloat16, device=cuda)
    g1 = torch.ones(d, device=cuda)
    v = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    a = torch.empty(M, N, device=cuda)
    before = pg.launch_count()
    status = lib.pg_project_gate_context_noalloc(N, Din, d, M, _p(e), _p(W), _p(h), _p(g1), _p(g1), 1e-6, _p(v),
                                                 _p(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert pg.STATUS[status] == "PG_ERR_SCRATCH_LIMIT"
    assert pg.launch_count() == before


def test_noalloc_takes_no_device_memory(cuda):
    # after a first call (which may load the library's device code, scratch array
    # included), further calls leave the device's free memory unchanged
    from hashed_head_gram_gb300 import pg
    lib = pg.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    N, Din, d, M = 512, 1280, 2560, 4
    e, W, h, gh, gk = _case(N, Din, d, M, 31, cuda)
    v = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    a = torch.empty(M, N, device=cuda)
    args = (N, Din, d, M, _p(e), _p(W), _p(h), _p(gh), _p(gk), 1e-6, _p(v), _p(a), stream)
    assert lib.pg_project_gate_context_noalloc(*args) == 0
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        assert lib.pg_project_gate_context_noalloc(*args) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert pg.device_error() == 0
