"""The bounded waits of the tensor-core kernels give up and report instead of hanging
(failure handling of this library; the pages have no counterpart). A wait is made to run
out on a barrier and a counter that nothing completes, inside a kernel that holds no copy,
tensor-core operation or TMEM, so the device stays usable; the test then runs the
tensor-core projection and checks it against the oracle."""
import time

import pytest
import torch

from oracle import dense
from tests._helpers import BF16_TOL, rel_l2, to_f64

pytestmark = pytest.mark.gpu


def test_bounded_waits_give_up_and_report(cuda):
    from hashed_head_gram_gb300 import pg
    pg.device_error(clear=True)
    zero = torch.full((1,), 7, dtype=torch.int32, device=cuda)   # the call zeroes it first
    t0 = time.perf_counter()
    pg.selftest_bounded_waits(zero)
    code = pg.device_error(clear=True)                            # synchronizes
    took = time.perf_counter() - t0
    assert code == 2048 | 4096
    assert 1.5 <= took <= 60.0                                    # two waits of about 1 s each
    assert int(zero.item()) == 0
    assert pg.device_error() == 0
    # the device still runs the tcgen05 projection correctly
    g = torch.Generator().manual_seed(5)
    N, Din, d = 300, 256, 512
    e = (torch.randint(-128, 128, (N, Din), generator=g).float() / 64).to(torch.bfloat16)
    W = (torch.randn(d, Din, generator=g) * 0.02).to(torch.bfloat16)
    v = torch.empty(N, d, dtype=torch.bfloat16, device=cuda)
    pg.project_gate(e.to(cuda), W.to(cuda), d, pg.GATE_NONE, v, pg.BF16)
    ref = dense.project(e.double().numpy(), W.double().numpy())
    assert rel_l2(to_f64(v), ref) <= BF16_TOL
    assert pg.device_error() == 0


def test_selftest_rejects_a_bad_word(cuda):
    from hashed_head_gram_gb300 import pg
    with pytest.raises(pg.PgError):
        pg.selftest_bounded_waits(torch.empty(4, dtype=torch.uint8, device=cuda)[1:2])   # misaligned
