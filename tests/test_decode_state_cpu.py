"""The streaming-decode state's ring arithmetic (no GPU): the ID ring returns the canonical
ID of position t - j for every t and j <= 3, and with a conv ring of (k - 1) dil + 1 slots
the slot a decode step writes (position t) is never one of the slots it reads (positions
t - j dil), so blocks of one launch never race on it; the state's size follows the layout
pg_decode_state_size documents."""
import itertools

import pytest

from hashed_head_gram_gb300 import workloads as W


def test_id_ring_returns_the_window():
    ring = [None] * 4
    history = []
    for t in range(40):
        # what a lookup at position t reads (the pages' suffix window, PAD before the start)
        window = [ring[(t - j) & 3] if t >= j else "PAD" for j in range(1, 4)]
        assert window == [history[t - j] if t >= j else "PAD" for j in range(1, 4)]
        ring[t & 3] = f"id{t}"
        history.append(f"id{t}")


@pytest.mark.parametrize("ks,dil", list(itertools.product(range(1, 5), range(1, 9))))
def test_conv_ring_reads_never_meet_the_write(ks, dil):
    D = (ks - 1) * dil + 1 if ks > 1 else 0
    if D == 0:
        return                      # a 1-tap conv reads no earlier position
    ring = {}
    for t in range(3 * D + 5):
        reads = [(t - j * dil) % D for j in range(1, ks) if t - j * dil >= 0]
        assert t % D not in reads
        for j in range(1, ks):
            p = t - j * dil
            if p >= 0:
                assert ring[p % D] == p   # the slot still holds the position the tap needs
        ring[t % D] = t


def test_state_size_matches_the_documented_layout():
    pytest.importorskip("ctypes")
    from hashed_head_gram_gb300.build import build
    build()
    from hashed_head_gram_gb300 import pg
    up = lambda x: (x + 255) // 256 * 256
    for B, d, M, dt, ks, dil in [(1, 0, 0, pg.BF16, 4, 3), (8, 2560, 4, pg.BF16, 4, 3), (3, 64, 8, pg.F32, 2, 8),
                                 (5, 256, 1, pg.BF16, 1, 3)]:
        D = (ks - 1) * dil + 1 if (M and ks > 1) else 0
        es = 4 if dt == pg.F32 else 2
        want = up(4 * B) + up(16 * B) + up(B * D * d * es) + up(B * D * M * 4) + up(B * D * 4)
        assert pg.decode_state_size(B, d, M, dt, ks, dil) == want, (B, d, M, ks, dil)


def test_workload_decode_geometry():
    # the Engram-27B module: kernel 4, dilation 3 -> 9 earlier conv inputs + the current one
    w = W.make_workload(5)
    assert (w.conv_kernel, w.dilation) == (4, 3)
    assert (w.conv_kernel - 1) * w.dilation + 1 == 10
