"""Multi-process host logic of bench.py on CPU (gloo, world size 2): each rank owns an
independent batch (no collective on the data path); timing is the max over ranks and
the reported rate counts the units of all ranks."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

from hashed_head_gram_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w_env, r_env, _ = bench.dist_env()
    my_time = 1.0 + rank                       # rank 1 is the slow one
    t_max = bench.reduce_max(my_time, world)
    bench.barrier(world)
    rate = bench.whole_job_rate(1000, world, t_max)
    toks = W.make_tokens(W.shrink(W.make_workload(2), 2, 64), rank=rank)
    q.put((rank, w_env, r_env, t_max, rate, toks))
    dist.destroy_process_group()


def test_two_rank_timing_and_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted([q.get(timeout=120) for _ in procs], key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, w_env, r_env, t_max, rate, _ in out:
        assert (w_env, r_env) == (2, rank)
        assert t_max == 2.0                    # max over ranks
        assert rate == 1000 * 2 / 2.0          # all ranks' units over the slowest time
    t0, t1 = out[0][5], out[1][5]
    assert not np.array_equal(t0, t1)          # independent shards
    assert np.array_equal(t0, W.make_tokens(W.shrink(W.make_workload(2), 2, 64)))  # rank 0 = default stream
