"""bench.py's multi-rank plumbing on CPU with gloo, world size 2: ranks are independent replicas
(no collective on the data path); the step time is the max over ranks and the reported value
aggregates all ranks' tokens."""
import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    my_ms = 1.0 + rank                      # rank 1 is the slower replica
    ms = bench.max_over_ranks(my_ms, w)
    tokens_per_rank = 16
    value = w * tokens_per_rank / (ms * 1e-3)
    q.put((rank, ms, value))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_replicas_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    assert [r[1] for r in res] == [2.0, 2.0]                    # max over ranks
    assert all(abs(r[2] - 2 * 16 / 2e-3) < 1e-6 for r in res)  # whole-job tokens/s
