"""The multi-process replica path on CPU: two gloo ranks reduce their timings the way the
benchmark does (max time, summed work)."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    from paged_kv_cache_147_gb300 import replicas
    replicas.init("gloo")
    assert replicas.world() == (rank, rank, world)
    replicas.barrier()
    t, u = replicas.aggregate(1.0 + rank, 10.0 * (rank + 1))
    q.put((rank, t, u))
    replicas.shutdown()


def test_two_gloo_ranks_reduce_time_and_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.0, 30.0), (1, 2.0, 30.0)]


def test_single_process_is_identity():
    from paged_kv_cache_147_gb300 import replicas
    assert replicas.aggregate(0.5, 7.0) == (0.5, 7.0)
