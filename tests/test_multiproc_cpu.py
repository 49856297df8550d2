"""Multi-process path of bench.py on CPU (gloo, world size 2).

The decode path shards by sequence / KV head with no exchange step, so with N
GPUs bench.py runs N independent replicas and reports the slowest rank's time
(max over ranks) and the whole-job throughput.  These tests run that host
logic with two gloo ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    vals = bench.max_over_ranks([10.0 + rank, 20.0 - rank, 5.0 * (rank + 1)])
    thr = bench.replica_throughput(vals[0], world)
    q.put((rank, vals, thr))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, vals, thr in out:
        assert vals == [11.0, 20.0, 10.0]                 # element-wise max over both ranks
        assert thr == pytest.approx(2 / 11e-6)            # two replicas, slowest rank's time


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.replica_throughput(100.0, 1) == pytest.approx(1e4)


def test_cycled_cache_copies_exceed_twice_l2():
    """The bench cycles its steps over cache copies: between two uses of a
    copy the others read more than 2x L2 (or one copy alone exceeds it)."""
    import bench
    l2 = 126 << 20
    for nbytes in (7 << 20, 33554432, 113246208, 134 << 20, 253 << 20, 906 << 20):
        c = bench.copies_for(nbytes, l2)
        if c == 1:
            assert nbytes > 2 * l2
        else:
            assert (c - 1) * nbytes >= 2 * l2
    assert bench.copies_for(113246208, l2) == 4
