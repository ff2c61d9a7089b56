"""The benchmark's multi-rank bookkeeping on CPU (gloo, world size 2): every rank
times its own GPU's batch (weak scaling, no collective on the data path); the
job's throughput is the units of all ranks over the slowest rank's time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r processed 1e9 * (r + 1) bytes and 8 tokens per step in 0.5 * (r + 1) s
    gbs, tok, t = bench.aggregate(1e9 * (rank + 1) / 10, 8, 0.5 * (rank + 1), 10)
    bench.barrier()
    q.put((rank, gbs, tok, t, bench.dist_env()))
    dist.destroy_process_group()


def test_aggregate_is_total_units_over_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, gbs, tok, t, env = q.get(timeout=120)
        res[rank] = (gbs, tok, t, env)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (gbs, tok, t, env) in res.items():
        assert t == pytest.approx(1.0)                     # max over ranks
        assert gbs == pytest.approx((1e9 + 2e9) / 1.0 / 1e9)
        assert tok == pytest.approx(2 * 8 * 10 / 1.0)
        assert env == (2, rank, rank)


def test_single_process_aggregate_is_identity():
    import bench
    gbs, tok, t = bench.aggregate(2e9, 8, 2.0, 4)
    assert (gbs, tok, t) == (pytest.approx(4.0), pytest.approx(16.0), 2.0)
