"""bench.py's multi-rank host logic (replicas: barrier, max / sum over ranks)
with two gloo ranks on CPU."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, l = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(w)
    mx = bench.reduce_max(10.0 + rank, w)
    sm = bench.reduce_sum(1.5 * (rank + 1), w)
    q.put((r, w, l, mx, sm))
    dist.destroy_process_group()


def test_two_rank_replica_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    for r in res:
        assert r[1] == 2 and r[3] == 11.0 and r[4] == pytest.approx(4.5)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.0, 1) == 3.0
    assert bench.reduce_sum(3.0, 1) == 3.0


def test_bytes_touched_closed_form():
    import bench
    from gen.configs import CONFIGS
    c = CONFIGS["full_b1"]
    b = bench.bytes_touched(c, 16, 1)
    assert b == 16 * 17547264 + 896 * 7168 * 2 + 4 * 896 + 3 * 7168 * 1536 * 2 + 2 * 7168 + 8 * 7168
    assert abs(b / 1e6 - 359.74) < 0.01
