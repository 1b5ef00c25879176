"""Host logic of the N>1 replica path, on CPU with the gloo backend and two
ranks: sharding covers every sequence once, timings combine as max/sum."""
import os
import socket

import torch.multiprocessing as mp

from sparse_kv_verification_gb300 import replicas as R


def test_shard_partitions():
    for total in (0, 1, 5, 16, 17):
        for world in (1, 2, 3, 8):
            spans = [R.shard(total, r, world) for r in range(world)]
            covered = [i for a, b in spans for i in range(a, b)]
            assert covered == list(range(total))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank),
                      WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    r, local, w = R.init("gloo")
    R.barrier()
    mx = R.reduce_max(10.0 + r)
    sm = R.reduce_sum(1.0 + r)
    out.put((r, w, mx, sm, R.shard(16, r, w)))
    R.shutdown()


def test_two_rank_gloo_reductions():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in results] == [0, 1]
    for r, w, mx, sm, span in results:
        assert w == 2 and mx == 11.0 and sm == 3.0
    assert results[0][4] == (0, 8) and results[1][4] == (8, 16)
