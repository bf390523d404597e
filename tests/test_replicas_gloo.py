"""The N>1 path (independent replicas) as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from activation_cnn_gb300 import replicas as R


def test_shard_covers_exactly():
    for total in (0, 1, 7, 8, 64):
        for world in (1, 2, 3, 8):
            spans = [R.shard(total, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == total
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert max(b - a for a, b in spans) - min(b - a for a, b in spans) <= 1
    with pytest.raises(ValueError):
        R.shard(8, 2, 2)


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
    try:
        r, w, lr = R.env()
        span = R.shard(16, w, r)
        local_time = 1.0 + r          # each rank times its own replica
        R.barrier()
        tmax = R.max_over_ranks(local_time)
        imgs = R.sum_over_ranks(span[1] - span[0])
        q.put((r, w, lr, span, tmax, imgs))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and all(o[1] == 2 for o in out)
    assert [o[3] for o in out] == [(0, 8), (8, 16)]
    assert all(o[4] == 2.0 for o in out)     # max over ranks
    assert all(o[5] == 16 for o in out)      # every image processed once
