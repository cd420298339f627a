"""Host logic of the multi-process benchmark path, on CPU with gloo.

The fused KV-cache write has no exchange step: each rank writes its own
batch (replicas), and only the timing is combined: slowest rank's time,
sum of the ranks' tokens."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms, tokens = bench.combine_ranks(1.0 + rank, 100 * (rank + 1), world)
    out.put((rank, ms, tokens))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_combine_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tokens in res:
        assert ms == float(world)  # slowest rank
        assert tokens == 100 * world * (world + 1) // 2


def test_single_rank_is_identity():
    import bench

    assert bench.combine_ranks(2.5, 7, 1) == (2.5, 7)
