"""Multi-rank host logic on CPU (gloo, world size 2): frequency sharding,
max-over-ranks timing and the final gather of solutions."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from mixed_precision_refinement_gb300 import sharding


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, nf, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        idx = sharding.shard(nf, world, rank)
        # a stand-in "solve": each frequency's solution is filled with its index
        x = np.stack([np.full((2, 5), complex(f, -f)) for f in idx]) if len(idx) else np.zeros((0, 2, 5), complex)
        t = sharding.max_over_ranks(10.0 * (rank + 1))
        full = sharding.gather_solutions(x, nf, world, rank)
        if rank == 0:
            q.put((t, full))
    finally:
        dist.destroy_process_group()


def test_shard_partition():
    for nf in (1, 5, 21):
        for world in (1, 2, 3, 8):
            got = np.sort(np.concatenate([sharding.shard(nf, world, r) for r in range(world)]))
            assert np.array_equal(got, np.arange(nf))
    with pytest.raises(ValueError):
        sharding.shard(4, 2, 2)


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    nf = 7
    procs = [ctx.Process(target=_worker, args=(r, 2, port, nf, q)) for r in range(2)]
    for p in procs:
        p.start()
    t, full = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert t == 20.0
    for f in range(nf):
        assert np.all(full[f] == complex(f, -f))
