"""Multi-rank host logic on CPU (gloo, world size 2): sharding covers every unit once, timings reduce by max."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, n_units, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env()[:2] == (rank, world)
    mine = torch.tensor(list(bench.shard(n_units, rank, world)), dtype=torch.int64)
    sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(sizes, torch.tensor([mine.numel()]))
    width = int(max(s.item() for s in sizes))
    padded = torch.full((width,), -1, dtype=torch.int64)
    padded[:mine.numel()] = mine
    gathered = [torch.zeros(width, dtype=torch.int64) for _ in sizes]
    dist.all_gather(gathered, padded)
    gathered = [g[g >= 0] for g in gathered]
    t = torch.tensor([1.0 + rank])                     # per-rank step time
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        out.put((torch.cat(gathered).tolist(), t.item()))
    dist.destroy_process_group()


@pytest.mark.parametrize("n_units", [1, 2, 7, 64])
def test_shards_cover_units_once(n_units):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, n_units, q)) for r in range(2)]
    for p in procs:
        p.start()
    units, tmax = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(units) == list(range(n_units))
    assert tmax == 2.0


def test_shard_single_rank():
    assert list(bench.shard(5, 0, 1)) == [0, 1, 2, 3, 4]
    assert [len(bench.shard(10, r, 3)) for r in range(3)] == [4, 3, 3]
