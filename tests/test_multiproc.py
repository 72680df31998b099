"""The bench's multi-process path on CPU (gloo, world size 2): one process
per rank, each with its own batch of sequences (weak scaling, independent
problems, no collective on the data path), a barrier around the timed region
and the time taken as the maximum over the ranks."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    import synth

    r, local, w = bench._dist()
    assert (r, local, w) == (rank, rank, world)
    assert dist.get_backend() == "gloo"
    # the slowest rank's time is the job's
    assert bench._max_over_ranks(1.0 + rank, world) == float(world)
    bench._barrier(world)
    # each rank's own batch: different keys, the layer's shared codebook
    wl = synth.scaled(synth.WORKLOADS["tiny"], N=256, K=16, M=64)
    keys, cb, _, _ = bench._inputs(wl, rank)
    sums = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
    mine = torch.tensor([keys.double().sum().item(), cb.double().sum().item()], dtype=torch.float64)
    dist.all_gather(sums, mine)
    out[rank] = [s.tolist() for s in sums]
    dist.destroy_process_group()


def test_two_ranks_on_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        if p.is_alive():
            p.kill()
            pytest.fail("a rank did not finish")
        assert p.exitcode == 0
    (k0, c0), (k1, c1) = out[0]
    assert k0 != k1          # independent batches
    assert c0 == c1          # one layer's codebook
    assert out[0] == out[1]  # both ranks saw the same gather
