"""The N > 1 plumbing of bench.py on CPU: two `gloo` ranks exchange their step
times and work as the bench does under torchrun (max time over ranks, summed
units: weak scaling, every rank running its own problem), and the reference
arm does no work on ranks other than 0."""
import multiprocessing as mp
import os
import socket
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, loc = bench.dist_env()
    ms, units = bench.aggregate(1.0 + rank, 10.0 * (rank + 1), w)
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, w, loc, ms, units))


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and all(o[1] == 2 for o in out)
    assert [o[2] for o in out] == [0, 1]
    for _, _, _, ms, units in out:
        assert ms == 2.0          # the slowest rank's step time
        assert units == 30.0      # 10 + 20: the work of both ranks


def test_single_rank_aggregate_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(3.5, 7.0, 1) == (3.5, 7.0)


def test_reference_arm_only_on_rank_zero(capsys):
    sys.path.insert(0, ROOT)
    import bench
    args = types.SimpleNamespace(config="mlp", steps=1, warmup=0)
    bench.main_reference(args, world=2, rank=1)
    assert capsys.readouterr().out == ""
