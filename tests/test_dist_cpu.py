"""Multi-rank paths on CPU (`gloo`).

* The N > 1 plumbing of bench.py: two ranks exchange their step times and work
  as the bench does under torchrun (max time over ranks, summed units: weak
  scaling, every rank running its own problem), and the reference arm does no
  work on ranks other than 0.
* The row-parallel layer's sum across devices (sharded_gemm_gb300.dist): 2
  and 4 ranks, each holding one shard, all-sum or reduce-scatter their
  float32 partials in rank order."""
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


# ---------------------------------------------------------------- the row-parallel sum across ranks
def _split_worker(rank, world, port, q, T, K, O, seed):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import torch.distributed as dist
    from sharded_gemm_gb300 import dist as tpdist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # every rank draws the whole problem (same seed) and keeps its own shard:
    # x_r = x[:, r K/N:(r+1) K/N], W_r = W[:, same columns]; its partial is
    # x_r W_r^T in float32, formed from zero
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K)).astype(np.float32)
    w = (rng.standard_normal((O, K)) * 0.05).astype(np.float32)
    b = rng.standard_normal(O).astype(np.float32)
    kn = K // world
    part = torch.from_numpy(x[:, rank * kn:(rank + 1) * kn]) @ torch.from_numpy(w[:, rank * kn:(rank + 1) * kn]).T
    y = tpdist.all_sum_rank_order(part, torch.from_numpy(b))
    blk = tpdist.reduce_scatter_rank_order(part, torch.from_numpy(b))
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, y.numpy().tobytes(), blk.numpy().tobytes(), tuple(blk.shape)))


@pytest.mark.parametrize("world", [2, 4])
def test_rank_order_sum_across_gloo_ranks_is_bit_identical(world):
    # The multi-device form of the row-parallel layer: every rank's all-sum
    # is the same bytes, equal to one process adding the same float32
    # partials in rank order then the bias; the reduce-scatter blocks are
    # the column blocks of that sum, bit for bit; both match the fp64
    # unsharded x W^T + b within the float32 tolerance.
    import numpy as np
    import torch
    import oracle
    T, K, O, seed = 5, 96, 24, 11
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_split_worker, args=(r, world, port, q, T, K, O, seed)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ys = [o[1] for o in out]
    assert len(set(ys)) == 1  # bit-identical on every rank
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K)).astype(np.float32)
    w = (rng.standard_normal((O, K)) * 0.05).astype(np.float32)
    b = rng.standard_normal(O).astype(np.float32)
    kn = K // world
    parts = [torch.from_numpy(x[:, r * kn:(r + 1) * kn]) @ torch.from_numpy(w[:, r * kn:(r + 1) * kn]).T
             for r in range(world)]
    ref = parts[0].clone()
    for p in parts[1:]:
        ref += p
    ref += torch.from_numpy(b)
    y = np.frombuffer(ys[0], dtype=np.float32).reshape(T, O)
    assert y.tobytes() == ref.numpy().tobytes()  # the single-process rank-order sum
    for c, (_, _, blk, shape) in enumerate(out):
        got = np.frombuffer(blk, dtype=np.float32).reshape(shape)
        assert got.tobytes() == np.ascontiguousarray(y[:, c * (O // world):(c + 1) * (O // world)]).tobytes()
    exact = oracle.sharded_to_all([x[:, r * kn:(r + 1) * kn].astype(np.float64) for r in range(world)],
                                  [w[:, r * kn:(r + 1) * kn].astype(np.float64) for r in range(world)],
                                  b.astype(np.float64))
    assert np.abs(y - exact).max() <= 1e-4 * (np.abs(exact).max() + 1)
