"""Fixed-order cross-device reductions of the row-parallel layer, for a run
with one process per GPU (``torch.distributed``).

On one GPU the row-parallel (sharded-to-all) layer sums its N rank partials
inside the kernel, in ascending rank order, and adds the bias once after the
sum (MLX tensor parallelism guide, sections 2.2 and 4; "sharded matrices"
notes, case 3).  With one rank per device the partials live on different
GPUs and the sum becomes a collective.  A ring or tree all-reduce adds them
in an order that depends on the algorithm and the group size, so its result
is not bit-identical to the rank-order sum; these helpers keep that order:

* ``all_sum_rank_order``: all-gather every rank's float32 partial, then every
  rank adds partials 0, 1, ..., N-1 locally, one rounding per add, and adds
  the bias once.  Every rank ends with the same bytes, equal to the
  single-device result.
* ``reduce_scatter_rank_order``: the same partial sums, but rank c keeps only
  column block c (the notes' ReduceScatter, which they recommend over
  AllReduce when the next layer is column-parallel): an all-to-all hands rank
  c every rank's block c (point-to-point sends and receives), and rank c
  adds them in rank order.

Both move N-1 partial blocks per rank, like their ring counterparts, but
gather them whole before adding, so they use N times the receive memory of
one partial.  The arithmetic is plain torch on whatever device the tensors
live on; the kernels of this package do not call these (every call of the
library runs on one GPU).
"""
from __future__ import annotations


def _dist():
    import torch.distributed as dist
    return dist


def all_sum_rank_order(partial, bias=None, group=None):
    """sum over ranks r = 0..N-1 of ``partial`` (ascending, left to right),
    then ``+ bias`` once; the same tensor on every rank."""
    import torch
    dist = _dist()
    n = dist.get_world_size(group)
    parts = [torch.empty_like(partial) for _ in range(n)]
    dist.all_gather(parts, partial.contiguous(), group=group)
    total = parts[0].clone()
    for p in parts[1:]:
        total += p
    if bias is not None:
        total += bias
    return total


def reduce_scatter_rank_order(partial, bias=None, group=None):
    """Column block c (of N equal blocks of the last axis) of the rank-order
    sum of every rank's ``partial``, on rank c; ``bias`` is the full-width
    bias, of which block c is added once after the sum."""
    import torch
    dist = _dist()
    n = dist.get_world_size(group)
    c = dist.get_rank(group)
    cols = partial.shape[-1]
    if cols % n:
        raise ValueError("cannot scatter %d columns over %d ranks" % (cols, n))
    w = cols // n
    send = [partial[..., k * w:(k + 1) * w].contiguous() for k in range(n)]
    recv = [torch.empty_like(send[0]) for _ in range(n)]
    # the all-to-all as point-to-point sends and receives (every backend has them)
    ops = []
    for k in range(n):
        if k == c:
            recv[k].copy_(send[k])
            continue
        peer = dist.get_global_rank(group, k) if group is not None else k
        ops.append(dist.P2POp(dist.isend, send[k], peer, group))
        ops.append(dist.P2POp(dist.irecv, recv[k], peer, group))
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()
    total = recv[0].clone()
    for p in recv[1:]:
        total += p
    if bias is not None:
        total += bias[..., c * w:(c + 1) * w]
    return total
