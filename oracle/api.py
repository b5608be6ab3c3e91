"""Whole-buffer oracle calls: the collectives over R ranks' raw buffers.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Raw buffers are numpy arrays holding the element type's storage: float32 for
fp32, uint16 bit patterns for fp16 / bf16.  Each call widens the inputs
exactly, runs the literal schedule of ``schedules`` over the partition of
``partition`` and the trees of ``topology``, and narrows the result once
(``numerics``).

* ``allreduce``: [Internals] API section (two buffers, count, dtype, op, the
  communicator, a stream) with the communicator reduced to R and the
  topology; the ring walks each channel in loops, the tree walks each
  channel in chunks over the channel's tree.
* ``fp64_sum`` / ``fp64_max``: the plain definition of AllReduce ([Interview]
  "先弄清楚": every rank ends with the element-wise total).
"""

import numpy as np

from . import numerics, partition, schedules, topology

RING, TREE = 0, 1


def _widen(raws, dtype):
    return [numerics.to_f32(x, dtype) for x in raws]


def allreduce(raws, dtype, op, algo, n_channels, chunk_bytes, local_ranks=1,
              counters=None, hop_rounding=False, pattern="tree", orders=None):
    """AllReduce of the R raw buffers.  Returns R raw output buffers.

    hop_rounding (ring only): every rank keeps its partials in the element
    type between hops, as a ring whose messages travel in that type does --
    each reduction's fp32 result is rounded to the element type (RNE) before
    it is sent on.  Without it partials stay in fp32 until the end.

    pattern / orders (tree only): the head pattern and per-channel intra-node
    orders of the trees (``topology.build_dtree``)."""
    R = len(raws)
    count = int(raws[0].size)
    E = numerics.ELEM_SIZE[dtype]
    if chunk_bytes <= 0 or chunk_bytes % 16:
        raise ValueError("chunk_bytes must be a positive multiple of 16")
    if R % local_ranks:
        raise ValueError("local_ranks must divide R")
    C = chunk_bytes // E
    xs = _widen(raws, dtype)
    out = [np.empty(count, dtype=np.float32) for _ in range(R)]
    chans = partition.channel_ranges(count, E, n_channels)
    hop = None
    if hop_rounding:
        if algo != RING:
            raise ValueError("per-hop rounding is defined for the ring")
        hop = lambda x: numerics.to_f32(numerics.from_f32(x, dtype), dtype)  # noqa: E731
    if algo == RING:
        for (cs, cn) in chans:
            for loop in partition.ring_blocks(cs, cn, R, C):
                res = schedules.ring_allreduce_loop(xs, loop, op, counters, hop=hop)
                for r in range(R):
                    for (bs, bn), blk in zip(loop, res[r]):
                        out[r][bs:bs + bn] = blk
    elif algo == TREE:
        trees = topology.build_dtree(R // local_ranks, local_ranks, n_channels,
                                     pattern=pattern, orders=orders)
        for k, (cs, cn) in enumerate(chans):
            for (s, n) in partition.tree_chunks(cs, cn, C):
                res = schedules.tree_allreduce_chunk(xs, trees[k], s, n, op, counters)
                for r in range(R):
                    out[r][s:s + n] = res[r]
    else:
        raise ValueError("unknown algorithm %r" % (algo,))
    return [numerics.from_f32(o, dtype) for o in out]


def reduce_scatter(raws, dtype, op, counters=None):
    """Ring ReduceScatter: raws[r] holds R*recvcount elements; returns R raw
    buffers of recvcount elements, rank r's being block r."""
    R = len(raws)
    recvcount = int(raws[0].size) // R
    xs = _widen(raws, dtype)
    res = schedules.ring_reduce_scatter(xs, recvcount, op, counters)
    return [numerics.from_f32(x, dtype) for x in res]


def allgather(raws, counters=None):
    """Ring AllGather (bit copies): returns R raw buffers of R*sendcount."""
    return schedules.ring_allgather([np.asarray(x) for x in raws], counters)


def fp64_sum(raws, dtype):
    """Element-wise sum over ranks in fp64 (the plain definition)."""
    acc = np.zeros(raws[0].size, dtype=np.float64)
    for x in _widen(raws, dtype):
        acc += x.astype(np.float64)
    return acc


def fp64_max(raws, dtype):
    acc = np.full(raws[0].size, -np.inf, dtype=np.float64)
    for x in _widen(raws, dtype):
        acc = np.maximum(acc, x.astype(np.float64))
    return acc
