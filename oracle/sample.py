"""Per-element closed forms of the schedules, for checking sampled outputs of
full-size runs one element at a time.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

These restate what the literal simulations in ``schedules`` compute, without
simulating messages:

* ring AllReduce, element in block j of its loop: fold the ranks j, j+1, ...,
  j+R-1 (mod R) left to right -- the block leaves rank j at step 0 and each
  later rank adds its own copy ([Interview] "手撕代码" and Figure 1);
* ring ReduceScatter, element of block b: fold ranks b+1, ..., b (mod R);
* tree AllReduce: P(v) = fold(x_v, P(down[0]), P(down[1]), P(down[2])) over
  present children, the root's P being the result ([Course13] "先固定方向",
  "每种 rank 的操作").

The tests check them against the literal simulations on small inputs.
"""

import numpy as np

from . import numerics, partition, topology


def ring_fold_start(e, count, elem_size, R, n_channels, chunk_elems):
    """Block number j of element e in the ring AllReduce partition."""
    for (cs, cn) in partition.channel_ranges(count, elem_size, n_channels):
        if cs <= e < cs + cn:
            for loop in partition.ring_blocks(cs, cn, R, chunk_elems):
                for j, (bs, bn) in enumerate(loop):
                    if bs <= e < bs + bn:
                        return j
    raise IndexError("element %d outside the message" % e)


def channel_of(e, count, elem_size, n_channels):
    for k, (cs, cn) in enumerate(partition.channel_ranges(count, elem_size, n_channels)):
        if cs <= e < cs + cn:
            return k
    raise IndexError("element %d outside the message" % e)


def fold_in_order(values, order, op):
    """Left fold of ``values[order[0]], values[order[1]], ...`` in fp32."""
    acc = np.float32(values[order[0]])
    for r in order[1:]:
        acc = numerics.combine(op, acc, np.float32(values[r]))
    return np.float32(acc)


def tree_fold(values, tree, op):
    """Post-order fold of one element over one channel's tree."""
    def P(v):
        acc = np.float32(values[v])
        for c in tree[v].down:
            if c != -1:
                acc = numerics.combine(op, acc, P(c))
        return np.float32(acc)
    root = [r for r in range(len(tree)) if tree[r].up == -1]
    assert len(root) == 1
    return P(root[0])


def allreduce_element(values_f32, e, count, dtype, op, algo, n_channels, chunk_bytes,
                      local_ranks=1):
    """Expected fp32 (before narrowing) result of element e, given the R
    widened input values of that element."""
    R = len(values_f32)
    E = numerics.ELEM_SIZE[dtype]
    if algo == 0:
        j = ring_fold_start(e, count, E, R, n_channels, chunk_bytes // E)
        return fold_in_order(values_f32, [(j + k) % R for k in range(R)], op)
    k = channel_of(e, count, E, n_channels)
    trees = topology.build_dtree(R // local_ranks, local_ranks, n_channels)
    return tree_fold(values_f32, trees[k], op)


def reduce_scatter_element(values_f32, block, op):
    """Expected fp32 result of an element of block ``block``."""
    R = len(values_f32)
    return fold_in_order(values_f32, [(block + 1 + k) % R for k in range(R)], op)
