"""Literal message-passing simulations of the ring and tree schedules.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Every rank's buffer is a numpy float32 array (already widened).  A "send"
copies the sender's block before any receiver applies it, so all ranks send
and receive at the same time, as the pages' simulation does.

Sources:
* [Interview] sections "先弄清楚:每个概念是什么" (reduce-scatter then
  all-gather is all-reduce; ring: each step every rank sends one 1/n block to
  its right-hand neighbour), Figure 1 (the 4-rank, 4-block trace), "推导 /
  关键公式" (each rank sends 2(n-1)/n * S), "手撕代码(NumPy 模拟 ring
  all-reduce)" (at reduce-scatter step s rank r sends block (r-s) mod n to
  r+1, which adds it to its own; at all-gather step s rank r sends block
  (r+1-s) mod n, which overwrites).
* [Internals] section "Ring：带宽友好，但启动步骤会随规模增长": first step
  sends a block, middle steps receive-reduce-send, then reduced blocks are
  forwarded, the last step receives the own final block.
* [Course13] sections "先固定方向" (Reduce: receive from down[], reduce the
  local input, send to up; Broadcast: receive from up, copy, send to down[])
  and "每种 rank 的操作" (root, internal and leaf roles; the chain
  0->1->2->3 trace).
* [CodeNotes] section "通讯时如何选择Channel": tree implements AllReduce only.

Readings:
* Operand order of a tree reduction (the pages are silent): a rank starts
  from its local input and folds each child's partial in down[] slot order.
* ReduceScatter alone: rank r keeps block r ("each card keeps the segment it
  is responsible for").  The reduce-scatter half of the ring AllReduce leaves
  rank r with block r+1; ReduceScatter shifts the block labels by one, so at
  step s rank r sends block (r-s-1) mod n.  Both fold a block starting at the
  rank after its owner and ending at the owner.
* AllGather: rank r's data starts in block r of its own output; at step s
  rank r forwards block (r-s) mod n.
"""

import numpy as np

from . import numerics


class Counters:
    """Per-rank sent element counts and the number of schedule steps."""

    def __init__(self, R):
        self.sent = [0] * R
        self.steps = 0


# ------------------------------------------------------------------ ring
def ring_allreduce_loop(xs, blocks, op, counters=None, trace=None, hop=None):
    """One ring loop over ``blocks`` (R (start, length) pairs, block j) of the
    R float32 buffers ``xs``.  Returns per rank the list of R result blocks.
    ``trace``, when a list, receives a snapshot of every rank's blocks after
    each step, reduce-scatter steps first.  ``hop``, when given, maps every
    partial a rank holds after a reduction to the value it can keep between
    hops (per-hop rounding to a narrower element type)."""
    R = len(xs)
    held = [[xs[r][s:s + n].copy() for (s, n) in blocks] for r in range(R)]

    def snap():
        if trace is not None:
            trace.append([[b.copy() for b in held[r]] for r in range(R)])

    for s in range(R - 1):                       # reduce-scatter
        out = [(r, (r - s) % R, held[r][(r - s) % R].copy()) for r in range(R)]
        for r, j, msg in out:
            dst = (r + 1) % R
            held[dst][j] = numerics.combine(op, held[dst][j], msg)
            if hop is not None:
                held[dst][j] = hop(held[dst][j])
            if counters is not None:
                counters.sent[r] += msg.size
        if counters is not None:
            counters.steps += 1
        snap()
    for s in range(R - 1):                       # all-gather
        out = [(r, (r + 1 - s) % R, held[r][(r + 1 - s) % R].copy()) for r in range(R)]
        for r, j, msg in out:
            held[(r + 1) % R][j] = msg
            if counters is not None:
                counters.sent[r] += msg.size
        if counters is not None:
            counters.steps += 1
        snap()
    return held


def ring_reduce_scatter(xs, recvcount, op, counters=None):
    """Ring ReduceScatter of R buffers of R*recvcount elements; rank r ends
    with block r.  Returns the R result blocks."""
    R = len(xs)
    held = [[xs[r][b * recvcount:(b + 1) * recvcount].copy() for b in range(R)]
            for r in range(R)]
    for s in range(R - 1):
        out = [(r, (r - s - 1) % R, held[r][(r - s - 1) % R].copy()) for r in range(R)]
        for r, b, msg in out:
            dst = (r + 1) % R
            held[dst][b] = numerics.combine(op, held[dst][b], msg)
            if counters is not None:
                counters.sent[r] += msg.size
        if counters is not None:
            counters.steps += 1
    return [held[r][r] for r in range(R)]


def ring_allgather(xs, counters=None):
    """Ring AllGather of R buffers (any dtype, copied bit-exactly): every
    rank ends with all R buffers, rank r's in block r.  Returns R arrays."""
    R = len(xs)
    held = [[None] * R for _ in range(R)]
    for r in range(R):
        held[r][r] = xs[r].copy()
    for s in range(R - 1):
        out = [(r, (r - s) % R, held[r][(r - s) % R].copy()) for r in range(R)]
        for r, b, msg in out:
            held[(r + 1) % R][b] = msg
            if counters is not None:
                counters.sent[r] += msg.size
        if counters is not None:
            counters.steps += 1
    return [np.concatenate(held[r]) for r in range(R)]


# ------------------------------------------------------------------ tree
def _heights(tree):
    """Height of every rank (0 for leaves) in one channel's tree."""
    R = len(tree)
    memo = {}

    def h(v):
        if v not in memo:
            kids = [c for c in tree[v].down if c != -1]
            memo[v] = 0 if not kids else 1 + max(h(c) for c in kids)
        return memo[v]

    return [h(v) for v in range(R)]


def tree_allreduce_chunk(xs, tree, start, length, op, counters=None):
    """Reduce-up then broadcast-down of one chunk [start, start+length) over
    one channel's tree (``tree[rank]`` has ``up`` and ``down``).  Ranks send
    up in rounds by height, leaves first; the root's partial is the result,
    which then travels down one level per round.  Returns per rank the
    chunk's result."""
    R = len(xs)
    hts = _heights(tree)
    roots = [r for r in range(R) if tree[r].up == -1]
    if len(roots) != 1:
        raise RuntimeError("tree must have exactly one root")
    root = roots[0]
    inbox = [dict() for _ in range(R)]          # child -> partial received
    partial = [None] * R
    for level in range(hts[root] + 1):          # reduce-up
        sent_any = False
        for v in range(R):
            if hts[v] != level:
                continue
            acc = xs[v][start:start + length].copy()          # local input first
            for c in tree[v].down:
                if c != -1:
                    acc = numerics.combine(op, acc, inbox[v].pop(c))
            partial[v] = acc
            if tree[v].up != -1:
                inbox[tree[v].up][v] = acc.copy()
                sent_any = True
                if counters is not None:
                    counters.sent[v] += length
        if sent_any and counters is not None:
            counters.steps += 1
    result = [None] * R
    result[root] = partial[root]
    frontier = [root]
    while frontier:                             # broadcast-down
        nxt = []
        for v in frontier:
            for c in tree[v].down:
                if c != -1:
                    result[c] = result[v].copy()
                    nxt.append(c)
                    if counters is not None:
                        counters.sent[v] += length
        if nxt and counters is not None:
            counters.steps += 1
        frontier = nxt
    if any(x is None for x in result):
        raise RuntimeError("tree does not reach every rank")
    return result
