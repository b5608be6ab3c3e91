"""Ring and double-binary-tree topology, written from the pages' description.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).  Pure-Python integers.

Sources:
* [Course13] "NCCL 专家课程 13：Tree、双树、层次化连接与真实交叉区间",
  sections "先固定方向" (up = parent, down[] = children), "数据结构不是纯二叉树"
  (ncclTree {depth, up, down[3]}), "节点内先形成链" (ncclTopoPreset: the
  intra-node chain and the head ranks), "节点间连接" (connectTrees: Dtree over
  the node index, heads joined, the depth formula), "Btree 的 bit 构造"
  (ncclGetBtree), "双树：偶数 mirror，奇数 shift" (ncclGetDtree).
* [Interview] "all-reduce 每张卡要发多少数据? ring 和 tree 有什么区别?",
  section "先弄清楚:每个概念是什么" (ring: every rank sends to its right-hand
  neighbour; two complementary trees each carry half of the data).

Readings where the pages are silent:
* setTreeUp / setTreeDown bodies are not shown.  setTreeUp assigns ``up``
  (nothing when the node-level parent is -1); setTreeDown appends the child to
  the first -1 slot of ``down[]`` (nothing when the child is -1) and fails past
  three slots.  Supported by the log "Tree 0 : -1 -> 0 -> 1/-1/-1" (a root's
  only child sits in slot 0) and by leaf detection through ``down[0] == -1``.
* With no topology search, the intra-node order ``treeIntra`` is the identity
  (local rank l of node k is global rank k*L + l) unless the caller gives one
  per channel.  The head pattern picks the parent and child heads from that
  order as section "节点内先形成链" shows: TREE uses position 0 for all three,
  SPLIT_TREE 0 / 1 / 1, and any other pattern (BALANCED_TREE) 0 / 1 / 0.
* The ring has no physical search either: every channel uses the identity ring.
* Channel -> tree: the channel metadata is duplicated so that one copy joins
  tree 0 and the other tree 1, each carrying half the data.  Channels
  [0, ceil(nCh/2)) use tree 0, the rest tree 1; one channel uses tree 0 only.
"""

import functools
import math
from dataclasses import dataclass, field
from typing import List


# ------------------------------------------------------------------- ring
def build_ring(R, n_channels):
    """Identity ring for every channel: next = r+1, prev = r-1 (mod R).
    Returns (next, prev), each a list of n_channels lists of R ints."""
    if R < 1 or n_channels < 1:
        raise ValueError("R and n_channels must be >= 1")
    nxt = [[(r + 1) % R for r in range(R)] for _ in range(n_channels)]
    prv = [[(r - 1 + R) % R for r in range(R)] for _ in range(n_channels)]
    return nxt, prv


# ------------------------------------------------------------------ trees
def _level(v):
    """A node's level in the bit-trick tree: the lowest set bit of its index
    (1, 2, 4, ...); node 0, the root, lies above every level."""
    return math.inf if v == 0 else v & -v


@functools.lru_cache(maxsize=None)
def _parents(n):
    """Every node's parent in the tree of the levels over n nodes (see
    ``btree``): the nearer-level of its nearest higher-level neighbours."""
    def parent(v):
        if v == 0:
            return -1
        lv = _level(v)
        left = next(u for u in range(v - 1, -1, -1) if _level(u) > lv)
        right = next((u for u in range(v + 1, n) if _level(u) > lv), None)
        if right is None or _level(left) < _level(right):
            return left
        return right
    return tuple(parent(v) for v in range(n))


def btree(n, r):
    """Node r of the bit-trick binary tree over n nodes ([Course13] "Btree 的
    bit 构造").

    The section builds the tree from each node's lowest set bit: the parent
    is found by clearing that bit and setting the next one up (only clearing
    it when that leaves the range), and the children sit half that bit to
    either side, the upper one pulled closer until it exists.  The tree those
    steps give is, read in index order, the tree of the levels: every node
    hangs under the nearer-level one of the nearest higher-level node on its
    left and the nearest higher-level node on its right (the left one when
    there is none on the right).  A node's lower child is then the child on
    its left and its upper child the child on its right.  That form is
    written out here by brute force over all n nodes, so it shares no step
    with the bit arithmetic (the pins compare it with the pages' tables).

    parentChildType is 0 when r lies below its parent, else 1 (-1 for the
    root, whose type the section leaves unset).

    Returns (up, d0, d1, parentChildType)."""
    if not (0 <= r < n):
        raise ValueError("rank %d outside [0, %d)" % (r, n))
    par = _parents(n)
    up = par[r]
    kids = [v for v in range(n) if par[v] == r]
    d0 = next((v for v in kids if v < r), -1)
    d1 = next((v for v in kids if v > r), -1)
    return (up, d0, d1, -1 if up == -1 else (0 if r < up else 1))


def dtree(n, r):
    """The two node-level trees of node r: tree 0 is btree(n, r); tree 1 is
    btree of a relabelled node mapped back -- mirror r -> n-1-r for even n,
    shift r -> r-1 (mod n) for odd n, with the outputs mapped back by the
    inverse relabelling (-1 stays -1, slot order kept).

    Returns ((u0, d0_0, d0_1, t0), (u1, d1_0, d1_1, t1))."""
    t0 = btree(n, r)
    if n % 2 == 1:
        u, a, b, t = btree(n, (r - 1 + n) % n)
        back = lambda x: -1 if x == -1 else (x + 1) % n  # noqa: E731
    else:
        u, a, b, t = btree(n, n - 1 - r)
        back = lambda x: -1 if x == -1 else n - 1 - x  # noqa: E731
    return t0, (back(u), back(a), back(b), t)


def log2i(n):
    """floor(log2 n) for n >= 1."""
    k = 0
    while n > 1:
        n >>= 1
        k += 1
    return k


@dataclass
class Tree:
    """One rank's view of one tree, the ncclTree record."""
    depth: int
    up: int
    down: List[int] = field(default_factory=lambda: [-1, -1, -1])


def _set_up(t, parent):
    if parent != -1:
        t.up = parent


def _set_down(t, child):
    if child == -1:
        return
    for s in range(3):
        if t.down[s] == -1:
            t.down[s] = child
            return
    raise RuntimeError("more than three children")


def channel_tree_index(channel, n_channels):
    """0 for the first half of the channels (rounded up), 1 for the rest."""
    return 0 if channel < (n_channels + 1) // 2 else 1


PATTERNS = ("tree", "split_tree", "balanced_tree")


def head_indices(pattern):
    """Positions in a node's intra order of the rank that joins the parent
    node, the rank that takes child d0 and the rank that takes child d1:
    TREE (0, 0, 0), SPLIT_TREE (0, 1, 1), BALANCED_TREE (0, 1, 0)."""
    if pattern == "tree":
        return 0, 0, 0
    if pattern == "split_tree":
        return 0, 1, 1
    if pattern == "balanced_tree":
        return 0, 1, 0
    raise ValueError("unknown pattern %r" % (pattern,))


def build_dtree(n_nodes, local_ranks, n_channels, pattern="tree", orders=None):
    """Per channel and rank, the hierarchical double-binary-tree record.

    Step 1 (preset): on channel c each node's ranks form a chain in the
    channel's intra order (``orders[c]``, a permutation of the local ranks;
    identity when None): up = the previous rank of the order, down[0] = the
    next one.  The pattern picks which positions of the order are the node's
    parent head and its two child heads.  Step 2 (connect): the node-level
    double tree over node indices (not rank indices) is attached: the parent
    head of node k takes up = the child head (child0 or child1 by k's
    parentChildType) of its parent node; the child0 head appends the parent
    head of child node d0, then the child1 head appends that of d1.  Every
    rank's depth is L - 1 + floor(log2 nNodes), the page's approximation.

    Returns trees[channel][rank] -> Tree."""
    if n_nodes < 1 or local_ranks < 1 or n_channels < 1:
        raise ValueError("sizes must be >= 1")
    L = local_ranks
    R = n_nodes * L
    pi, c0i, c1i = head_indices(pattern)
    if max(pi, c0i, c1i) >= L:
        raise ValueError("pattern needs more local ranks")
    depth = L - 1 + log2i(n_nodes)
    node_trees = [dtree(n_nodes, k) for k in range(n_nodes)]
    out = []
    for c in range(n_channels):
        t_idx = channel_tree_index(c, n_channels)
        order = list(range(L)) if orders is None else list(orders[c])
        if sorted(order) != list(range(L)):
            raise ValueError("intra order must be a permutation of the local ranks")
        intra = [[k * L + order[i] for i in range(L)] for k in range(n_nodes)]
        per_rank = [None] * R
        for k in range(n_nodes):
            for i, rank in enumerate(intra[k]):
                per_rank[rank] = Tree(depth=depth,
                                      up=-1 if i == 0 else intra[k][i - 1],
                                      down=[-1 if i == L - 1 else intra[k][i + 1], -1, -1])
        ttp = [intra[k][pi] for k in range(n_nodes)]
        ttc0 = [intra[k][c0i] for k in range(n_nodes)]
        ttc1 = [intra[k][c1i] for k in range(n_nodes)]
        for k in range(n_nodes):
            u, d0, d1, ptype = node_trees[k][t_idx]
            if u != -1:
                _set_up(per_rank[ttp[k]], (ttc0 if ptype == 0 else ttc1)[u])
            if d0 != -1:
                _set_down(per_rank[ttc0[k]], ttp[d0])
            if d1 != -1:
                _set_down(per_rank[ttc1[k]], ttp[d1])
        out.append(per_rank)
    return out


# ------------------------------------------------------- tree inspection
def root_of(trees_one_channel):
    roots = [r for r, t in enumerate(trees_one_channel) if t.up == -1]
    return roots


def exact_depth(trees_one_channel):
    """Edges from the root to the deepest leaf (walks every rank to the root)."""
    worst = 0
    for r in range(len(trees_one_channel)):
        d, v, seen = 0, r, set()
        while trees_one_channel[v].up != -1:
            if v in seen:
                raise RuntimeError("cycle")
            seen.add(v)
            v = trees_one_channel[v].up
            d += 1
        worst = max(worst, d)
    return worst


def internal_nodes(trees_one_channel):
    """Non-leaf ranks, the root included."""
    return {r for r, t in enumerate(trees_one_channel) if any(c != -1 for c in t.down)}


def format_tree_log(trees_one_channel, channel, style="arrow"):
    """The two log line styles the pages quote: "Tree c : up -> rank ->
    d0/d1/d2" and "Trees [c] d0/d1/d2->rank->up", one line per rank."""
    lines = []
    for r, t in enumerate(trees_one_channel):
        kids = "/".join(str(x) for x in t.down)
        if style == "arrow":
            lines.append("Tree %d : %d -> %d -> %s" % (channel, t.up, r, kids))
        else:
            lines.append("Trees [%d] %s->%d->%d" % (channel, kids, r, t.up))
    return lines
