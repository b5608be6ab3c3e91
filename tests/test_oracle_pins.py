"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself: the expected values are the
pages' printed examples (tests/golden), hand evaluations of the stated
rules, closed forms, invariants, or brute force on inputs where every
summation order is exact.
"""

import itertools

import numpy as np
import pytest

import oracle
from oracle import numerics, partition, sample, schedules, topology
from tests.tolerances import check_against_fp64

F32, F16, BF16 = numerics.FLOAT32, numerics.FLOAT16, numerics.BFLOAT16
SUM, MAX = numerics.SUM, numerics.MAX
RING, TREE = 0, 1


# ------------------------------------------------------------ worked examples
@pytest.mark.parametrize("algo", [RING, TREE])
def test_two_rank_example(algo):
    # [Interview] "先弄清楚": 2 cards (1, 2), (3, 4) -> both get (4, 6)
    xs = [np.array([1, 2], np.float32), np.array([3, 4], np.float32)]
    out = oracle.allreduce(xs, F32, SUM, algo, n_channels=1, chunk_bytes=16)
    for o in out:
        assert o.tolist() == [4.0, 6.0]


LETTER = {"a": 1, "b": 2, "c": 4, "d": 8, "S": 15}


def _mask(cell):
    return sum(LETTER[t] for t in cell.split("+"))


def test_ring_trace_figure1(golden):
    # [Interview] Figure 1: every cell of the 4-GPU, 4-block ring trace.
    # Rank r holds 2**r, so a cell's value is the bitmask of its contributors.
    rows = golden("ring4_trace.txt")
    states = {}
    for row in rows:
        name, rest = row.split(None, 1)
        states[name] = [[_mask(c) for c in gpu.split()] for gpu in rest.split("|")]
    xs = [np.full(4, 2.0 ** r, np.float32) for r in range(4)]
    blocks = [(j, 1) for j in range(4)]
    trace = []
    schedules.ring_allreduce_loop(xs, blocks, SUM, trace=trace)
    assert len(trace) == 6
    assert [[int(xs[r][j]) for j in range(4)] for r in range(4)] == states["start"]
    for name, snap in zip(["rs1", "rs2", "rs3", "ag1", "ag2", "ag3"], trace):
        got = [[int(snap[r][j][0]) for j in range(4)] for r in range(4)]
        assert got == states[name], name


@pytest.mark.parametrize("R", [2, 3, 4, 5, 8, 9])
def test_ring_traffic_closed_form(R):
    # [Interview] "推导 / 关键公式": each rank sends 2(n-1) * S/n; 2(n-1) steps
    S = R * 6
    xs = [np.ones(S, np.float32) for _ in range(R)]
    cnt = schedules.Counters(R)
    blocks = partition.split_ranges(S, R)
    schedules.ring_allreduce_loop(xs, blocks, SUM, counters=cnt)
    assert cnt.sent == [2 * (R - 1) * S // R] * R
    assert cnt.steps == 2 * (R - 1)


def test_ring_four_ranks_sends_one_and_a_half_S():
    # [Interview] Figure 1 caption: 6 sends of S/4 = 1.5 S per card
    xs = [np.ones(4, np.float32) for _ in range(4)]
    cnt = schedules.Counters(4)
    schedules.ring_allreduce_loop(xs, partition.split_ranges(4, 4), SUM, counters=cnt)
    assert cnt.sent == [6, 6, 6, 6]


def test_step_counts_figure2():
    # [Interview] Figure 2: 8 cards, ring 2(n-1) = 14 steps, tree ~ 2 log2 n = 6
    xs = [np.ones(8, np.float32) for _ in range(8)]
    cnt = schedules.Counters(8)
    schedules.ring_allreduce_loop(xs, partition.split_ranges(8, 8), SUM, counters=cnt)
    assert cnt.steps == 14
    tree = topology.build_dtree(8, 1, 1)[0]
    cnt = schedules.Counters(8)
    schedules.tree_allreduce_chunk(xs, tree, 0, 8, SUM, counters=cnt)
    assert cnt.steps == 6


def test_tree_steps_1024_nodes():
    # [Interview] Figure 2: at n = 1024 the tree needs about 20 steps
    tree = topology.build_dtree(1024, 1, 1)[0]
    assert topology.exact_depth(tree) == 10


# ------------------------------------------------------------------ topology
def test_dtree4_figure(golden):
    want = {}
    for row in golden("dtree4_figure.txt"):
        t, node, up, kids = row.split()
        want[(int(t), int(node))] = (int(up), [] if kids == "-" else [int(k) for k in kids.split(",")])
    for c, t in [(0, 0), (1, 1)]:
        trees = topology.build_dtree(4, 1, 2)[c]
        for node in range(4):
            got = (trees[node].up, [d for d in trees[node].down if d != -1])
            assert got == want[(t, node)], (t, node)
    assert topology.internal_nodes(topology.build_dtree(4, 1, 2)[0]) == {0, 2}
    assert topology.internal_nodes(topology.build_dtree(4, 1, 2)[1]) == {1, 3}


def test_probe_table(golden):
    for row in golden("dtree_probe.txt"):
        n, how, roots, depths, overlap = row.split()
        n = int(n)
        ch = topology.build_dtree(n, 1, 2)
        t0, t1 = ch[0], ch[1]
        assert "%d/%d" % (topology.root_of(t0)[0], topology.root_of(t1)[0]) == roots
        assert "%d/%d" % (topology.exact_depth(t0), topology.exact_depth(t1)) == depths
        ov = topology.internal_nodes(t0) & topology.internal_nodes(t1)
        assert (",".join(str(x) for x in sorted(ov)) or "none") == overlap
        if how in ("mirror", "shift"):
            assert (how == "mirror") == (n % 2 == 0)


@pytest.mark.parametrize("n", [3, 5, 7])
def test_odd_overlap_at_node0(n):
    # [Course13] "真实交叉区间" summary: odd 3, 5, 7 node counts overlap at node 0
    ch = topology.build_dtree(n, 1, 2)
    assert topology.internal_nodes(ch[0]) & topology.internal_nodes(ch[1]) == {0}


def test_hand_derived_trees_r8_r7():
    # Worked by hand from the Btree bit rules and the mirror / shift relabel.
    def kids(tr):
        return {r: [d for d in t.down if d != -1] for r, t in enumerate(tr) if t.down[0] != -1}
    c8 = topology.build_dtree(8, 1, 2)
    assert kids(c8[0]) == {0: [4], 4: [2, 6], 2: [1, 3], 6: [5, 7]}
    assert kids(c8[1]) == {7: [3], 3: [5, 1], 5: [6, 4], 1: [2, 0]}
    c7 = topology.build_dtree(7, 1, 2)
    assert kids(c7[0]) == {0: [4], 4: [2, 6], 2: [1, 3], 6: [5]}
    assert kids(c7[1]) == {1: [5], 5: [3, 0], 3: [2, 4], 0: [6]}


def test_btree_root_and_parent_types():
    # rank 0 is the root with one child, the largest power of two below n
    for n in range(2, 70):
        up, d0, d1, _ = topology.btree(n, 0)
        assert (up, d0) == (-1, -1) and d1 == 1 << (n - 1).bit_length() - 1
    assert topology.btree(1, 0)[:3] == (-1, -1, -1)
    # parentChildType: 0 when the rank is below its parent
    for n in range(2, 40):
        for r in range(1, n):
            up, _, _, t = topology.btree(n, r)
            assert t == (0 if r < up else 1)


def test_active_chains_and_log_line(golden):
    rows = dict(row.split(None, 1) for row in golden("active_trees.txt"))
    for N in (2, 3, 4):
        tr = topology.build_dtree(1, N, 1)[0]
        order, v = [], topology.root_of(tr)[0]
        while v != -1:
            order.append(v)
            v = tr[v].down[0]
        want_order, want_depth, want_fan = rows["chain_1node_%dranks" % N].split()
        assert "-".join(map(str, order)) == want_order
        assert "depth=%d" % topology.exact_depth(tr) == want_depth
        assert "fanout=%d" % max(sum(d != -1 for d in t.down) for t in tr) == want_fan
    tr = topology.build_dtree(1, 2, 1)[0]
    assert topology.format_tree_log(tr, 0)[0] == rows["log_line"]
    assert topology.format_tree_log(tr, 0, style="trees")[1] == "Trees [0] -1/-1/-1->1->0"
    assert topology.build_dtree(1, 4, 3)[2][1].depth == int(rows["depth_field_4ranks_1node"])


def _check_invariants(tr, R):
    roots = [r for r in range(R) if tr[r].up == -1]
    assert len(roots) == 1
    edges = 0
    for r, t in enumerate(tr):
        kids = [d for d in t.down if d != -1]
        # compacted: the present children come first
        assert t.down[:len(kids)] == kids
        assert len(set(kids)) == len(kids)
        for c in kids:
            assert tr[c].up == r
        if t.up != -1:
            assert r in tr[t.up].down
            edges += 1
        assert len(kids) <= (2 if t.up == -1 else 3)
    assert edges == R - 1
    topology.exact_depth(tr)          # raises on a cycle; every walk reaches the root


@pytest.mark.parametrize("L", [1, 2, 4, 8])
def test_tree_invariants(L):
    # [Course13] "从 GRAPH 日志复原 active tree": parent/child agree both ways,
    # one root, N-1 edges, no cycle, every rank reaches the root; root fan-out
    # <= NCCL_MAX_TREE_ARITY_TOP = 2, others <= NCCL_MAX_TREE_ARITY = 3.
    for n in range(1, 64 // L + 1):
        R = n * L
        ch = topology.build_dtree(n, L, 2)
        for tr in ch:
            _check_invariants(tr, R)
            assert all(t.depth == L - 1 + topology.log2i(n) for t in tr)
        if n % 2 == 0:
            node_int = [{r // L for r in topology.internal_nodes(tr) if r % L == 0 and
                         any(d != -1 and d % L == 0 and d // L != r // L for d in tr[r].down)}
                        for tr in ch]
            assert not (node_int[0] & node_int[1])


def test_log2i_is_floor():
    # the depth field's floor(log2 nNodes): hand values, and the bit length
    # of n minus one for every n up to 4096
    assert [topology.log2i(n) for n in (1, 2, 3, 4, 5, 7, 8, 9, 1023, 1024, 1025)] == \
        [0, 1, 1, 2, 2, 2, 3, 3, 9, 10, 10]
    assert all(topology.log2i(n) == n.bit_length() - 1 for n in range(1, 4097))
    # R = 6 as 3 nodes x 2 ranks: depth 2 - 1 + floor(log2 3) = 2
    assert {t.depth for t in topology.build_dtree(3, 2, 1)[0]} == {2}


def test_channel_to_tree_split():
    for nch in range(1, 25):
        idx = [topology.channel_tree_index(c, nch) for c in range(nch)]
        assert idx == [0] * ((nch + 1) // 2) + [1] * (nch // 2)


def test_ring_topology():
    nxt, prv = topology.build_ring(5, 3)
    for c in range(3):
        assert nxt[c] == [1, 2, 3, 4, 0] and prv[c] == [4, 0, 1, 2, 3]


# ----------------------------------------------------------------- partition
def test_partition_small_ring_case():
    # R=4, 1024 fp32, 1 channel, chunk = count/R: 4 blocks of 256
    (cs, cn), = partition.channel_ranges(1024, 4, 1)
    loops = partition.ring_blocks(cs, cn, 4, 256)
    assert loops == [[(0, 256), (256, 256), (512, 256), (768, 256)]]


def test_partition_covers_message():
    rng = np.random.default_rng(0)
    for _ in range(200):
        count = int(rng.integers(0, 5000))
        E = int(rng.choice([2, 4]))
        nch = int(rng.integers(1, 13))
        R = int(rng.integers(1, 9))
        C = int(rng.integers(1, 40)) * (16 // E)
        seen = np.zeros(count, int)
        for (cs, cn) in partition.channel_ranges(count, E, nch):
            assert cs % (16 // E) == 0 or cn == 0
            for loop in partition.ring_blocks(cs, cn, R, C):
                assert len(loop) == R
                sizes = [n for _, n in loop]
                assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)
                for s, n in loop:
                    seen[s:s + n] += 1
        assert (seen == 1).all()


# ------------------------------------------------------------------ numerics
def test_chain_fold_order():
    # [Course13] "每种 rank 的操作": on the chain 0->1->2->3 rank 2 adds input3,
    # rank 1 adds partial(2+3), rank 0 adds partial(1+2+3): x0 + (x1 + (x2 + x3)).
    # By hand in fp32: x2 + x3 = 2**24 + 1 -> 2**24 (tie to even); + x1 -> 2**24;
    # + x0 = -2**24 -> 0.  (Left to right in rank order would give 2.)
    xs = [np.array([v], np.float32) for v in (-2.0 ** 24, 1.0, 1.0, 2.0 ** 24)]
    out = oracle.allreduce(xs, F32, SUM, TREE, 1, 16, local_ranks=4)
    assert [o[0] for o in out] == [0.0] * 4


def test_tree_local_first_then_children_in_slot_order():
    # Reading: a rank folds its local input first, then its children's partials
    # in down[] order.  Tree 0 of 4 nodes is 0 -> 2 -> {1, 3}; x = (0, 1,
    # 2**24 + 2, -1).  Above 2**24 fp32 steps by 2 and ties go to the even
    # significand.  By hand, P(2) = (x2 + x1) + x3:
    # 2**24 + 3 -> 2**24 + 4, then 2**24 + 3 -> 2**24 + 4; P(0) = 0 + P(2).
    # Children in reverse slot order, (x2 + x3) + x1: 2**24 + 1 -> 2**24, then
    # 2**24 + 1 -> 2**24.  Children first, (x1 + x3) + x2: 2**24 + 2.
    xs = [np.array([v], np.float32) for v in (0.0, 1.0, 2.0 ** 24 + 2, -1.0)]
    out = oracle.allreduce(xs, F32, SUM, TREE, 1, 16)
    assert [o[0] for o in out] == [2.0 ** 24 + 4] * 4


def test_ring_fold_starts_at_block_owner():
    # [Interview] simulation: block j leaves rank j first and is added to by
    # j+1, j+2, ... in turn.  With one element per block (R=3, 3 elements):
    # block 0: (x0 + x1) + x2, block 1: (x1 + x2) + x0, block 2: (x2 + x0) + x1.
    # x = (2**24, 1, 1) per rank position -> by hand:
    # block 0: (2**24 + 1 -> 2**24) + 1 -> 2**24
    # block 1: (1 + 1) + 2**24 = 2**24 + 2
    # block 2: (1 + 2**24 -> 2**24) + 1 -> 2**24
    xs = [np.full(3, v, np.float32) for v in (2.0 ** 24, 1.0, 1.0)]
    out = oracle.allreduce(xs, F32, SUM, RING, 1, 16)
    for o in out:
        assert o.tolist() == [2.0 ** 24, 2.0 ** 24 + 2, 2.0 ** 24]


@pytest.mark.parametrize("algo", [RING, TREE])
def test_brute_force_exact_small_integers(algo):
    # integers in [-8, 8]: every partial sum is exact in fp32, so every order
    # must give the fp64 sum exactly; Max must give the exact maximum
    rng = np.random.default_rng(1)
    for R, L in [(1, 1), (2, 1), (3, 1), (4, 1), (5, 1), (7, 1), (8, 1), (4, 2), (6, 3), (8, 4)]:
        for count in (0, 1, 3, 17, 250):
            xs = [rng.integers(-8, 9, count).astype(np.float32) for _ in range(R)]
            for nch, cb in [(1, 16), (3, 32), (12, 48)]:
                s = oracle.fp64_sum(xs, F32)
                for o in oracle.allreduce(xs, F32, SUM, algo, nch, cb, local_ranks=L):
                    assert np.array_equal(o.astype(np.float64), s)
                m = oracle.fp64_max(xs, F32) if count else np.zeros(0)
                for o in oracle.allreduce(xs, F32, MAX, algo, nch, cb, local_ranks=L):
                    assert np.array_equal(o.astype(np.float64), m)


@pytest.mark.parametrize("algo", [RING, TREE])
def test_each_rank_contributes_once(algo):
    # rank r holds 2**r: any fold that uses every rank exactly once gives
    # 2**R - 1, exactly, at every element
    for R, L in [(3, 1), (4, 1), (7, 1), (8, 1), (12, 1), (12, 4), (16, 2), (20, 1)]:
        xs = [np.full(101, 2.0 ** r, np.float32) for r in range(R)]
        for o in oracle.allreduce(xs, F32, SUM, algo, 5, 32, local_ranks=L):
            assert (o == 2.0 ** R - 1).all()
    for R in (2, 5, 9):
        xs = [np.full(R * 7, 2.0 ** r, np.float32) for r in range(R)]
        for o in oracle.reduce_scatter(xs, F32, SUM):
            assert (o == 2.0 ** R - 1).all()


def test_reduce_scatter_blocks_and_order():
    # rank r keeps block r; block b folds b+1, ..., b.  R=3, one element per
    # block, x = (2**24, 1, 1) by rank -> by hand:
    # block 0 (rank 0): (x1 + x2) + x0 = 2 + 2**24
    # block 1 (rank 1): (x2 + x0) + x1 = 2**24
    # block 2 (rank 2): (x0 + x1) + x2 = 2**24
    xs = [np.full(3, v, np.float32) for v in (2.0 ** 24, 1.0, 1.0)]
    out = oracle.reduce_scatter(xs, F32, SUM)
    assert [o.tolist() for o in out] == [[2.0 ** 24 + 2], [2.0 ** 24], [2.0 ** 24]]


def test_allgather_is_concatenation():
    rng = np.random.default_rng(2)
    for R in (1, 2, 3, 8):
        xs = [rng.integers(0, 65535, 11).astype(np.uint16) for _ in range(R)]
        cnt = schedules.Counters(R)
        out = oracle.allgather(xs, cnt)
        for o in out:
            assert np.array_equal(o, np.concatenate(xs))
        assert cnt.sent == [(R - 1) * 11] * R


def test_reduce_scatter_then_allgather_is_allreduce():
    # [Interview] "先弄清楚": reduce-scatter then all-gather is all-reduce
    rng = np.random.default_rng(3)
    R, rc = 5, 13
    xs = [rng.integers(-8, 9, R * rc).astype(np.float32) for _ in range(R)]
    ag = oracle.allgather(oracle.reduce_scatter(xs, F32, SUM))
    ar = oracle.allreduce(xs, F32, SUM, RING, 1, 16 * 64)
    for a, b in zip(ag, ar):
        assert np.array_equal(a, b)


def test_tree_sends_at_most_2S_per_rank_even_mirror():
    # [Interview] "推导": tree sends ~ 2S per card; with two complementary
    # trees each carrying half the data no rank exceeds 2S for even counts
    for n in (2, 4, 8, 16, 32, 64):
        S = 64
        xs = [np.ones(S, np.float32) for _ in range(n)]
        cnt = schedules.Counters(n)
        oracle.allreduce(xs, F32, SUM, TREE, 2, 16 * 64, counters=cnt)
        assert max(cnt.sent) <= 2 * S
        assert sum(cnt.sent) == 2 * (n - 1) * S


# --------------------------------------------------------------- converters
def _edge_bits():
    specials = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9,
                2.0 ** -24, 2.0 ** -25, 1.5 * 2.0 ** -25, 2.0 ** -14, 2.0 ** -15 * 3,
                np.inf, -np.inf, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 3.4e38, 1e-40]
    return np.array(specials, np.float32)


def test_f16_rne_matches_numpy_and_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    bits = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    x = np.concatenate([x, _edge_bits(), rng.standard_normal(50000).astype(np.float32)])
    ours = numerics.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        assert np.array_equal(ours, x.astype(np.float16).view(np.uint16))
    assert np.array_equal(ours, torch.from_numpy(x).half().view(torch.int16).numpy().view(np.uint16))
    every = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    every = every[~np.isnan(every.view(np.float16))]
    assert np.array_equal(numerics.f16_bits_to_f32(every), every.view(np.float16).astype(np.float32))


def test_bf16_rne_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    x = np.concatenate([x, _edge_bits(), rng.standard_normal(50000).astype(np.float32)])
    ours = numerics.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    every = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    back = torch.from_numpy(every.view(np.int16)).view(torch.bfloat16).float().numpy()
    ok = ~np.isnan(back)
    assert np.array_equal(numerics.bf16_bits_to_f32(every)[ok], back[ok])


def test_max_total_order_on_signed_zero():
    a = np.array([0.0, -0.0, -0.0, 0.0, 1.0, -2.0], np.float32)
    b = np.array([-0.0, 0.0, -0.0, 0.0, -1.0, -1.0], np.float32)
    for x, y in ((a, b), (b, a)):
        m = numerics.combine(MAX, x, y)
        assert m.tolist() == [0.0, 0.0, -0.0, 0.0, 1.0, -1.0]
        assert np.signbit(m).tolist() == [False, False, True, False, False, True]


# -------------------------------------------------------- fp64 and samplers
@pytest.mark.parametrize("dtype", [F32, F16, BF16])
@pytest.mark.parametrize("algo", [RING, TREE])
def test_within_fp64_bounds(dtype, algo):
    rng = np.random.default_rng(6)
    for R, L in [(2, 1), (7, 1), (8, 1), (16, 4)]:
        f = rng.standard_normal((R, 999)).astype(np.float32)
        raws = [numerics.from_f32(f[r], dtype) for r in range(R)]
        out = oracle.allreduce(raws, dtype, SUM, algo, 3, 64, local_ranks=L)
        s = oracle.fp64_sum(raws, dtype)
        a = sum(np.abs(numerics.to_f32(x, dtype).astype(np.float64)) for x in raws)
        for o in out:
            check_against_fp64(numerics.to_f32(o, dtype), s, a, R, dtype)


def test_fp64_sum_exact_where_fp64_is():
    # By hand: 2**24 + 1 - 2**24 is 1 (fp32 partials would round it to 0).
    xs = [np.array([v], np.float32) for v in (2.0 ** 24, 1.0, -2.0 ** 24)]
    assert oracle.fp64_sum(xs, F32).tolist() == [1.0]
    # fp32 values with exponents in [-10, 10]: the grid is 2**-33 and up to 64
    # of them sum below 2**17, so every partial fits in 53 bits and the fp64
    # sum in any order is the exact sum, which math.fsum returns.
    import math
    rng = np.random.default_rng(12)
    for R in (2, 7, 64):
        m = rng.uniform(1, 2, (R, 40)) * np.exp2(rng.integers(-10, 11, (R, 40)))
        f = (m * rng.choice([-1.0, 1.0], (R, 40))).astype(np.float32)
        got = oracle.fp64_sum([f[r] for r in range(R)], F32)
        want = [math.fsum(float(v) for v in f[:, e]) for e in range(40)]
        assert got.tolist() == want
    # widened 16-bit inputs: Max is the plain maximum of the decoded values
    for dtype in (F16, BF16):
        raws = [numerics.from_f32(rng.standard_normal(40).astype(np.float32), dtype)
                for _ in range(5)]
        dec = [numerics.to_f32(x, dtype).astype(np.float64) for x in raws]
        assert oracle.fp64_max(raws, dtype).tolist() == [max(v[e] for v in dec) for e in range(40)]


@pytest.mark.parametrize("algo", [RING, TREE])
def test_sampler_matches_literal_simulation(algo):
    rng = np.random.default_rng(7)
    for R, L, count, nch, cb in [(4, 1, 1024, 1, 1024), (8, 1, 1000, 3, 48), (7, 1, 333, 2, 16),
                                 (8, 4, 257, 5, 32), (3, 1, 10, 4, 16), (16, 2, 700, 12, 64)]:
        f = rng.standard_normal((R, count)).astype(np.float32)
        xs = [f[r] for r in range(R)]
        out = oracle.allreduce(xs, F32, SUM, algo, nch, cb, local_ranks=L)
        for e in range(count):
            v = sample.allreduce_element(f[:, e], e, count, F32, SUM, algo, nch, cb, L)
            assert v.view(np.uint32) == out[0][e:e + 1].view(np.uint32)[0]
        for o in out[1:]:
            assert np.array_equal(o.view(np.uint32), out[0].view(np.uint32))


def test_reduce_scatter_sampler_matches_literal():
    rng = np.random.default_rng(8)
    for R, rc in [(2, 5), (5, 7), (8, 3)]:
        f = rng.standard_normal((R, R * rc)).astype(np.float32)
        out = oracle.reduce_scatter([f[r] for r in range(R)], F32, SUM)
        for b in range(R):
            for p in range(rc):
                v = sample.reduce_scatter_element(f[:, b * rc + p], b, SUM)
                assert v.view(np.uint32) == out[b][p:p + 1].view(np.uint32)[0]


def test_workloads_are_seeded():
    import workloads
    a = workloads.generate(3, 100, workloads.BFLOAT16, "normal", 2)
    b = workloads.generate(3, 100, workloads.BFLOAT16, "normal", 2)
    assert all(bool((x.view(__import__("torch").int16) == y.view(__import__("torch").int16)).all())
               for x, y in zip(a, b))
    assert list(itertools.chain(*[t.tolist() for t in workloads.two_rank()])) == [1.0, 2.0, 3.0, 4.0]


# ------------------------------------------------------- per-hop rounding
def test_hop_rounding_bf16_by_hand():
    # R=3, one element per block; block 0 folds ranks 0, 1, 2.  Values
    # (1, 2**-8, 2**-8) at element 0.  In fp32: (1 + 2**-8) + 2**-8 = 1 + 2**-7,
    # exactly a bf16 value.  Rounded at each hop: 1 + 2**-8 lies halfway between
    # the bf16 neighbours 1 and 1 + 2**-7 and rounds to even, 1; again 1.
    x = [np.array([1.0, 0.0, 0.0], np.float32), np.array([2.0 ** -8, 0.0, 0.0], np.float32),
         np.array([2.0 ** -8, 0.0, 0.0], np.float32)]
    raws = [numerics.f32_to_bf16_bits(v) for v in x]
    fused = oracle.allreduce(raws, BF16, SUM, RING, 1, 16)
    hop = oracle.allreduce(raws, BF16, SUM, RING, 1, 16, hop_rounding=True)
    assert numerics.bf16_bits_to_f32(fused[0])[0] == 1.0 + 2.0 ** -7
    assert numerics.bf16_bits_to_f32(hop[0])[0] == 1.0


def test_hop_rounding_is_identity_for_fp32_and_max():
    rng = np.random.default_rng(21)
    for R in (2, 5, 8):
        f = [rng.standard_normal(777).astype(np.float32) for _ in range(R)]
        a = oracle.allreduce(f, F32, SUM, RING, 3, 48)
        b = oracle.allreduce(f, F32, SUM, RING, 3, 48, hop_rounding=True)
        assert all(np.array_equal(x.view(np.uint32), y.view(np.uint32)) for x, y in zip(a, b))
        h = [numerics.f32_to_f16_bits(v) for v in f]
        a = oracle.allreduce(h, F16, MAX, RING, 3, 48)
        b = oracle.allreduce(h, F16, MAX, RING, 3, 48, hop_rounding=True)
        assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_hop_rounding_small_integers_exact():
    # integers in [-8, 8] over up to 8 ranks stay exact in bf16 and fp16
    rng = np.random.default_rng(22)
    for dtype in (F16, BF16):
        for R in (2, 3, 8):
            f = [rng.integers(-8, 9, 300).astype(np.float32) for _ in range(R)]
            raws = [numerics.from_f32(v, dtype) for v in f]
            out = oracle.allreduce(raws, dtype, SUM, RING, 2, 32, hop_rounding=True)
            s = oracle.fp64_sum(raws, dtype)
            for o in out:
                assert np.array_equal(numerics.to_f32(o, dtype).astype(np.float64), s)


# --------------------------------------------- intra orders, head patterns
def _chain_from_root(tr):
    order, v = [], topology.root_of(tr)[0]
    while v != -1:
        order.append(v)
        v = tr[v].down[0]
    return order


def test_active_trees_table(golden):
    # [Course13] "本机真实树形": one node, 12 channels, each channel's chain in
    # its intra order; root-to-leaf order, depth N-1 and fan-out 1
    rows = [r.split() for r in golden("active_trees_table.txt")]
    for N in (2, 3, 4):
        mine = [r for r in rows if int(r[0]) == N]
        orders = [None] * 12
        for _, chans, order, _, _ in mine:
            for c in chans.split(","):
                orders[int(c)] = [int(x) for x in order.split("-")]
        ch = topology.build_dtree(1, N, 12, orders=orders)
        for _, chans, order, depth, fan in mine:
            for c in chans.split(","):
                tr = ch[int(c)]
                assert "-".join(map(str, _chain_from_root(tr))) == order
                assert topology.exact_depth(tr) == int(depth)
                assert max(sum(d != -1 for d in t.down) for t in tr) == int(fan)
                _check_invariants(tr, N)


def test_split_tree_two_by_two_by_hand():
    # SPLIT_TREE: parent head = local 0, child heads = local 1.  Two nodes of
    # two ranks; node tree 0 is node 0 -> node 1 (as node 0's d1).  Node 1's
    # parent head (rank 2) goes up to node 0's child1 head (rank 1), which is
    # the end of node 0's chain: the whole tree is the chain 0-1-2-3.
    tr = topology.build_dtree(2, 2, 1, pattern="split_tree")[0]
    assert _chain_from_root(tr) == [0, 1, 2, 3]
    assert [t.up for t in tr] == [-1, 0, 1, 2]
    # TREE on the same layout hangs node 1 under rank 0 beside its chain child
    tr = topology.build_dtree(2, 2, 1, pattern="tree")[0]
    assert tr[0].down == [1, 2, -1] and tr[2].up == 0


def test_balanced_tree_four_by_two_by_hand():
    # BALANCED_TREE: child0 head = local 1, child1 head = local 0.  Node tree
    # 0 of 4 nodes: 0 -> 2 -> {1 (d0), 3 (d1)}.  Node 2 = ranks 4, 5: node 1's
    # parent head (rank 2) hangs under rank 5 (child0 head), node 3's (rank 6)
    # under rank 4 (child1 head); node 2's parent head (rank 4) hangs under
    # node 0's child1 head (rank 0), since node 2 is node 0's d1.
    tr = topology.build_dtree(4, 2, 1, pattern="balanced_tree")[0]
    assert tr[2].up == 5 and tr[6].up == 4 and tr[4].up == 0
    assert tr[5].down == [2, -1, -1] and tr[4].down == [5, 6, -1]
    assert tr[0].down == [1, 4, -1]


@pytest.mark.parametrize("pattern", ["tree", "split_tree", "balanced_tree"])
def test_pattern_invariants(pattern):
    rng = np.random.default_rng(30)
    for L in (2, 3, 4, 8):
        for n in range(1, 64 // L + 1):
            orders = [list(rng.permutation(L)) for _ in range(3)]
            for ch in (topology.build_dtree(n, L, 2, pattern=pattern),
                       topology.build_dtree(n, L, 3, pattern=pattern, orders=orders)):
                for tr in ch:
                    _check_invariants(tr, n * L)


# -------------------------------------------------------------- cost model
def test_cost_model_step_counts_and_traffic():
    from oracle import costmodel as cm
    # [Interview] Figure 2 / "推导": n = 8: ring 14 stages, tree 2 log2 8 = 6;
    # n = 1024: 2046 and about 20; ring traffic 2(n-1)/n S, 1.5 S at n = 4
    tr8 = topology.build_dtree(8, 1, 1)[0]
    assert cm.ring_terms(8, 1)[0] == 14
    assert cm.tree_terms(topology.exact_depth(tr8), 1)[0] == 6
    assert cm.ring_terms(1024, 1)[0] == 2046
    assert cm.tree_terms(topology.exact_depth(topology.build_dtree(1024, 1, 1)[0]), 1)[0] == 20
    assert cm.ring_terms(4, 64)[1] == 96.0 and cm.tree_terms(2, 64)[1] == 128.0
    # [Course13] "理想成本模型": a 4-rank chain (depth N-1 = 3) has no latency
    # advantage over the ring: 2D = 6 = 2(N-1)
    chain = topology.build_dtree(1, 4, 1)[0]
    assert cm.tree_terms(topology.exact_depth(chain), 1)[0] == cm.ring_terms(4, 1)[0]


def test_cost_model_crossover_matches_search():
    from oracle import costmodel as cm
    rng = np.random.default_rng(31)
    for _ in range(200):
        N = int(rng.integers(2, 65))
        D = int(rng.integers(1, 8))
        ring = (float(rng.uniform(0.1, 10)), float(rng.uniform(1e-6, 1e-3)))
        tree = (float(rng.uniform(0.1, 10)), float(rng.uniform(1e-6, 1e-3)))
        m = cm.crossover(N, D, ring, tree)
        grid = np.geomspace(1e-3, 1e12, 4000)
        diff = np.array([cm.t_ring(N, x, *ring) - cm.t_tree(D, x, *tree) for x in grid])
        sign_change = np.nonzero(np.sign(diff[1:]) != np.sign(diff[:-1]))[0]
        if m is None:
            assert sign_change.size == 0
        else:
            assert sign_change.size == 1
            lo, hi = grid[sign_change[0]], grid[sign_change[0] + 1]
            assert lo <= m * (1 + 1e-9) and m <= hi * (1 + 1e-9)
            # the choice flips at the crossover
            assert cm.select(N, D, m * 0.5, ring, tree) != cm.select(N, D, m * 2, ring, tree)


def test_cost_model_selects_lower_prediction_by_hand():
    # N = 4 ranks, tree depth D = 2: ring 6 alpha + 1.5 M beta, tree 4 alpha
    # + 2 M beta.  Ring (alpha 1, beta 1e-3), tree (alpha 0.5, beta 1e-3):
    # at M = 0 ring 6 vs tree 2 -> tree; at M = 1e6 ring 1506 vs tree 2002 ->
    # ring; they cross at 4 / 0.5e-3 = 8000 bytes.
    from oracle import costmodel as cm
    ring, tree = (1.0, 1e-3), (0.5, 1e-3)
    assert cm.t_ring(4, 0, *ring) == 6.0 and cm.t_tree(2, 0, *tree) == 2.0
    assert cm.select(4, 2, 0, ring, tree) == "tree"
    assert cm.select(4, 2, 1e6, ring, tree) == "ring"
    assert abs(cm.crossover(4, 2, ring, tree) - 8000.0) < 1e-6


def test_cost_model_fit_recovers_parameters():
    from oracle import costmodel as cm
    stages = [6] * 10 + [14] * 10
    traffic = list(np.geomspace(8, 1e9, 10)) * 2
    times = [cm.predict(s, b, 2.5, 3e-4) for s, b in zip(stages, traffic)]
    a, ib = cm.fit(stages, traffic, times)
    assert abs(a - 2.5) < 1e-9 and abs(ib - 3e-4) < 1e-12


def test_cost_model_relative_fit_by_hand():
    # samples (stages, traffic, t): (1, 0, 1), (0, 1, 1), (1, 1, 3).  Relative
    # rows (s/t, b/t) = (1, 0), (0, 1), (1/3, 1/3) against 1; normal equations
    # [[10/9, 1/9], [1/9, 10/9]] (a, b) = (4/3, 4/3), so a = b = 12/11.  The
    # absolute fit of the same samples gives 4/3: the weighting is the pin.
    # Samples whose time is not positive are left out.
    from oracle import costmodel as cm
    a, b = cm.fit_relative([1, 0, 1], [0, 1, 1], [1.0, 1.0, 3.0])
    assert abs(a - 12 / 11) < 1e-12 and abs(b - 12 / 11) < 1e-12
    a2, b2 = cm.fit([1, 0, 1], [0, 1, 1], [1.0, 1.0, 3.0])
    assert abs(a2 - 4 / 3) < 1e-12 and abs(b2 - 4 / 3) < 1e-12
    a3, b3 = cm.fit_relative([1, 0, 5, 1, 2], [0, 1, 5, 1, 3], [1.0, 1.0, 0.0, 3.0, -1.0])
    assert abs(a3 - 12 / 11) < 1e-12 and abs(b3 - 12 / 11) < 1e-12


def test_cost_model_relative_fit_properties():
    from oracle import costmodel as cm
    rng = np.random.default_rng(32)
    stages = list(rng.integers(2, 130, 40).astype(float))
    traffic = list(np.geomspace(8, 1e9, 40) * (1 + rng.random(40)))
    exact = [cm.predict(s, b, 0.4, 7e-7) for s, b in zip(stages, traffic)]
    a, ib = cm.fit_relative(stages, traffic, exact)           # a planted model
    assert abs(a - 0.4) < 1e-9 and abs(ib / 7e-7 - 1) < 1e-9
    noisy = [t * (1 + 0.3 * rng.standard_normal()) for t in exact]
    a, ib = cm.fit_relative(stages, traffic, noisy)
    # the relative residuals are orthogonal to both relative columns (the
    # minimum of a least-squares objective)
    r = [(a * s + ib * b - t) / t for s, b, t in zip(stages, traffic, noisy)]
    assert abs(sum(ri * s / t for ri, s, t in zip(r, stages, noisy))) < 1e-8 * len(r)
    assert abs(sum(ri * b / t for ri, b, t in zip(r, traffic, noisy))) < 1e-8 * len(r)
    # and no nearby point does better
    def obj(x, y):
        return sum(((x * s + y * b - t) / t) ** 2 for s, b, t in zip(stages, traffic, noisy))
    best = obj(a, ib)
    for da, db in ((1e-3, 0), (-1e-3, 0), (0, 1e-3), (0, -1e-3), (1e-3, 1e-3)):
        assert obj(a * (1 + da), ib * (1 + db)) > best
    # a sample scaled as a whole (stages, traffic and time by the same factor)
    # weighs the same: the fit does not change
    s2, b2, t2 = list(stages), list(traffic), list(noisy)
    s2[0], b2[0], t2[0] = s2[0] * 1000, b2[0] * 1000, t2[0] * 1000
    a2, ib2 = cm.fit_relative(s2, b2, t2)
    assert abs(a2 / a - 1) < 1e-9 and abs(ib2 / ib - 1) < 1e-9
