"""Host-side checks of libvr.so that need no GPU: the library loads and
exports every entry point of include/vr.h; its topology and partition
outputs equal the oracle's bit for bit; argument errors are reported
synchronously, before anything touches the GPU.

Every collective call below is rejected by validation (or is a count == 0
no-op), so the fake pointers are never dereferenced or launched on.
"""

import ctypes
import os
import re

import numpy as np
import pytest

from oracle import partition as opart, sample as osample, topology as otopo
from tests.conftest import ROOT

import double_binary_tree_gb300 as vr


def test_exports_every_declared_symbol():
    header = open(os.path.join(ROOT, "include", "vr.h"), encoding="utf-8").read()
    declared = set(re.findall(r"^[a-z_ *]+?\b(vr_[a-z_]+)\(", header, flags=re.M))
    assert {"vr_allreduce", "vr_reduce_scatter", "vr_allgather", "vr_build_ring",
            "vr_build_dtree"} <= declared
    lib = ctypes.CDLL(vr.library_path())
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(vr.EXPORTED)


def test_every_option_is_documented_and_settable():
    """The option table of the library (options.cc) and the header's option
    list name the same switches, and each can be read through the API."""
    src = open(os.path.join(ROOT, "double_binary_tree_gb300", "csrc", "options.cc"),
               encoding="utf-8").read()
    table = src[src.index("kSpecs[kOptCount] = {"):]
    table = table[:table.index("};")]
    names = re.findall(r'"(VR_[A-Z_]+)"', table)
    assert len(names) == len(set(names)) >= 16
    header = open(os.path.join(ROOT, "include", "vr.h"), encoding="utf-8").read()
    for name in names:
        assert name in header, name
        vr.vr_get_option(name)


@pytest.mark.parametrize("nch", [1, 2, 12, 24, 64])
def test_ring_matches_oracle(nch):
    for R in range(1, 65):
        nxt, prv = vr.vr_build_ring(R, nch)
        onx, opv = otopo.build_ring(R, nch)
        assert nxt == [x for row in onx for x in row]
        assert prv == [x for row in opv for x in row]


@pytest.mark.parametrize("L", [1, 2, 3, 4, 8, 16])
def test_dtree_matches_oracle(L):
    for n in range(1, 64 // L + 1):
        for nch in (1, 2, 3, 12):
            got = vr.vr_build_dtree(n, L, nch)
            want = otopo.build_dtree(n, L, nch)
            R = n * L
            for c in range(nch):
                for r in range(R):
                    g, w = got[c * R + r], want[c][r]
                    assert (g.depth, g.up, list(g.down)) == (w.depth, w.up, w.down), (n, L, c, r)


def test_partition_matches_oracle():
    rng = np.random.default_rng(11)
    cases = [(0, 4, 1), (1, 4, 12), (1024, 4, 1), (16 * 2 ** 20, 4, 12), (8 * 2 ** 20, 2, 12),
             (2 * 2 ** 20 + 5, 2, 2), (7, 2, 64)]
    cases += [(int(rng.integers(0, 10 ** 7)), int(rng.choice([2, 4])), int(rng.integers(1, 65)))
              for _ in range(50)]
    for count, E, nch in cases:
        dtype = vr.VR_FLOAT32 if E == 4 else vr.VR_FLOAT16
        want = opart.channel_ranges(count, E, nch)
        for c in range(nch):
            assert vr.vr_partition(count, dtype, nch, c) == want[c]


def test_ring_block_matches_oracle():
    rng = np.random.default_rng(12)
    for _ in range(60):
        count = int(rng.integers(1, 5000))
        E = int(rng.choice([2, 4]))
        dtype = vr.VR_FLOAT32 if E == 4 else vr.VR_BFLOAT16
        R = int(rng.integers(1, 65))
        nch = int(rng.integers(1, 13))
        cb = 16 * int(rng.integers(1, 20))
        for e in rng.integers(0, count, 10):
            e = int(e)
            k, j = vr.vr_ring_block(count, dtype, R, nch, cb, e)
            assert j == osample.ring_fold_start(e, count, E, R, nch, cb // E)
            assert k == osample.channel_of(e, count, E, nch)


def _err(fn, *a):
    with pytest.raises(vr.VrError) as ei:
        fn(*a)
    return ei.value.code


FAKE = [0x100000 * (i + 1) for i in range(64)]        # never dereferenced
FAKE_R = [0x8000000 + 0x100000 * (i + 1) for i in range(64)]


def test_argument_errors_are_synchronous():
    INV, UNS = vr.VR_ERR_INVALID_ARGUMENT, vr.VR_ERR_UNSUPPORTED
    F32, SUM, RING, TREE = vr.VR_FLOAT32, vr.VR_SUM, vr.VR_ALGO_RING, vr.VR_ALGO_TREE
    ar = vr.vr_allreduce
    before = vr.vr_launch_count()
    assert _err(ar, FAKE[:0], FAKE_R[:0], 0, 16, F32, SUM, RING, 1, 16) == INV
    assert _err(ar, FAKE, FAKE_R, 65, 16, F32, SUM, RING, 1, 16) == INV
    assert _err(ar, FAKE[:4], FAKE_R[:4], 4, 16, F32, SUM, RING, 0, 16) == INV
    assert _err(ar, FAKE[:4], FAKE_R[:4], 4, 16, F32, SUM, RING, 65, 16) == INV
    assert _err(ar, FAKE[:4], FAKE_R[:4], 4, 16, F32, SUM, RING, 1, 0) == INV
    assert _err(ar, FAKE[:4], FAKE_R[:4], 4, 16, F32, SUM, RING, 1, 8) == INV
    assert _err(ar, FAKE[:4], FAKE_R[:4], 4, 16, 7, SUM, RING, 1, 16) == INV
    assert _err(ar, FAKE[:4], FAKE_R[:4], 4, 16, F32, 9, RING, 1, 16) == INV
    assert _err(ar, FAKE[:4], FAKE_R[:4], 4, 16, F32, SUM, 5, 1, 16) == INV
    assert _err(ar, None, FAKE_R[:4], 4, 16, F32, SUM, RING, 1, 16) == INV
    assert _err(ar, FAKE[:3] + [0], FAKE_R[:4], 4, 16, F32, SUM, RING, 1, 16) == INV
    # recv buffers of two ranks overlap
    assert _err(ar, FAKE[:2], [FAKE_R[0], FAKE_R[0] + 8], 2, 4, F32, SUM, RING, 1, 16) == INV
    # a recv buffer overlaps another rank's send buffer
    assert _err(ar, FAKE[:2], [FAKE[1] + 4, FAKE_R[1]], 2, 4, F32, SUM, RING, 1, 16) == INV
    # buffers must be aligned to the element size
    assert _err(ar, [FAKE[0] + 2, FAKE[1]], FAKE_R[:2], 2, 4, F32, SUM, RING, 1, 16) == INV
    assert _err(ar, FAKE[:2], [FAKE_R[0], FAKE_R[1] + 1], 2, 4, vr.VR_FLOAT16, SUM, RING, 1,
                16) == INV
    assert _err(vr.vr_allgather, FAKE[:2], [FAKE_R[0] + 2, FAKE_R[1]], 2, 4, F32, RING, 1,
                16) == INV
    # partial overlap with the own send buffer (in place must be exact)
    assert _err(ar, FAKE[:2], [FAKE[0] + 4, FAKE_R[1]], 2, 4, F32, SUM, RING, 1, 16) == INV
    assert _err(vr.vr_allreduce_ex, FAKE[:8], FAKE_R[:8], 8, 16, F32, SUM, TREE, 1, 16, 3) == INV
    assert _err(vr.vr_allreduce_ex, FAKE[:8], FAKE_R[:8], 8, 16, F32, SUM, TREE, 1, 16, 0) == INV
    # AUTO resolves only for valid arguments, and is AllReduce-only
    AUTO = vr.VR_ALGO_AUTO
    assert _err(vr.vr_allreduce_ex, FAKE[:8], FAKE_R[:8], 8, 16, F32, SUM, AUTO, 1, 16, 3) == INV
    assert _err(ar, FAKE[:4], FAKE_R[:4], 4, 16, F32, SUM, AUTO, 0, 16) == INV
    assert _err(ar, FAKE[:3] + [0], FAKE_R[:4], 4, 16, F32, SUM, AUTO, 1, 16) == INV
    assert _err(vr.vr_reduce_scatter, FAKE[:4], FAKE_R[:4], 4, 16, F32, SUM, AUTO, 1, 16) == INV
    # tree is AllReduce-only
    assert _err(vr.vr_reduce_scatter, FAKE[:4], FAKE_R[:4], 4, 16, F32, SUM, TREE, 1, 16) == UNS
    assert _err(vr.vr_allgather, FAKE[:4], FAKE_R[:4], 4, 16, F32, TREE, 1, 16) == UNS
    # ReduceScatter in place must sit at block r; AllGather in place at block r
    assert _err(vr.vr_reduce_scatter, FAKE[:2], [FAKE[0] + 4, FAKE_R[1]], 2, 4, F32, SUM, RING,
                1, 16) == INV
    assert _err(vr.vr_allgather, [FAKE_R[0] + 8, FAKE[1]], FAKE_R[:2], 2, 4, F32, RING, 1,
                16) == INV
    # count == 0 enqueues nothing
    vr.vr_allreduce(FAKE[:4], FAKE_R[:4], 4, 0, F32, SUM, RING, 1, 16)
    vr.vr_reduce_scatter(FAKE[:4], FAKE_R[:4], 4, 0, F32, SUM, RING, 1, 16)
    vr.vr_allgather(FAKE[:4], FAKE_R[:4], 4, 0, F32, RING, 1, 16)
    vr.vr_allreduce(FAKE[:4], FAKE_R[:4], 4, 0, F32, SUM, AUTO, 1, 16)
    assert vr.vr_launch_count() == before


def test_topology_argument_errors():
    INV = vr.VR_ERR_INVALID_ARGUMENT
    assert _err(vr.vr_build_ring, 0, 1) == INV
    assert _err(vr.vr_build_ring, 65, 1) == INV
    assert _err(vr.vr_build_ring, 4, 0) == INV
    assert _err(vr.vr_build_dtree, 0, 1, 1) == INV
    assert _err(vr.vr_build_dtree, 9, 8, 1) == INV      # 72 ranks
    assert _err(vr.vr_build_dtree, 4, 1, 65) == INV
    assert _err(vr.vr_partition, 10, 4, 1, 0) == INV     # bad dtype
    assert _err(vr.vr_partition, 10, vr.VR_FLOAT32, 2, 2) == INV
    assert _err(vr.vr_ring_block, 10, vr.VR_FLOAT32, 4, 1, 16, 10) == INV
    assert vr.vr_get_error_string(4) == "device-side wait timed out"
    assert vr.vr_get_error_string(99) == "unknown result"


def test_fold_programs_fit_the_register_stack():
    """Every tree the library can build folds with at most 8 live partials:
    all valid AllReduce arguments plan without an internal error (checked
    through the public call with count == 0 first, then with a fake
    pointer set that validation rejects only for the buffer overlap)."""
    F32 = vr.VR_FLOAT32
    for L in (1, 2, 4, 8, 16, 32, 64):
        for n in range(1, 64 // L + 1):
            tr = otopo.build_dtree(n, L, 2)
            for t in tr:
                depth = _stack_depth(t)
                assert depth <= 8, (n, L, depth)
    # planning happens after validation: count 0 returns before planning
    vr.vr_allreduce_ex(FAKE[:64], FAKE_R[:64], 64, 0, F32, vr.VR_SUM, vr.VR_ALGO_TREE, 12, 16, 8)


def _stack_depth(tree):
    """Deepest partial stack of the fold "first child, then local, then each
    further child pushed and folded" -- computed independently of the C++
    emitter, from the tree alone."""
    root = [r for r, t in enumerate(tree) if t.up == -1][0]

    def need(v):
        kids = [c for c in tree[v].down if c != -1]
        if not kids:
            return 1
        d = need(kids[0])
        for c in kids[1:]:
            d = max(d, 1 + need(c))
        return d

    return need(root)


def test_stepwise_ring_scratch_rules():
    """Scratch validation happens before anything is launched."""
    INV = vr.VR_ERR_INVALID_ARGUMENT
    F32, F16 = vr.VR_FLOAT32, vr.VR_FLOAT16
    assert vr.vr_ring_stepwise_scratch_bytes(1000, F32) == 4000
    assert vr.vr_ring_stepwise_scratch_bytes(1001, F16) == 2016
    assert vr.vr_ring_stepwise_scratch_bytes(5, 9) == 0
    before = vr.vr_launch_count()
    step = vr.vr_allreduce_ring_stepwise
    # missing, short, or overlapping scratch
    assert _err(step, FAKE[:4], FAKE_R[:4], 4, 16, F32, vr.VR_SUM, 1, 16, 0, 64) == INV
    assert _err(step, FAKE[:4], FAKE_R[:4], 4, 16, F32, vr.VR_SUM, 1, 16, 0x9000000, 63) == INV
    assert _err(step, FAKE[:4], FAKE_R[:4], 4, 16, F32, vr.VR_SUM, 1, 16, FAKE_R[2] + 8, 64) == INV
    assert _err(step, FAKE[:4], FAKE_R[:4], 4, 16, F32, vr.VR_SUM, 1, 16, FAKE[3] - 8, 64) == INV
    assert _err(step, FAKE[:4], FAKE_R[:4], 4, 16, F32, vr.VR_SUM, 1, 16, 0x9000002, 64) == INV
    # the usual argument errors
    assert _err(step, FAKE[:4], FAKE_R[:4], 4, 16, F32, 7, 1, 16, 0x9000000, 64) == INV
    assert _err(vr.vr_allreduce_tree_updown, FAKE[:8], FAKE_R[:8], 8, 16, F32, vr.VR_SUM, 1, 16,
                3) == INV
    # count == 0: nothing to do, nothing launched
    step(FAKE[:4], FAKE_R[:4], 4, 0, F32, vr.VR_SUM, 1, 16, 0, 0)
    vr.vr_allreduce_tree_updown(FAKE[:4], FAKE_R[:4], 4, 0, F32, vr.VR_SUM, 1, 16, 1)
    assert vr.vr_launch_count() == before


PATTERN_NAMES = {vr.VR_PATTERN_TREE: "tree", vr.VR_PATTERN_SPLIT_TREE: "split_tree",
                 vr.VR_PATTERN_BALANCED_TREE: "balanced_tree"}


@pytest.mark.parametrize("pattern", sorted(PATTERN_NAMES))
def test_dtree_ex_matches_oracle(pattern):
    rng = np.random.default_rng(40)
    for L in (1, 2, 3, 4, 8):
        if L == 1 and pattern != vr.VR_PATTERN_TREE:
            continue
        for n in range(1, 64 // L + 1, 3):
            for nch in (1, 2, 5):
                orders = [list(map(int, rng.permutation(L))) for _ in range(nch)]
                for o in (None, orders):
                    got = vr.vr_build_dtree_ex(n, L, nch, pattern, o)
                    want = otopo.build_dtree(n, L, nch, pattern=PATTERN_NAMES[pattern], orders=o)
                    R = n * L
                    for c in range(nch):
                        for r in range(R):
                            g, w = got[c * R + r], want[c][r]
                            assert (g.depth, g.up, list(g.down)) == (w.depth, w.up, w.down)


def test_dtree_ex_argument_errors():
    INV = vr.VR_ERR_INVALID_ARGUMENT
    assert _err(vr.vr_build_dtree_ex, 4, 1, 1, vr.VR_PATTERN_SPLIT_TREE) == INV
    assert _err(vr.vr_build_dtree_ex, 4, 2, 1, 7) == INV
    assert _err(vr.vr_build_dtree_ex, 2, 3, 1, vr.VR_PATTERN_TREE, [[0, 0, 1]]) == INV
    assert _err(vr.vr_build_dtree_ex, 2, 3, 1, vr.VR_PATTERN_TREE, [[0, 1, 3]]) == INV


def test_allreduce_trees_rejects_invalid_trees():
    INV, UNS = vr.VR_ERR_INVALID_ARGUMENT, vr.VR_ERR_UNSUPPORTED
    F32, SUM = vr.VR_FLOAT32, vr.VR_SUM
    good = vr.vr_build_dtree_ex(2, 2, 1)

    def copy(ts):
        return [vr.vr_tree_t(t.depth, t.up, (ctypes_int3)(*t.down)) for t in ts]
    import ctypes
    ctypes_int3 = ctypes.c_int * 3
    before = vr.vr_launch_count()
    bad = copy(good); bad[3].up = -1                 # two roots
    assert _err(vr.vr_allreduce_trees, FAKE[:4], FAKE_R[:4], 4, 16, F32, SUM, 1, 16, bad) == INV
    bad = copy(good); bad[0].down[2] = 3             # child whose up disagrees
    assert _err(vr.vr_allreduce_trees, FAKE[:4], FAKE_R[:4], 4, 16, F32, SUM, 1, 16, bad) == INV
    bad = copy(good); bad[1].up = 1                  # self loop
    assert _err(vr.vr_allreduce_trees, FAKE[:4], FAKE_R[:4], 4, 16, F32, SUM, 1, 16, bad) == INV
    bad = copy(good); bad[0].down[0], bad[0].down[1] = -1, bad[0].down[0]   # not compacted
    assert _err(vr.vr_allreduce_trees, FAKE[:4], FAKE_R[:4], 4, 16, F32, SUM, 1, 16, bad) == INV
    # seventeen distinct trees over seventeen channels: more than a call carries
    many = []
    for c in range(17):
        order = [(c + i) % 17 for i in range(17)]
        many += vr.vr_build_dtree_ex(1, 17, 1, vr.VR_PATTERN_TREE, [order])
    assert _err(vr.vr_allreduce_trees, FAKE[:17], FAKE_R[:17], 17, 64, F32, SUM, 17, 16,
                many) == UNS
    assert vr.vr_launch_count() == before


# ------------------------------------------------------------ cost model
from oracle import costmodel as ocost  # noqa: E402

# The library's built-in constants (fitted on GB300, 4 ranks); the oracle is
# evaluated with the same numbers so that only the formulas are compared.
BUILTIN = ((0.343939, 0.473172), (8.66964e-7, 6.13639e-7))
# Cheap tree stages, cheap ring bytes (the pages' picture: the tree for small
# messages, the ring for large ones): a crossover exists.
OTHER = ((5.0, 1.0), (1e-5, 2e-5))


def _oracle_depth(R, L):
    trees = otopo.build_dtree(R // L, L, 2)
    return max(otopo.exact_depth(trees[0]), otopo.exact_depth(trees[1]))


@pytest.mark.parametrize("R,L", [(1, 1), (2, 1), (4, 1), (7, 1), (8, 1), (16, 4), (64, 8), (48, 3)])
@pytest.mark.parametrize("model", [None, OTHER])
def test_predict_matches_oracle(R, L, model):
    (a0, a1), (b0, b1) = model or BUILTIN
    D = _oracle_depth(R, L)
    for M in (0, 8, 4096, 1 << 20, 64 << 20, 3 << 30):
        ring = vr.vr_predict_us(vr.VR_ALGO_RING, R, L, M, model)
        tree = vr.vr_predict_us(vr.VR_ALGO_TREE, R, L, M, model)
        assert ring == pytest.approx(ocost.t_ring(R, M, a0, b0), rel=1e-12, abs=1e-12)
        assert tree == pytest.approx(ocost.t_tree(D, M, a1, b1), rel=1e-12, abs=1e-12)
        want = ocost.select(R, D, M, (a0, b0), (a1, b1))
        got = vr.vr_select_algo(R, L, M, model)
        assert got == (vr.VR_ALGO_RING if want == "ring" else vr.VR_ALGO_TREE)


def test_select_switches_at_the_oracle_crossover():
    """The tree wins small messages and the ring large ones; the switch sits
    at the closed-form crossover."""
    R, L = 8, 1
    (a0, a1), (b0, b1) = OTHER
    m = ocost.crossover(R, _oracle_depth(R, L), (a0, b0), (a1, b1))
    assert m is not None and m > 0
    assert vr.vr_select_algo(R, L, int(m * 0.9), OTHER) == vr.VR_ALGO_TREE
    assert vr.vr_select_algo(R, L, int(m * 1.1), OTHER) == vr.VR_ALGO_RING


def test_set_cost_model_replaces_the_default():
    try:
        vr.vr_set_cost_model(OTHER)
        assert vr.vr_predict_us(vr.VR_ALGO_RING, 8, 1, 0) == pytest.approx(14 * 5.0)
        vr.vr_set_cost_model(None)
        assert vr.vr_predict_us(vr.VR_ALGO_RING, 8, 1, 0) == pytest.approx(14 * BUILTIN[0][0])
        for bad in (((-1.0, 0.0), (0.0, 0.0)), ((0.0, float("nan")), (0.0, 0.0)),
                    ((0.0, 0.0), (float("inf"), 0.0))):
            with pytest.raises(vr.VrError):
                vr.vr_set_cost_model(bad)
    finally:
        vr.vr_set_cost_model(None)


def test_cost_model_argument_errors():
    for args in ((vr.VR_ALGO_AUTO, 8, 1, 0), (vr.VR_ALGO_RING, 0, 1, 0),
                 (vr.VR_ALGO_RING, 65, 1, 0), (vr.VR_ALGO_TREE, 8, 3, 0),
                 (vr.VR_ALGO_TREE, 8, 0, 0)):
        with pytest.raises(vr.VrError):
            vr.vr_predict_us(*args)
    with pytest.raises(vr.VrError):
        vr.vr_select_algo(6, 4, 0)


def test_allreduce_host_argument_errors():
    """Rejected before any CUDA call: nothing is enqueued, no stream is made."""
    INV = vr.VR_ERR_INVALID_ARGUMENT
    F32, SUM, RING = vr.VR_FLOAT32, vr.VR_SUM, vr.VR_ALGO_RING
    W = [0x40000000 + 0x100000 * (i + 1) for i in range(64)]
    h = vr.vr_allreduce_host
    before = vr.vr_launch_count()
    assert _err(h, FAKE[:4], FAKE_R[:4], 4, 64, F32, SUM, RING, 1, 16, 1, W[:4], 8) == INV
    assert _err(h, FAKE[:4], FAKE_R[:4], 4, 64, F32, SUM, RING, 1, 16, 1, None, 0) == INV
    assert _err(h, FAKE[:4], FAKE_R[:4], 4, 64, F32, SUM, RING, 0, 16, 1, W[:4], 0) == INV
    assert _err(h, FAKE[:4], FAKE_R[:4], 4, 64, F32, SUM, 7, 1, 16, 1, W[:4], 0) == INV
    assert _err(h, FAKE[:4], FAKE_R[:4], 4, 64, F32, SUM, RING, 1, 16, 3, W[:4], 0) == INV
    # overlapping host buffers, overlapping workspace buffers
    assert _err(h, FAKE[:2], [FAKE_R[0], FAKE_R[0] + 8], 2, 4, F32, SUM, RING, 1, 16, 1, W[:2],
                0) == INV
    assert _err(h, FAKE[:2], FAKE_R[:2], 2, 4, F32, SUM, RING, 1, 16, 1, [W[0], W[0] + 4],
                0) == INV
    assert _err(h, FAKE[:2], FAKE_R[:2], 2, 4, F32, SUM, RING, 1, 16, 1, [W[0] + 2, W[1]],
                0) == INV
    # count == 0 enqueues nothing
    h(FAKE[:4], FAKE_R[:4], 4, 0, F32, SUM, RING, 1, 16, 1, W[:4], 0)
    assert vr.vr_launch_count() == before


# ------------------------------------------------ run-time specialised trees
@pytest.mark.parametrize("nodes,L,dtype,op", [(1, 8, vr.VR_FLOAT32, vr.VR_SUM),
                                              (7, 1, vr.VR_BFLOAT16, vr.VR_MAX),
                                              (2, 4, vr.VR_FLOAT16, vr.VR_SUM)])
def test_specialised_tree_kernels_compile_for_sm103a(nodes, L, dtype, op):
    """The generated straight-line folds compile (NVRTC, no device) with the
    kernel sources beside the library."""
    enabled, _, _ = vr.vr_jit_status()
    if not enabled:
        pytest.skip("NVRTC or the kernel sources not found")
    assert vr.vr_jit_compile_dtree(nodes, L, dtype, op, 103) > 0


def test_specialised_tree_argument_errors():
    INV = vr.VR_ERR_INVALID_ARGUMENT
    assert _err(vr.vr_jit_compile_dtree, 1, 8, 7, vr.VR_SUM, 103) == INV
    assert _err(vr.vr_jit_compile_dtree, 1, 8, vr.VR_FLOAT32, 5, 103) == INV
    assert _err(vr.vr_jit_compile_dtree, 1, 8, vr.VR_FLOAT32, vr.VR_SUM, 80) == INV
    assert _err(vr.vr_jit_compile_dtree, 0, 8, vr.VR_FLOAT32, vr.VR_SUM, 103) == INV
    assert _err(vr.vr_jit_compile_dtree, 9, 8, vr.VR_FLOAT32, vr.VR_SUM, 103) == INV


@pytest.mark.parametrize("R,L", [(4, 1), (8, 1), (16, 4), (64, 8)])
@pytest.mark.parametrize("model", [None, OTHER])
def test_crossover_matches_oracle(R, L, model):
    (a0, a1), (b0, b1) = model or BUILTIN
    want = ocost.crossover(R, _oracle_depth(R, L), (a0, b0), (a1, b1))
    got = vr.vr_crossover_bytes(R, L, model)
    if want is None:
        assert got is None
    else:
        assert got == pytest.approx(want, rel=1e-9)


def _samples(rng):
    Rs, Ls, Ms = [], [], []
    for R, L in ((4, 1), (8, 1), (16, 4), (64, 8), (7, 1)):
        for M in (8, 4096, 1 << 16, 1 << 20, 1 << 24, 1 << 28):
            Rs.append(R); Ls.append(L); Ms.append(int(M * (1 + rng.random())))
    return Rs, Ls, Ms


def test_fit_recovers_a_planted_model():
    rng = np.random.default_rng(5)
    Rs, Ls, Ms = _samples(rng)
    (a0, a1), (b0, b1) = (0.7, 1.9), (1.3e-6, 7.5e-7)
    ring = [ocost.t_ring(R, M, a0, b0) for R, M in zip(Rs, Ms)]
    tree = [ocost.t_tree(_oracle_depth(R, L), M, a1, b1) for R, L, M in zip(Rs, Ls, Ms)]
    (fa0, fa1), (fb0, fb1) = vr.vr_fit_cost_model(Rs, Ls, Ms, ring, tree)
    assert (fa0, fa1) == pytest.approx((a0, a1), rel=1e-9)
    assert (fb0, fb1) == pytest.approx((b0, b1), rel=1e-9)


def test_fit_minimises_relative_squared_error():
    """Noisy times: the library's fit equals the oracle's relative
    least-squares fit (oracle.costmodel.fit_relative) of the same samples,
    with the oracle's stage and traffic terms; samples <= 0 are left out."""
    rng = np.random.default_rng(6)
    Rs, Ls, Ms = _samples(rng)
    ring = [ocost.t_ring(R, M, 0.6, 1.2e-6) * (1 + 0.2 * rng.standard_normal())
            for R, M in zip(Rs, Ms)]
    tree = [ocost.t_tree(_oracle_depth(R, L), M, 0.8, 9e-7) * (1 + 0.2 * rng.standard_normal())
            for R, L, M in zip(Rs, Ls, Ms)]
    tree[3] = 0.0                              # left out
    ring[7] = -1.0                             # left out
    got = vr.vr_fit_cost_model(Rs, Ls, Ms, ring, tree)
    for alg, t in ((0, ring), (1, tree)):
        terms = [ocost.ring_terms(R, M) if alg == 0 else
                 ocost.tree_terms(_oracle_depth(R, L), M) for R, L, M in zip(Rs, Ls, Ms)]
        a, ib = ocost.fit_relative([x[0] for x in terms], [x[1] for x in terms], t)
        assert got[0][alg] == pytest.approx(a, rel=1e-7)
        assert got[1][alg] == pytest.approx(ib, rel=1e-7)


def test_fit_argument_errors():
    with pytest.raises(vr.VrError):
        vr.vr_fit_cost_model([8], [1], [1024], [1.0], [1.0])           # n < 2
    with pytest.raises(vr.VrError):
        vr.vr_fit_cost_model([8, 8], [1, 1], [1024, 1024], [1.0, 2.0], [1.0, 0.0])  # 1 tree sample
    with pytest.raises(vr.VrError):
        vr.vr_fit_cost_model([8, 6], [1, 4], [1024, 2048], [1.0, 2.0], [1.0, 2.0])  # 6 % 4


def test_specialised_ring_kernels_compile_for_sm103a():
    enabled, _, _ = vr.vr_jit_status()
    if not enabled:
        pytest.skip("NVRTC or the kernel sources not found")
    assert vr.vr_jit_compile_ring(4, vr.VR_FLOAT32, vr.VR_SUM, 103) > 0
    with pytest.raises(vr.VrError):
        vr.vr_jit_compile_ring(0, vr.VR_FLOAT32, vr.VR_SUM, 103)


def _brute_force_ok(kind, send, recv, sb, rb):
    """The buffer rules of include/vr.h, pair by pair."""
    def ov(a, an, b, bn):
        return an and bn and a < b + bn and b < a + an
    R = len(send)
    for r in range(R):
        for q in range(R):
            if q != r and (ov(recv[r], rb, recv[q], rb) or ov(recv[r], rb, send[q], sb)):
                return False
        inplace = {"ar": recv[r] == send[r], "rs": recv[r] == send[r] + r * rb,
                   "ag": send[r] == recv[r] + r * sb}[kind]
        if not inplace and ov(send[r], sb, recv[r], rb):
            return False
    return True


@pytest.mark.parametrize("kind", ["ar", "rs", "ag"])
def test_buffer_rules_match_brute_force(kind):
    """Random layouts in a small address space (so that overlaps are common):
    the library accepts exactly what the pairwise rules accept.  Accepted
    calls go on to look for a device and fail there with another code."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        # accepted layouts hold fake pointers: they must never reach a launch
        pytest.skip("runs only where no device can be reached")
    rng = np.random.default_rng({"ar": 1, "rs": 2, "ag": 3}[kind])
    INV = vr.VR_ERR_INVALID_ARGUMENT
    E, base = 4, 1 << 24
    seen = {True: 0, False: 0}
    for trial in range(3000):
        R = int(rng.integers(1, 9))
        n = int(rng.integers(1, 5))                  # count per rank / per block
        sb, rb = {"ar": (n * E, n * E), "rs": (R * n * E, n * E), "ag": (n * E, R * n * E)}[kind]
        span = 4 * R * max(sb, rb)
        send = [base + E * int(rng.integers(0, span // E)) for _ in range(R)]
        recv = [base + E * int(rng.integers(0, span // E)) for _ in range(R)]
        if rng.random() < 0.3:                       # plant in-place positions
            for r in range(R):
                if rng.random() < 0.7:
                    if kind == "ar":
                        recv[r] = send[r]
                    elif kind == "rs":
                        recv[r] = send[r] + r * rb
                    else:
                        send[r] = recv[r] + r * sb
        want = _brute_force_ok(kind, send, recv, sb, rb)
        if kind == "ar":
            fn = lambda: vr.vr_allreduce_ex(send, recv, R, n, vr.VR_FLOAT32, vr.VR_SUM,  # noqa: E731
                                            vr.VR_ALGO_RING, 1, 16, 1)
        elif kind == "rs":
            fn = lambda: vr.vr_reduce_scatter(send, recv, R, n, vr.VR_FLOAT32, vr.VR_SUM,  # noqa: E731
                                              vr.VR_ALGO_RING, 1, 16)
        else:
            fn = lambda: vr.vr_allgather(send, recv, R, n, vr.VR_FLOAT32,  # noqa: E731
                                         vr.VR_ALGO_RING, 1, 16)
        try:
            fn()
            code = 0
        except vr.VrError as e:
            code = e.code
        assert (code != INV) == want, (trial, R, n, send, recv)
        seen[want] += 1
    assert seen[True] > 100 and seen[False] > 100


def test_options_set_get_and_restore():
    assert vr.vr_get_option("VR_KERNEL_PATH") in (0, 1, 2)
    old = vr.vr_get_option("VR_STAGED_TILE_BYTES")
    vr.vr_set_option("VR_STAGED_TILE_BYTES", 4096)
    assert vr.vr_get_option("VR_STAGED_TILE_BYTES") == 4096
    vr.vr_set_option("VR_STAGED_TILE_BYTES", -1)      # the built-in default
    assert vr.vr_get_option("VR_STAGED_TILE_BYTES") == 0
    vr.vr_set_option("VR_STAGED_TILE_BYTES", old)
    if "VR_SCHED" not in os.environ:
        assert vr.vr_get_option("VR_SCHED") == 1          # tiles drawn where faster
    for bad in (("VR_NO_SUCH_OPTION", 1), ("VR_PDL", -2)):
        with pytest.raises(vr.VrError) as e:
            vr.vr_set_option(*bad)
        assert e.value.code == vr.VR_ERR_INVALID_ARGUMENT
    with pytest.raises(vr.VrError):
        vr.vr_get_option("VR_NO_SUCH_OPTION")


def test_options_read_from_the_environment_once():
    """A fresh process sees the environment's values at first use; changing
    the environment later has no effect (no getenv on the call path)."""
    import subprocess
    import sys
    code = (
        "import os, double_binary_tree_gb300 as vr\n"
        "a = vr.vr_get_option('VR_KERNEL_PATH'), vr.vr_get_option('VR_STAGED_STAGES'), "
        "vr.vr_get_option('VR_DEBUG')\n"
        "os.environ['VR_KERNEL_PATH'] = 'register'\n"
        "os.environ['VR_STAGED_STAGES'] = '9'\n"
        "b = vr.vr_get_option('VR_KERNEL_PATH'), vr.vr_get_option('VR_STAGED_STAGES')\n"
        "print(a, b)\n")
    env = dict(os.environ, VR_KERNEL_PATH="staged", VR_STAGED_STAGES="3", VR_DEBUG="X,GRAPH")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, check=True,
                         capture_output=True, text=True).stdout.strip()
    assert out == "(2, 3, 1) (2, 3)"


def test_byte_counts_that_overflow_are_invalid_arguments():
    """A count whose byte size does not fit a signed 64-bit offset (for
    ReduceScatter and AllGather: R blocks of it) is rejected before any
    multiplication could wrap; the fake pointers are never touched."""
    R = 4
    fake = [0x1000 * (i + 1) << 32 for i in range(R)]
    out = [0x9000 * (i + 1) << 32 for i in range(R)]
    huge = 1 << 62                       # * 4 bytes wraps a 64-bit count
    calls = [
        lambda: vr.vr_allreduce(fake, out, R, huge, vr.VR_FLOAT32, 0, 0, 1, 16),
        lambda: vr.vr_allreduce(fake, out, R, huge, vr.VR_FLOAT32, 0, vr.VR_ALGO_AUTO, 1, 16),
        lambda: vr.vr_allreduce_tree_updown(fake, out, R, huge, vr.VR_FLOAT32, 0, 1, 16, 1),
        lambda: vr.vr_reduce_scatter(fake, out, R, 1 << 60, vr.VR_FLOAT32, 0, 0, 1, 16),
        lambda: vr.vr_allgather(fake, out, R, 1 << 60, vr.VR_FLOAT32, 0, 1, 16),
        lambda: vr.vr_allreduce_ring_stepwise(fake, out, R, huge, vr.VR_FLOAT32, 0, 1, 16,
                                              0x77 << 40, 1 << 20),
        lambda: vr.vr_allreduce_ring_stepwise_noalloc(fake, out, R, huge, vr.VR_FLOAT32, 0, 1,
                                                      16),
    ]
    for i, call in enumerate(calls):
        with pytest.raises(vr.VrError) as e:
            call()
        assert e.value.code == vr.VR_ERR_INVALID_ARGUMENT, i
    assert vr.vr_ring_stepwise_scratch_bytes(huge, vr.VR_FLOAT32) == 0


def test_noalloc_checks_arguments_before_its_size_limit():
    """A call that is wrong in itself is INVALID_ARGUMENT even when it is
    also too large for the array (too large alone: UNSUPPORTED, checked on
    the GPU)."""
    big = vr.VR_NOALLOC_SCRATCH_BYTES  # elements: 4x the array in fp32
    fake = [0x1000 * (i + 1) << 32 for i in range(2)]
    for args in [([None, fake[1]], fake, 2, big, 0, 0, 1, 16),     # NULL send buffer
                 (fake, fake[:1] + [fake[0]], 2, big, 0, 0, 1, 16),  # two ranks, one buffer
                 (fake, [f + (1 << 40) for f in fake], 0, big, 0, 0, 1, 16),  # R = 0
                 (fake, [f + (1 << 40) for f in fake], 2, big, 0, 7, 1, 16),  # op
                 (fake, [f + (1 << 40) for f in fake], 2, big, 0, 0, 1, 15)]:  # chunk bytes
        with pytest.raises(vr.VrError) as e:
            vr.vr_allreduce_ring_stepwise_noalloc(*args)
        assert e.value.code == vr.VR_ERR_INVALID_ARGUMENT, args


def _graph_log(code):
    """stderr of a fresh process that runs `code` with VR_DEBUG=GRAPH."""
    import subprocess
    import sys
    env = dict(os.environ, VR_DEBUG="GRAPH")
    r = subprocess.run([sys.executable, "-c", "import double_binary_tree_gb300 as vr\n" + code],
                       cwd=ROOT, env=env, check=True, capture_output=True, text=True)
    return r.stderr.splitlines()


def test_graph_log_of_the_topology_builders(golden):
    """VR_DEBUG=GRAPH: vr_build_dtree(_ex) prints, per channel, the pages' two
    log formats for every rank, equal line for line to the oracle's
    formatting of the oracle's trees; vr_build_ring prints each channel's
    ring order.  Without the option nothing is printed."""
    lines = _graph_log("vr.vr_build_dtree(2, 4, 3)\nvr.vr_build_ring(5, 2)\n"
                       "vr.vr_build_dtree(1, 2, 1)\n"
                       "vr.vr_build_dtree_ex(1, 4, 2, 0, [[0, 2, 1, 3], [1, 0, 3, 2]])\n")
    want = []
    for c, tr in enumerate(otopo.build_dtree(2, 4, 3)):
        want += otopo.format_tree_log(tr, c, "arrow") + otopo.format_tree_log(tr, c, "bracket")
    nxt, _ = otopo.build_ring(5, 2)
    for c in range(2):
        order, v = [], 0
        for _ in range(5):
            order.append(v)
            v = nxt[c][v]
        want.append("Ring %d : %s" % (c, " ".join(map(str, order))))
    tr = otopo.build_dtree(1, 2, 1)[0]
    want += otopo.format_tree_log(tr, 0, "arrow") + otopo.format_tree_log(tr, 0, "bracket")
    for c, tr in enumerate(otopo.build_dtree(1, 4, 2, orders=[[0, 2, 1, 3], [1, 0, 3, 2]])):
        want += otopo.format_tree_log(tr, c, "arrow") + otopo.format_tree_log(tr, c, "bracket")
    assert lines == want
    # the pages' own line for the 2-rank chain
    page_line = dict(row.split(None, 1) for row in golden("active_trees.txt"))["log_line"]
    assert page_line in lines
    import subprocess
    import sys
    quiet = subprocess.run([sys.executable, "-c", "import double_binary_tree_gb300 as vr\n"
                            "vr.vr_build_dtree(2, 4, 3)\nvr.vr_build_ring(5, 2)\n"], cwd=ROOT,
                           env={k: v for k, v in os.environ.items() if k != "VR_DEBUG"},
                           check=True, capture_output=True, text=True)
    assert quiet.stderr == ""


def test_bounds_predicate_edges():
    """The bounds-checked build's predicate, run on the host: an access is
    allowed when it lies wholly inside one extent (a writable one for a
    store)."""
    A, B = 1 << 40, 1 << 41
    ext = [(A, 4096, 0), (B, 64, 1)]
    ok = vr.vr_debug_access_ok
    assert ok(ext, A, 16, False) == 1
    assert ok(ext, A + 4080, 16, False) == 1          # the last unit
    assert ok(ext, A + 4081, 16, False) == 0          # straddles the end
    assert ok(ext, A + 4096, 1, False) == 0           # one past the end
    assert ok(ext, A - 1, 1, False) == 0              # one before
    assert ok(ext, A + 4096, 0, False) == 1           # empty access at the end
    assert ok(ext, A, 16, True) == 0                  # send buffers are read-only
    assert ok(ext, B + 48, 16, True) == 1
    assert ok(ext, B + 48, 17, True) == 0
    assert ok(ext, A, 1 << 63, False) == 0            # no wrap-around
    assert ok([(None, 1 << 62, 1)], 0, 16, True) == 0  # a missing buffer matches nothing
    assert ok([], A, 1, False) == 0
    assert ok([(A, 1, 1)] * 130, A, 1, False) == -1   # more extents than a call has


def test_bounds_predicate_matches_brute_force():
    rng = np.random.default_rng(12)
    hits = 0
    for _ in range(300):
        n = int(rng.integers(1, 9))
        ext = [(int(rng.integers(1, 1 << 20)) * 16, int(rng.integers(0, 4096)),
                int(rng.integers(0, 2))) for _ in range(n)]
        a, b, _ = ext[int(rng.integers(0, n))]        # near one of the extents
        p = a + int(rng.integers(-32, b + 33))
        size = int(rng.choice([0, 1, 2, 4, 16, 4096]))
        store = bool(rng.integers(0, 2))
        want = any(p >= a and p + size <= a + b and (w or not store) for a, b, w in ext)
        assert vr.vr_debug_access_ok(ext, p, size, store) == int(want)
        hits += want
    assert 60 < hits < 240                             # both outcomes well represented


def test_bounds_checked_build_is_loaded_on_request():
    import subprocess
    import sys
    code = "import double_binary_tree_gb300 as vr; print(vr.vr_debug_bounds_checked())"
    for flag, want in (("1", "True"), ("0", "False")):
        env = dict(os.environ, VR_BOUNDS_CHECKED=flag)
        out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, check=True,
                             capture_output=True, text=True).stdout.strip()
        assert out == want


def test_bounds_checked_specialised_kernels_compile():
    """In the bounds-checked build the folds specialised at run time are
    compiled with the checks too (NVRTC, no device)."""
    import subprocess
    import sys
    if not vr.vr_jit_status()[0]:
        pytest.skip("NVRTC or the kernel sources not found")
    code = ("import double_binary_tree_gb300 as vr\n"
            "assert vr.vr_debug_bounds_checked()\n"
            "print(vr.vr_jit_compile_dtree(2, 4, vr.VR_BFLOAT16, vr.VR_SUM, 103) > 0,\n"
            "      vr.vr_jit_compile_ring(4, vr.VR_FLOAT32, vr.VR_MAX, 103) > 0)\n")
    env = dict(os.environ, VR_BOUNDS_CHECKED="1")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, check=True,
                         capture_output=True, text=True).stdout.strip()
    assert out == "True True"
