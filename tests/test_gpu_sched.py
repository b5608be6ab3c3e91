"""Run-time tile scheduling of the staged AllReduce kernels (VR_SCHED).

A staged AllReduce (tree or ring) may let its CTAs draw tiles from a counter
in a scheduler slot instead of taking fixed runs.  Which CTA folds a tile never
changes the tile's fold, so the results must be the oracle's bit for bit
whichever way the tiles are shared out; the slot must be free again after
every call; launches on two streams at once, and the replays of a captured
graph, must each get every tile exactly once; a slot held by something else
must end in a bounded wait and VR_ERR_TIMEOUT, not a hang.  Nothing here
faults or waits without a bound.
"""

import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import workloads  # noqa: E402
from tests.options import options  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA device", allow_module_level=True)

import double_binary_tree_gb300 as vr  # noqa: E402

F32, F16, BF16 = vr.VR_FLOAT32, vr.VR_FLOAT16, vr.VR_BFLOAT16
SUM, MAX = vr.VR_SUM, vr.VR_MAX
RING, TREE = vr.VR_ALGO_RING, vr.VR_ALGO_TREE
NCH, CB = 12, 512 * 1024
FREE = (0, 0, 0, 0)
HELD = 0xC000000000003039  # an owner no launch has (grid ids stay far below 2^62)


def expected(inputs, dtype, op, L=1, nch=NCH, cb=CB, algo=TREE):
    raws = [workloads.raw_numpy(t) for t in inputs]
    return oracle.allreduce(raws, dtype, op, algo, nch, cb, local_ranks=L)[0]


def run(src, dst, R, count, dtype, op, L=1, stream=None, nch=NCH, cb=CB, algo=TREE):
    vr.vr_allreduce_ex(src, dst, R, count, dtype, op, algo, nch, cb, L, stream)


def same_everywhere(dst):
    v = dst[0].view(torch.int16 if dst[0].element_size() == 2 else torch.int32)
    for d in dst[1:]:
        assert torch.equal(d.view(v.dtype), v)


def assert_exact(dst, want):
    same_everywhere(dst)
    assert np.array_equal(workloads.raw_numpy(dst[0]), want)


# Staged-kernel sizes: 32 MiB per rank for 4-7 ranks (their staged
# threshold), 16 MiB above; trees that draw their tiles start at 24 MiB
# (5-7 ranks) and 8 MiB (9 and more).
FULL = [
    (4, 8 << 20, F32, SUM, 1, "normal"),
    (6, 6 << 20, F32, SUM, 1, "normal"),      # 24 MiB: staged only when drawn
    (12, 4 << 20, BF16, SUM, 1, "normal"),    # 8 MiB: staged only when drawn
    (12, 4 << 20, F32, MAX, 1, "normal"),     # 16 MiB: fp32 rings of 9-15 ranks draw
    (5, 16 << 20, BF16, SUM, 1, "normal"),
    (7, 8 << 20, F32, MAX, 1, "normal"),
    (16, 8 << 20, F16, SUM, 1, "uniform"),
    (33, 8 << 20, F16, SUM, 1, "uniform"),
    (63, 8 << 20, F16, MAX, 9, "uniform"),
]


@pytest.mark.parametrize("algo", [TREE, RING])
@pytest.mark.parametrize("R,count,dtype,op,L,dist", FULL)
def test_drawn_tiles_are_the_oracle_and_the_fixed_split(R, count, dtype, op, L, dist, algo):
    inp = workloads.generate(R, count, dtype, dist, 700 + R)
    src = [t.cuda() for t in inp]
    dst = [torch.empty_like(s) for s in src]
    stream = torch.cuda.current_stream()
    want = expected(inp, dtype, op, L, algo=algo)
    for sched in (2, 0):
        with options(vr, VR_SCHED=sched):
            for d in dst:
                d.zero_()
            run(src, dst, R, count, dtype, op, L, algo=algo)
            assert vr.vr_stream_status(stream) == vr.VR_SUCCESS
            assert_exact(dst, want)
    assert vr.vr_debug_sched_slot(stream) == FREE


# Small and ragged messages on the staged kernel (forced), tiles drawn: a
# few tiles for many CTAs, trailing partial units, one tile.
SMALL = [(3, 1000), (4, 4093), (7, 65536 + 5), (16, 3 * 4096 + 1), (33, 777), (64, 8192 + 3)]


@pytest.mark.parametrize("algo", [TREE, RING])
@pytest.mark.parametrize("R,count", SMALL)
@pytest.mark.parametrize("dtype", [F32, BF16])
def test_drawn_tiles_small_and_ragged(R, count, dtype, algo):
    inp = workloads.generate(R, count, dtype, "normal", 800 + R)
    src = [t.cuda() for t in inp]
    dst = [torch.empty_like(s) for s in src]
    stream = torch.cuda.current_stream()
    with options(vr, VR_KERNEL_PATH="staged", VR_SCHED=2):
        run(src, dst, R, count, dtype, SUM, nch=2, cb=4096, algo=algo)
        assert vr.vr_stream_status(stream) == vr.VR_SUCCESS
    assert_exact(dst, expected(inp, dtype, SUM, nch=2, cb=4096, algo=algo))
    assert vr.vr_debug_sched_slot(stream) == FREE


@pytest.mark.parametrize("R,count,cb", [(16, (4 << 20) + 7, 4096), (5, (8 << 20) + 3, 1040)])
def test_drawn_ring_tiles_across_many_blocks(R, count, cb):
    """Ring blocks much smaller than a tile (small chunks): every drawn tile
    crosses ring blocks and loops, and the consumers step through them from
    the producer's mark."""
    inp = workloads.generate(R, count, F32, "normal", 850 + R)
    src = [t.cuda() for t in inp]
    dst = [torch.empty_like(s) for s in src]
    stream = torch.cuda.current_stream()
    with options(vr, VR_KERNEL_PATH="staged", VR_SCHED=2):
        run(src, dst, R, count, F32, SUM, nch=3, cb=cb, algo=RING)
        assert vr.vr_stream_status(stream) == vr.VR_SUCCESS
    assert_exact(dst, expected(inp, F32, SUM, nch=3, cb=cb, algo=RING))
    assert vr.vr_debug_sched_slot(stream) == FREE


def test_two_streams_at_once_each_get_every_tile():
    R, count = 16, 8 << 20
    inps = [workloads.generate(R, count, F16, "uniform", 900 + i) for i in range(2)]
    srcs = [[t.cuda() for t in inp] for inp in inps]
    dsts = [[torch.empty_like(s) for s in src] for src in srcs]
    streams = [torch.cuda.Stream() for _ in range(2)]
    torch.cuda.synchronize()
    with options(vr, VR_SCHED=2):
        for _ in range(3):
            for src, dst, st in zip(srcs, dsts, streams):
                run(src, dst, R, count, F16, SUM, stream=st)
        for st in streams:
            assert vr.vr_stream_status(st) == vr.VR_SUCCESS
    for inp, dst, st in zip(inps, dsts, streams):
        assert_exact(dst, expected(inp, F16, SUM))
        assert vr.vr_debug_sched_slot(st) == FREE


def test_graph_replays_each_get_every_tile():
    R, count = 16, 8 << 20
    inp = workloads.generate(R, count, F16, "uniform", 950)
    src = [t.cuda() for t in inp]
    dst = [torch.empty_like(s) for s in src]
    dst2 = [torch.empty_like(s) for s in src]
    want = expected(inp, F16, SUM)
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with options(vr, VR_SCHED=2):
        with torch.cuda.stream(st):
            run(src, dst, R, count, F16, SUM, stream=st)   # warm-up (plans, kernels)
            st.synchronize()
            with torch.cuda.graph(g, stream=st):
                run(src, dst, R, count, F16, SUM, stream=st)
                run(src, dst2, R, count, F16, SUM, stream=st)
        for _ in range(3):
            for d in dst + dst2:
                d.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert vr.vr_stream_status(st) == vr.VR_SUCCESS
            assert_exact(dst, want)
            assert_exact(dst2, want)


def test_held_slot_times_out_then_recovers():
    R, count = 16, 8 << 20
    inp = workloads.generate(R, count, F16, "uniform", 960)
    src = [t.cuda() for t in inp]
    dst = [torch.empty_like(s) for s in src]
    stream = torch.cuda.current_stream()
    with options(vr, VR_SCHED=2):
        vr.vr_debug_sched_slot(stream, (HELD, 0, 0, 0))
        t0 = time.time()
        run(src, dst, R, count, F16, SUM)
        assert vr.vr_stream_status(stream) == vr.VR_ERR_TIMEOUT
        assert time.time() - t0 < 30.0
        # the held slot was left alone: nobody joined it
        assert vr.vr_debug_sched_slot(stream) == (HELD, 0, 0, 0)
        vr.vr_debug_sched_slot(stream, FREE)
        run(src, dst, R, count, F16, SUM)
        assert vr.vr_stream_status(stream) == vr.VR_SUCCESS
    assert_exact(dst, expected(inp, F16, SUM))
    assert vr.vr_debug_sched_slot(stream) == FREE


def test_slot_left_behind_is_reported_then_recovers():
    """More joins recorded than the grid has CTAs: state an incomplete
    earlier execution would leave.  Every CTA refuses it."""
    R, count = 16, 8 << 20
    inp = workloads.generate(R, count, F16, "uniform", 970)
    src = [t.cuda() for t in inp]
    dst = [torch.empty_like(s) for s in src]
    stream = torch.cuda.current_stream()
    with options(vr, VR_SCHED=2):
        vr.vr_debug_sched_slot(stream, (0, 0, 1 << 20, 0))
        run(src, dst, R, count, F16, SUM)
        assert vr.vr_stream_status(stream) == vr.VR_ERR_INTERNAL
        vr.vr_debug_sched_slot(stream, FREE)
        run(src, dst, R, count, F16, SUM)
        assert vr.vr_stream_status(stream) == vr.VR_SUCCESS
    assert_exact(dst, expected(inp, F16, SUM))
    assert vr.vr_debug_sched_slot(stream) == FREE


def test_stalled_tile_with_drawn_tiles_times_out_then_recovers():
    R, count = 16, 8 << 20
    inp = workloads.generate(R, count, F16, "uniform", 980)
    src = [t.cuda() for t in inp]
    dst = [torch.empty_like(s) for s in src]
    stream = torch.cuda.current_stream()
    with options(vr, VR_SCHED=2):
        vr.vr_debug_stall_next(0)
        run(src, dst, R, count, F16, SUM)
        assert vr.vr_stream_status(stream) == vr.VR_ERR_TIMEOUT
        assert vr.vr_debug_sched_slot(stream) == FREE   # every CTA still left
        run(src, dst, R, count, F16, SUM)
        assert vr.vr_stream_status(stream) == vr.VR_SUCCESS
    assert_exact(dst, expected(inp, F16, SUM))
