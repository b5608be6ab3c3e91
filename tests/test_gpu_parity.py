"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bar: bit-exact against the oracle's literal schedule simulation (the same
reduction order), and within the fp64 bounds of tests/tolerances.py.  Every
output buffer is surrounded by canary bytes that must survive the call.
Inputs come from workloads.py only; no expected value comes from the GPU.
"""

import itertools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import workloads  # noqa: E402
from oracle import numerics, partition, schedules, topology  # noqa: E402
from tests.options import options  # noqa: E402
from tests.tolerances import check_against_fp64  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect these
    pytest.skip("needs a CUDA device", allow_module_level=True)

import double_binary_tree_gb300 as vr  # noqa: E402

F32, F16, BF16 = vr.VR_FLOAT32, vr.VR_FLOAT16, vr.VR_BFLOAT16
SUM, MAX = vr.VR_SUM, vr.VR_MAX
RING, TREE = vr.VR_ALGO_RING, vr.VR_ALGO_TREE
TDT = workloads.TORCH_DTYPE
PAD = 64            # canary elements before and after every output
CANARY = 0x5A


@pytest.fixture(params=["register", "staged"])
def path(request):
    """Runs the test on one kernel family: the register path or the
    shared-memory-staged path (unaligned buffers always take the register
    path's element kernels)."""
    with options(vr, VR_KERNEL_PATH=request.param):
        yield request.param


class Bufs:
    """R device outputs, each inside a canary-filled allocation; `shift`
    elements of misalignment for the element-path tests."""

    def __init__(self, R, count, dtype, shift=0):
        E = vr.ELEM_SIZE[dtype]
        self.raw = [torch.full(((2 * PAD + count + shift) * E,), CANARY, dtype=torch.uint8,
                               device="cuda") for _ in range(R)]
        lo = (PAD + shift) * E
        self.views = [b[lo:lo + count * E].view(TDT[dtype]) for b in self.raw]
        self.lo, self.hi = lo, lo + count * E

    def check_canaries(self):
        for b in self.raw:
            assert bool((b[:self.lo] == CANARY).all()) and bool((b[self.hi:] == CANARY).all())


def to_device(inputs, shift=0):
    out = []
    for t in inputs:
        if shift:
            base = torch.zeros(t.numel() + shift, dtype=t.dtype, device="cuda")
            v = base[shift:]
            v.copy_(t)
            out.append(v)
        else:
            out.append(t.cuda())
    return out


@pytest.fixture(autouse=True)
def no_refused_access():
    """Under the bounds-checked build, no test's calls touched memory outside
    their buffers."""
    yield
    if vr.vr_debug_bounds_checked():
        assert vr.vr_debug_bounds_fault() == 0


def bits(t):
    return workloads.raw_numpy(t.cpu())


def assert_status_ok():
    assert vr.vr_stream_status(torch.cuda.current_stream()) == 0


def run_allreduce(inputs, dtype, op, algo, nch, cb, L=1, inplace=False, shift=0):
    R, count = len(inputs), inputs[0].numel()
    src = to_device(inputs, shift)
    if inplace:
        dst, bufs = src, None
    else:
        bufs = Bufs(R, count, dtype, shift)
        dst = bufs.views
    vr.vr_allreduce_ex(src, dst, R, count, dtype, op, algo, nch, cb, L,
                       torch.cuda.current_stream())
    assert_status_ok()
    if bufs is not None:
        bufs.check_canaries()
    return [bits(d) for d in dst]


def expect_allreduce(inputs, dtype, op, algo, nch, cb, L=1):
    raws = [workloads.raw_numpy(t) for t in inputs]
    return raws, oracle.allreduce(raws, dtype, op, algo, nch, cb, local_ranks=L)


def assert_bits_equal(got, want, what=""):
    for r, (g, w) in enumerate(zip(got, want)):
        if not np.array_equal(g, w):
            bad = np.nonzero(g != w)[0]
            raise AssertionError("%s rank %d: %d elements differ, first %s: got %r want %r" % (
                what, r, bad.size, bad[:5], g[bad[:5]], w[bad[:5]]))


# ------------------------------------------------------------ worked cases
def test_two_rank_example_ring_and_tree(path):
    inp = workloads.two_rank()
    for algo in (RING, TREE):
        got = run_allreduce(inp, F32, SUM, algo, 1, 16)
        for g in got:
            assert g.tolist() == [4.0, 6.0]


def test_small_ring_workload_exact():
    w = workloads.workload("small_ring")
    raws, want = expect_allreduce(w["inputs"], F32, SUM, RING, w["n_channels"], w["chunk_bytes"])
    got = run_allreduce(w["inputs"], F32, SUM, RING, w["n_channels"], w["chunk_bytes"])
    assert_bits_equal(got, want)
    s = oracle.fp64_sum(raws, F32)
    for g in got:
        assert np.array_equal(g.astype(np.float64), s)     # integers: exact


def test_ring_trace_bitmask(path):
    # rank r holds 2**r: every output is 2**R - 1 whatever the order
    for R in (2, 3, 4, 8, 16, 24):
        inp = workloads.generate(R, 333, F32, "pow2", 0)
        for algo in (RING, TREE):
            for g in run_allreduce(inp, F32, SUM, algo, 5, 32):
                assert (g == 2.0 ** R - 1).all()


# ------------------------------------------------- bit-exact, many shapes
RING_CASES = [
    # R, count, nch, chunk_bytes
    (1, 1000, 1, 16), (2, 1, 1, 16), (2, 3, 4, 16), (3, 17, 2, 16), (4, 1024, 1, 1024),
    (4, 4099, 12, 48), (5, 10000, 3, 16 * 7), (7, 65537, 12, 1024), (8, 100003, 12, 4096),
    (8, 262147, 12, 512 * 1024), (16, 30011, 5, 160), (64, 9001, 12, 64), (64, 70000, 64, 512),
]


@pytest.mark.parametrize("dtype", [F32, F16, BF16])
@pytest.mark.parametrize("R,count,nch,cb", RING_CASES)
def test_ring_bit_exact(R, count, nch, cb, dtype, path):
    inp = workloads.generate(R, count, dtype, "normal", 100 + R)
    _, want = expect_allreduce(inp, dtype, SUM, RING, nch, cb)
    assert_bits_equal(run_allreduce(inp, dtype, SUM, RING, nch, cb), want)


TREE_CASES = [
    # R, local ranks, count, nch, chunk_bytes
    (1, 1, 100, 1, 16), (2, 1, 7, 2, 16), (3, 1, 1001, 2, 32), (4, 1, 4099, 12, 64),
    (5, 1, 3333, 3, 16), (7, 1, 65539, 2, 1024), (8, 1, 65536, 2, 512 * 1024),
    (8, 1, 100003, 12, 4096), (16, 1, 20000, 4, 64), (64, 1, 5000, 12, 512),
    (4, 4, 3000, 2, 16), (8, 2, 7777, 3, 48), (12, 3, 4000, 2, 64), (16, 4, 9001, 12, 256),
    (64, 8, 12345, 12, 1024), (32, 8, 4096, 7, 16), (63, 7, 3000, 5, 64),
]


@pytest.mark.parametrize("dtype", [F32, F16, BF16])
@pytest.mark.parametrize("R,L,count,nch,cb", TREE_CASES)
def test_tree_bit_exact(R, L, count, nch, cb, dtype, path):
    inp = workloads.generate(R, count, dtype, "normal", 200 + R)
    _, want = expect_allreduce(inp, dtype, SUM, TREE, nch, cb, L)
    assert_bits_equal(run_allreduce(inp, dtype, SUM, TREE, nch, cb, L), want)


@pytest.mark.parametrize("algo", [RING, TREE])
@pytest.mark.parametrize("R", [3, 5, 6, 7])
def test_few_rank_geometry_at_32_mib(R, algo):
    """2-7 ranks from 32 MiB per rank take the staged kernel with the
    few-rank tile and stage table (the 6-rank ring keeps the register path):
    every element equal to the oracle, with a ragged tail."""
    count = (8 << 20) + 3
    inp = workloads.generate(R, count, F32, "normal", 170 + R)
    _, want = expect_allreduce(inp, F32, SUM, algo, 12, 512 * 1024)
    assert_bits_equal(run_allreduce(inp, F32, SUM, algo, 12, 512 * 1024), want)


@pytest.mark.parametrize("dtype", [F32, F16, BF16])
@pytest.mark.parametrize("op", [SUM, MAX])
def test_two_rank_ring_at_64_mib(dtype, op):
    """The ring of two ranks runs the tree kernels (two operands fold to the
    same bits in either order): every element equal to the oracle's ring."""
    count = (64 << 20) // vr.ELEM_SIZE[dtype] + 5
    inp = workloads.generate(2, count, dtype, "normal", 160 + dtype)
    _, want = expect_allreduce(inp, dtype, op, RING, 12, 512 * 1024)
    assert_bits_equal(run_allreduce(inp, dtype, op, RING, 12, 512 * 1024), want)


@pytest.mark.parametrize("algo", [RING, TREE])
@pytest.mark.parametrize("dtype,count", [(F32, (4 << 20) + 3), (BF16, (8 << 20) + 7)])
def test_ragged_tail_at_16_mib(algo, dtype, count):
    """16 MiB per rank plus a partial 16-byte unit (3 fp32 or 7 bf16
    elements): the default kernel choice (the staged kernel), whose trailing
    elements are folded by separate threads."""
    inp = workloads.generate(8, count, dtype, "normal", 150)
    _, want = expect_allreduce(inp, dtype, SUM, algo, 12, 512 * 1024)
    assert_bits_equal(run_allreduce(inp, dtype, SUM, algo, 12, 512 * 1024), want)


@pytest.mark.parametrize("algo", [RING, TREE])
@pytest.mark.parametrize("dtype", [F32, F16, BF16])
def test_max_exact(algo, dtype, path):
    for R, L, count in [(2, 1, 1000), (7, 1, 4097), (64, 8, 3001)]:
        inp = workloads.generate(R, count, dtype, "uniform", 300 + R)
        raws, want = expect_allreduce(inp, dtype, MAX, algo, 12, 64, L)
        got = run_allreduce(inp, dtype, MAX, algo, 12, 64, L)
        assert_bits_equal(got, want)
        m = oracle.fp64_max(raws, dtype)
        assert np.array_equal(numerics.to_f32(got[0], dtype).astype(np.float64), m)


def test_max_signed_zero_total_order(path):
    # +0 above -0, whatever the order in which they meet
    a = torch.tensor([0.0, -0.0, -0.0, -0.0, 0.0])
    b = torch.tensor([-0.0, 0.0, -0.0, -1.0, -0.0])
    c = torch.tensor([-0.0, -0.0, -0.0, -2.0, 0.0])
    for algo in (RING, TREE):
        got = run_allreduce([a, b, c], F32, MAX, algo, 1, 16)
        want = oracle.allreduce([workloads.raw_numpy(t) for t in (a, b, c)], F32, MAX, algo, 1, 16)
        for g, w in zip(got, want):
            assert g.view(np.uint32).tolist() == w.view(np.uint32).tolist()
        assert np.signbit(got[0]).tolist() == [False, False, True, True, False]


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_max_every_16bit_value(dtype, path):
    """Max on 16-bit keys, exhaustively: every non-NaN bit pattern of the type
    meets others in both halves of a 32-bit word, and every ordered triple of
    +-0, +-smallest subnormal, +-largest finite and +-inf meets in both
    halves too.  Three ranks; bit-exact to the oracle, and equal to the plain
    maximum of the decoded values."""
    allbits = np.arange(65536, dtype=np.uint16)
    keep = allbits[~np.isnan(numerics.to_f32(allbits, dtype))]
    rng = np.random.default_rng(21)
    one = numerics.from_f32(np.array([1.0], np.float32), dtype)[0]
    sub = np.uint16(1)                                   # smallest subnormal
    big = np.uint16(0x7BFF if dtype == F16 else 0x7F7F)  # largest finite
    inf = np.uint16(0x7C00 if dtype == F16 else 0x7F80)
    special = np.array([0, 0x8000, sub, sub | 0x8000, big, big | 0x8000, inf, inf | 0x8000],
                       np.uint16)
    trip = np.array(list(itertools.product(special, repeat=3)), np.uint16).T   # 3 x 512
    cols = []
    for r in range(3):
        a = np.concatenate([keep, rng.permutation(keep), np.roll(keep, r + 1)])
        cols.append(np.concatenate([a, trip[r], [one], trip[r]]))    # triples in both lanes
    inp = [torch.from_numpy(c.view(np.int16).copy()).view(TDT[dtype]) for c in cols]
    assert inp[0].numel() > 65536                        # the ring's vector kernels
    for algo in (RING, TREE):
        raws, want = expect_allreduce(inp, dtype, MAX, algo, 12, 4096)
        got = run_allreduce(inp, dtype, MAX, algo, 12, 4096)
        assert_bits_equal(got, want, "algo %d" % algo)
        dec = np.maximum.reduce([numerics.to_f32(x, dtype) for x in raws])
        zero = dec == 0
        assert np.array_equal(numerics.to_f32(got[0], dtype)[~zero], dec[~zero])


@pytest.mark.parametrize("algo", [RING, TREE])
def test_in_place(algo, path):
    for dtype in (F32, BF16):
        inp = workloads.generate(8, 50001, dtype, "normal", 400)
        _, want = expect_allreduce(inp, dtype, SUM, algo, 12, 1024)
        assert_bits_equal(run_allreduce(inp, dtype, SUM, algo, 12, 1024, inplace=True), want)


@pytest.mark.parametrize("algo", [RING, TREE])
def test_misaligned_buffers_take_element_path(algo):
    for dtype, shift in ((F32, 1), (F16, 3), (BF16, 1)):
        inp = workloads.generate(4, 3001, dtype, "normal", 500)
        _, want = expect_allreduce(inp, dtype, SUM, algo, 3, 48)
        assert_bits_equal(run_allreduce(inp, dtype, SUM, algo, 3, 48, shift=shift), want)


@pytest.mark.parametrize("dtype", [F32, F16, BF16])
def test_within_fp64_tolerance(dtype, path):
    inp = workloads.generate(8, 200003, dtype, "normal", 600)
    raws = [workloads.raw_numpy(t) for t in inp]
    s = oracle.fp64_sum(raws, dtype)
    a = sum(np.abs(numerics.to_f32(x, dtype).astype(np.float64)) for x in raws)
    for algo in (RING, TREE):
        got = run_allreduce(inp, dtype, SUM, algo, 12, 4096)
        check_against_fp64(numerics.to_f32(got[0], dtype), s, a, 8, dtype)


def test_zero_count_is_a_no_op():
    d = [torch.ones(4, device="cuda") for _ in range(2)]
    before = vr.vr_launch_count()
    vr.vr_allreduce(d, d, 2, 0, F32, SUM, RING, 1, 16)
    assert vr.vr_launch_count() == before
    assert_status_ok()


# ------------------------------------------------- ReduceScatter, AllGather
@pytest.mark.parametrize("dtype", [F32, F16, BF16])
@pytest.mark.parametrize("op", [SUM, MAX])
def test_reduce_scatter_bit_exact(dtype, op, path):
    for R, rc, inplace in [(1, 5, False), (2, 3, False), (4, 1000, False), (7, 3001, True),
                           (8, 4096, False), (64, 513, False), (64, 1024, True)]:
        inp = workloads.generate(R, R * rc, dtype, "normal", 700 + R)
        raws = [workloads.raw_numpy(t) for t in inp]
        want = oracle.reduce_scatter(raws, dtype, op)
        src = to_device(inp)
        if inplace:
            E = vr.ELEM_SIZE[dtype]
            dst = [s[r * rc:(r + 1) * rc] for r, s in enumerate(src)]
            bufs = None
        else:
            bufs = Bufs(R, rc, dtype)
            dst = bufs.views
        vr.vr_reduce_scatter(src, dst, R, rc, dtype, op, RING, 12, 512)
        assert_status_ok()
        if bufs:
            bufs.check_canaries()
        assert_bits_equal([bits(d) for d in dst], want, "rs R=%d" % R)


@pytest.mark.parametrize("order", [1, 2])
@pytest.mark.parametrize("dtype", [F32, BF16])
def test_allgather_tma_both_orders(order, dtype):
    """The TMA AllGather, source-major (1) and destination-major (2): bit
    copies equal to the oracle's, in place and out of place, ragged tiles."""
    E = vr.ELEM_SIZE[dtype]
    for R, sc, inplace in [(2, 4096, False), (8, 40960 // E, True), (5, 100000 - 100000 % 8, False),
                           (64, 8192 // E + 8, False), (3, 8, False)]:
        inp = workloads.generate(R, sc, dtype, "normal", 850 + R)
        want = oracle.allgather([workloads.raw_numpy(t) for t in inp])
        if inplace:
            outs = [torch.empty(R * sc, dtype=TDT[dtype], device="cuda") for _ in range(R)]
            for r in range(R):
                outs[r][r * sc:(r + 1) * sc].copy_(inp[r].cuda())
            src, dst, bufs = [outs[r][r * sc:(r + 1) * sc] for r in range(R)], outs, None
        else:
            src = to_device(inp)
            bufs = Bufs(R, R * sc, dtype)
            dst = bufs.views
        with options(vr, VR_AG_ORDER=order):
            vr.vr_allgather(src, dst, R, sc, dtype, RING, 12, 512)
        assert_status_ok()
        if bufs:
            bufs.check_canaries()
        assert_bits_equal([bits(d) for d in dst], want, "ag order %d R=%d" % (order, R))


@pytest.mark.parametrize("dtype", [F32, F16, BF16])
def test_allgather_exact(dtype, path):
    for R, sc, inplace, shift in [(1, 7, False, 0), (2, 1, False, 0), (3, 1001, False, 0),
                                  (8, 4096, True, 0), (64, 333, False, 0), (5, 100, False, 1)]:
        inp = workloads.generate(R, sc, dtype, "normal", 800 + R)
        want = oracle.allgather([workloads.raw_numpy(t) for t in inp])
        if inplace:
            outs = [torch.empty(R * sc, dtype=TDT[dtype], device="cuda") for _ in range(R)]
            for r in range(R):
                outs[r][r * sc:(r + 1) * sc].copy_(inp[r].cuda())
            src = [outs[r][r * sc:(r + 1) * sc] for r in range(R)]
            dst, bufs = outs, None
        else:
            src = to_device(inp, shift)
            bufs = Bufs(R, R * sc, dtype, shift)
            dst = bufs.views
        vr.vr_allgather(src, dst, R, sc, dtype, RING, 12, 512)
        assert_status_ok()
        if bufs:
            bufs.check_canaries()
        assert_bits_equal([bits(d) for d in dst], want, "ag R=%d" % R)


# ------------------------------------------------------- full-size cases
def _channel_slice_sim(raws_f32, count, E, R, nch, C, k, op):
    """Oracle literal ring simulation of channel k only (its own loops)."""
    cs, cn = partition.channel_ranges(count, E, nch)[k]
    out = np.empty(cn, np.float32)
    for loop in partition.ring_blocks(cs, cn, R, C):
        res = schedules.ring_allreduce_loop(raws_f32, loop, op)
        for (bs, bn), blk in zip(loop, res[0]):
            out[bs - cs:bs - cs + bn] = blk
    return cs, cn, out


def test_ring_64mib_fp32_full_size(path):
    """The bench workload (R=8 x 64 MiB fp32, 12 channels, 512 KiB chunks),
    every element of every rank bit-exact to the oracle's literal ring
    simulation, and within the fp64 bound."""
    w = workloads.workload("ring_64mib")
    R, count, nch, cb = w["R"], w["count"], w["n_channels"], w["chunk_bytes"]
    src = [t.cuda() for t in w["inputs"]]
    dst = [torch.empty_like(s) for s in src]
    vr.vr_allreduce(src, dst, R, count, F32, SUM, RING, nch, cb, torch.cuda.current_stream())
    assert_status_ok()
    raws = [workloads.raw_numpy(t) for t in w["inputs"]]
    want = oracle.allreduce(raws, F32, SUM, RING, nch, cb)
    got = [bits(d) for d in dst]
    assert_bits_equal(got, want, "ring_64mib")
    s = oracle.fp64_sum(raws, F32)
    a = sum(np.abs(x.astype(np.float64)) for x in raws)
    check_against_fp64(got[0], s, a, R, F32)


@pytest.mark.parametrize("name", ["tree_4mib_r8", "tree_4mib_r7"])
@pytest.mark.parametrize("nch", [2, 12])
def test_tree_4mib_bf16_full_size(name, nch, path):
    w = workloads.workload(name)
    inp = w["inputs"]
    raws, want = expect_allreduce(inp, BF16, SUM, TREE, nch, w["chunk_bytes"])
    got = run_allreduce(inp, BF16, SUM, TREE, nch, w["chunk_bytes"])
    assert_bits_equal(got, want)
    s = oracle.fp64_sum(raws, BF16)
    a = sum(np.abs(numerics.to_f32(x, BF16).astype(np.float64)) for x in raws)
    check_against_fp64(numerics.to_f32(got[0], BF16), s, a, w["R"], BF16)


@pytest.fixture(scope="module")
def hier():
    return workloads.workload("hier_16mib")


@pytest.mark.parametrize("op", [SUM, MAX])
def test_hier_16mib_fp16_tree_full_size(hier, op):
    w = hier
    R, count, nch, cb, L = w["R"], w["count"], w["n_channels"], w["chunk_bytes"], w["local_ranks"]
    src = [t.cuda() for t in w["inputs"]]
    dst = [torch.empty_like(s) for s in src]
    vr.vr_allreduce_ex(src, dst, R, count, F16, op, TREE, nch, cb, L, None)
    assert_status_ok()
    for d in dst[1:]:
        assert torch.equal(d.view(torch.int16), dst[0].view(torch.int16))
    raws = [workloads.raw_numpy(t) for t in w["inputs"]]
    xs = [numerics.to_f32(x, F16) for x in raws]
    trees = topology.build_dtree(R // L, L, nch)
    got = bits(dst[0])
    for k in range(nch):                      # every channel, whole
        cs, cn = partition.channel_ranges(count, 2, nch)[k]
        for (s, n) in partition.tree_chunks(cs, cn, cb // 2):
            res = schedules.tree_allreduce_chunk(xs, trees[k], s, n, op)
            assert np.array_equal(got[s:s + n], numerics.from_f32(res[0], F16)), (k, s)
    if op == SUM:
        s64 = oracle.fp64_sum(raws, F16)
        a = sum(np.abs(x.astype(np.float64)) for x in xs)
        check_against_fp64(numerics.to_f32(got, F16), s64, a, R, F16)
    else:
        assert np.array_equal(numerics.to_f32(got, F16).astype(np.float64),
                              oracle.fp64_max(raws, F16))


@pytest.mark.parametrize("op", [SUM, MAX])
def test_hier_16mib_fp16_ring_full_size(hier, op, path):
    w = hier
    R, count, nch, cb = w["R"], w["count"], w["n_channels"], w["chunk_bytes"]
    src = [t.cuda() for t in w["inputs"]]
    dst = [torch.empty_like(s) for s in src]
    vr.vr_allreduce(src, dst, R, count, F16, op, RING, nch, cb, None)
    assert_status_ok()
    for d in dst[1:]:
        assert torch.equal(d.view(torch.int16), dst[0].view(torch.int16))
    raws = [workloads.raw_numpy(t) for t in w["inputs"]]
    xs = [numerics.to_f32(x, F16) for x in raws]
    got = bits(dst[0])
    for k in range(nch):                      # every channel, whole
        cs, cn, want = _channel_slice_sim(xs, count, 2, R, nch, cb // 2, k, op)
        assert np.array_equal(got[cs:cs + cn], numerics.from_f32(want, F16)), k
    if op == MAX:                             # no rounding: every element exact
        assert np.array_equal(numerics.to_f32(got, F16).astype(np.float64),
                              oracle.fp64_max(raws, F16))
        return
    s64 = oracle.fp64_sum(raws, F16)
    a = sum(np.abs(x.astype(np.float64)) for x in xs)
    check_against_fp64(numerics.to_f32(got, F16), s64, a, R, F16)


def test_hier_16mib_reduce_scatter_and_allgather(hier):
    w = hier
    R, count = w["R"], w["count"]
    rc = count // R
    src = [t.cuda() for t in w["inputs"]]
    rs = [torch.empty(rc, dtype=torch.float16, device="cuda") for _ in range(R)]
    vr.vr_reduce_scatter(src, rs, R, rc, F16, SUM, RING, 12, 512 * 1024, None)
    ag = [torch.empty(count, dtype=torch.float16, device="cuda") for _ in range(R)]
    vr.vr_allgather(rs, ag, R, rc, F16, RING, 12, 512 * 1024, None)
    assert_status_ok()
    raws = [workloads.raw_numpy(t) for t in w["inputs"]]
    want_rs = oracle.reduce_scatter(raws, F16, SUM)
    assert_bits_equal([bits(t) for t in rs], want_rs, "rs")
    cat = np.concatenate(want_rs)
    for t in ag:
        assert np.array_equal(bits(t), cat)


# --------------------------------------------- caller trees: orders, patterns
@pytest.mark.parametrize("pattern", [vr.VR_PATTERN_TREE, vr.VR_PATTERN_SPLIT_TREE,
                                     vr.VR_PATTERN_BALANCED_TREE])
@pytest.mark.parametrize("dtype", [F32, BF16])
def test_allreduce_trees_patterns_and_orders(pattern, dtype, path):
    names = {0: "tree", 1: "split_tree", 2: "balanced_tree"}
    rng = np.random.default_rng(50 + pattern)
    for n, L, count, nch in [(1, 4, 30001, 12), (2, 2, 9999, 3), (4, 2, 65537, 12),
                             (8, 8, 4099, 5), (3, 3, 7777, 2)]:
        R = n * L
        pool = [list(map(int, rng.permutation(L))) for _ in range(3)]
        orders = [pool[c % 3] for c in range(nch)]   # at most 6 distinct trees
        trees = vr.vr_build_dtree_ex(n, L, nch, pattern, orders)
        inp = workloads.generate(R, count, dtype, "normal", 60 + R)
        want = oracle.allreduce([workloads.raw_numpy(t) for t in inp], dtype, SUM, TREE, nch,
                                1024, local_ranks=L, pattern=names[pattern], orders=orders)
        src = [t.cuda() for t in inp]
        bufs = Bufs(R, count, dtype)
        vr.vr_allreduce_trees(src, bufs.views, R, count, dtype, SUM, nch, 1024, trees)
        assert_status_ok()
        bufs.check_canaries()
        assert_bits_equal([bits(d) for d in bufs.views], want, "trees n=%d L=%d" % (n, L))


def test_active_trees_of_the_pages_on_gpu():
    # one node of 4 ranks, 12 channels in the three chain orders the pages
    # show ([Course13] "本机真实树形")
    per = {0: [0, 1, 2, 3], 1: [0, 1, 2, 3], 6: [0, 1, 2, 3], 7: [0, 1, 2, 3],
           2: [0, 2, 1, 3], 3: [0, 2, 1, 3], 8: [0, 2, 1, 3], 9: [0, 2, 1, 3],
           4: [1, 0, 3, 2], 5: [1, 0, 3, 2], 10: [1, 0, 3, 2], 11: [1, 0, 3, 2]}
    orders = [per[c] for c in range(12)]
    trees = vr.vr_build_dtree_ex(1, 4, 12, vr.VR_PATTERN_TREE, orders)
    inp = workloads.generate(4, 1 << 20, F32, "normal", 70)
    want = oracle.allreduce([workloads.raw_numpy(t) for t in inp], F32, SUM, TREE, 12,
                            512 * 1024, local_ranks=4, orders=orders)
    src = [t.cuda() for t in inp]
    dst = [torch.empty_like(s) for s in src]
    vr.vr_allreduce_trees(src, dst, 4, 1 << 20, F32, SUM, 12, 512 * 1024, trees)
    assert_status_ok()
    assert_bits_equal([bits(d) for d in dst], want, "active trees")


# ------------------------------------------------------- VR_ALGO_AUTO
def test_auto_runs_the_algorithm_the_oracle_cost_model_picks():
    """With a model whose crossover sits near 2.8 MB (cheap tree stages,
    cheap ring bytes), AUTO takes the tree below it and the ring above; the
    output equals the oracle of the algorithm the oracle's model selects."""
    from oracle import costmodel
    ring_m, tree_m = (5.0, 1e-5), (1.0, 2e-5)
    R = 8
    trees = topology.build_dtree(R, 1, 2)
    D = max(topology.exact_depth(trees[0]), topology.exact_depth(trees[1]))
    vr.vr_set_cost_model(((ring_m[0], tree_m[0]), (ring_m[1], tree_m[1])))
    try:
        picked = set()
        for count, seed in ((3000, 11), (1 << 20, 12)):
            inp = workloads.generate(R, count, F32, "normal", seed)
            algo = costmodel.select(R, D, count * 4, ring_m, tree_m)
            picked.add(algo)
            _, want = expect_allreduce(inp, F32, SUM, RING if algo == "ring" else TREE, 4, 1 << 16)
            got = run_allreduce(inp, F32, SUM, vr.VR_ALGO_AUTO, 4, 1 << 16)
            assert_bits_equal(got, want, "AUTO(%s)" % algo)
        assert picked == {"ring", "tree"}
    finally:
        vr.vr_set_cost_model(None)


# ------------------------------------------------ host buffers, pipelined
def _host_run(inputs, dtype, op, algo, nch, cb, L=1, piece=0, pinned=True, inplace=False,
              shift=0):
    R, count = len(inputs), inputs[0].numel()
    send = [t.clone().pin_memory() if pinned else t.clone() for t in inputs]
    recv = send if inplace else [torch.full_like(t, 7).pin_memory() if pinned
                                 else torch.full_like(t, 7) for t in inputs]
    work = [torch.empty(count + shift, dtype=t.dtype, device="cuda")[shift:] for t in inputs]
    st = torch.cuda.current_stream()
    vr.vr_allreduce_host(send, recv, R, count, dtype, op, algo, nch, cb, L, work, piece, st)
    st.synchronize()
    assert_status_ok()
    return [workloads.raw_numpy(t) for t in recv]


@pytest.mark.parametrize("dtype", [F32, F16, BF16])
@pytest.mark.parametrize("algo", [RING, TREE])
def test_allreduce_host_equals_oracle(dtype, algo, path):
    """Pieces of 48 KiB per rank (the last one ragged) over a message whose
    ring blocks and channels do not line up with them."""
    R, count = 8, 100_003 if dtype == F32 else 200_011
    inp = workloads.generate(R, count, dtype, "normal", 21)
    _, want = expect_allreduce(inp, dtype, SUM, algo, 5, 1 << 14)
    got = _host_run(inp, dtype, SUM, algo, 5, 1 << 14, piece=48 << 10)
    assert_bits_equal(got, want, "host pieces")


def test_allreduce_host_variants():
    """Default piece size, pageable memory, in place, Max, a hierarchical
    tree, an unaligned workspace (element kernels) and one piece."""
    R, count = 8, 3 * (1 << 20) + 5
    inp = workloads.generate(R, count, F32, "normal", 22)
    _, want = expect_allreduce(inp, F32, SUM, RING, 12, 1 << 19)
    assert_bits_equal(_host_run(inp, F32, SUM, RING, 12, 1 << 19), want, "default")
    assert_bits_equal(_host_run(inp, F32, SUM, RING, 12, 1 << 19, pinned=False), want, "pageable")
    assert_bits_equal(_host_run(inp, F32, SUM, RING, 12, 1 << 19, inplace=True), want, "in place")
    assert_bits_equal(_host_run(inp, F32, SUM, RING, 12, 1 << 19, piece=1 << 30), want, "1 piece")
    assert_bits_equal(_host_run(inp, F32, SUM, RING, 12, 1 << 19, piece=1 << 16, shift=1), want,
                      "unaligned workspace")
    _, want = expect_allreduce(inp, F32, MAX, TREE, 3, 1 << 16, L=4)
    assert_bits_equal(_host_run(inp, F32, MAX, TREE, 3, 1 << 16, L=4, piece=1 << 20), want,
                      "hier tree max")


def test_allreduce_host_orders_with_the_stream():
    """Work enqueued before the call is done before the copy in; work after
    it sees the copied-out result."""
    R, count = 4, 1 << 20
    st = torch.cuda.current_stream()
    dev_in = [torch.zeros(count, device="cuda") for _ in range(R)]
    send = [torch.empty(count).pin_memory() for _ in range(R)]
    recv = [torch.empty(count).pin_memory() for _ in range(R)]
    work = [torch.empty(count, device="cuda") for _ in range(R)]
    for r in range(R):
        dev_in[r].fill_(float(r + 1))
        send[r].copy_(dev_in[r], non_blocking=True)   # on the stream, before the call
    vr.vr_allreduce_host(send, recv, R, count, F32, SUM, RING, 2, 1 << 16, 1, work, 1 << 18, st)
    back = torch.empty(count, device="cuda")
    back.copy_(recv[0], non_blocking=True)            # on the stream, after the call
    st.synchronize()
    assert_status_ok()
    assert bool((back == 10.0).all())
    for r in range(R):
        assert bool((recv[r] == 10.0).all())


def test_allreduce_host_null_receive_buffers():
    """Only rank 0's result is copied out; every rank's result stays in the
    workspace, all equal to the oracle."""
    R, count = 8, (1 << 20) + 3
    inp = workloads.generate(R, count, BF16, "normal", 23)
    _, want = expect_allreduce(inp, BF16, SUM, TREE, 4, 1 << 16)
    send = [t.clone().pin_memory() for t in inp]
    out0 = torch.full_like(inp[0], 7).pin_memory()
    work = [torch.empty(count, dtype=inp[0].dtype, device="cuda") for _ in range(R)]
    st = torch.cuda.current_stream()
    vr.vr_allreduce_host(send, [out0] + [None] * (R - 1), R, count, BF16, SUM, TREE, 4, 1 << 16,
                         1, work, 1 << 18, st)
    st.synchronize()
    assert_status_ok()
    assert_bits_equal([workloads.raw_numpy(out0)], want[:1], "rank 0 copied out")
    assert_bits_equal([bits(w) for w in work], want, "workspace")


# --------------------------------------------- back-to-back dependent calls
@pytest.mark.parametrize("algo", [RING, TREE])
@pytest.mark.parametrize("R,count,dtype", [(8, 1 << 22, F32), (4, 65539, BF16), (16, 300007, F16)])
def test_in_place_chain_without_sync(algo, R, count, dtype, path):
    """Three in-place AllReduces enqueued back to back with no host sync: each
    reads what the previous one wrote (launches overlap, so every kernel must
    wait for its predecessor before touching memory)."""
    inp = workloads.generate(R, count, dtype, "uniform", 500 + R)
    raws = [workloads.raw_numpy(t) for t in inp]
    want = raws
    for _ in range(3):
        want = oracle.allreduce(want, dtype, SUM, algo, 12, 1 << 19)
    bufs = [t.cuda() for t in inp]
    st = torch.cuda.current_stream()
    for _ in range(3):
        vr.vr_allreduce(bufs, bufs, R, count, dtype, SUM, algo, 12, 1 << 19, st)
    assert_status_ok()
    assert_bits_equal([bits(b) for b in bufs], want, "chain")


# ------------------------------------------------------------- maximum size
@pytest.mark.parametrize("algo", [RING, TREE])
def test_more_than_2_pow_32_elements_per_rank(algo, path):
    """R=2 x (2^32 + 37) bf16 per rank (8 GiB each; 32 GiB in all): element
    indices and byte offsets past 32 bits.  Inputs are small integers, so
    every result is an exact sum: checked for every element in chunks, and
    bit-exact against the oracle at sampled elements (the first ones, around
    2^31 and 2^32, the ragged tail)."""
    free, _ = torch.cuda.mem_get_info()
    if free < (40 << 30):
        pytest.skip("needs 40 GiB of free device memory")
    R, count, nch, cb = 2, (1 << 32) + 37, 12, 1 << 19
    g = torch.Generator(device="cuda")
    g.manual_seed(600)
    src = [torch.empty(count, dtype=torch.bfloat16, device="cuda").random_(-8, 9, generator=g)
           for _ in range(R)]
    dst = [torch.empty_like(s) for s in src]
    vr.vr_allreduce(src, dst, R, count, BF16, SUM, algo, nch, cb, torch.cuda.current_stream())
    assert_status_ok()
    step = 1 << 28
    for lo in range(0, count, step):
        hi = min(count, lo + step)
        want = (src[0][lo:hi].float() + src[1][lo:hi].float()).to(torch.bfloat16)
        for d in dst:
            assert torch.equal(d[lo:hi].view(torch.int16), want.view(torch.int16)), lo
    idx = sorted(set([0, 1, 7, 8, 9, (1 << 31) - 1, 1 << 31, (1 << 31) + 5, (1 << 32) - 8,
                      (1 << 32) - 1, 1 << 32, (1 << 32) + 1, count - 1]
                     + [int(x) for x in np.random.default_rng(1).integers(0, count, 40)]))
    it = torch.tensor(idx, device="cuda")
    vals = [workloads.raw_numpy(s[it].cpu()) for s in src]
    got = workloads.raw_numpy(dst[1][it].cpu())
    for n, e in enumerate(idx):
        v = [numerics.to_f32(np.array([vals[r][n]]), BF16)[0] for r in range(R)]
        from oracle import sample
        f = sample.allreduce_element(v, e, count, BF16, SUM, algo, nch, cb)
        assert numerics.from_f32(np.array([f], dtype=np.float32), BF16)[0] == got[n], e
    del src, dst
    torch.cuda.empty_cache()


# ------------------------------------------- the sweep configuration, sampled
@pytest.mark.parametrize("algo", [RING, TREE])
@pytest.mark.parametrize("size", [8 << k for k in range(26)])
def test_sweep_configuration(size, algo):
    """R=4 fp32, 12 channels, 512 KiB chunks, uniform [-1, 1) drawn on the
    device as the sweep does: every element of every rank bit-exact to the
    oracle at every size, and within the fp64 bound."""
    R, count, nch, cb = 4, size // 4, 12, 512 * 1024
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    src = [torch.rand(count, generator=g, device="cuda") * 2 - 1 for _ in range(R)]
    dst = [torch.empty_like(s) for s in src]
    vr.vr_allreduce(src, dst, R, count, F32, SUM, algo, nch, cb, torch.cuda.current_stream())
    assert_status_ok()
    raws = [workloads.raw_numpy(s.cpu()) for s in src]
    got = bits(dst[2])
    want = oracle.allreduce(raws, F32, SUM, algo, nch, cb)
    assert_bits_equal([bits(d) for d in dst], want, "sweep %d" % size)
    del want
    s = oracle.fp64_sum(raws, F32)
    a = sum(np.abs(x.astype(np.float64)) for x in raws)
    check_against_fp64(got, s, a, R, F32)
