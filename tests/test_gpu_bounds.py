"""The bounds-checked build on the GPU (libvr_debug.so, VR_BOUNDS_CHECKED=1).

1. The small parity cases (rings and trees of 1-64 ranks, three dtypes, Sum
   and Max, both kernel paths, ragged and misaligned buffers, in place,
   ReduceScatter, AllGather in both tile orders, the non-fused variants, the
   folds specialised at run time, the bounded-wait failure path, the
   allocation-free entry point) run against the checked library in a child
   process: every call's status is what the test expects, no address was
   refused, and every output still equals the oracle bit for bit.
2. The checks fire: with the recorded extents of one launch shortened by
   16 bytes (vr_debug_shrink_next -- the buffers themselves stay whole, so
   no access ever leaves real memory), the accesses to the last 16 bytes
   are refused: VR_ERR_INTERNAL (not a timeout: a refused bulk copy still
   completes its barrier), the refused address is reported, and the
   outputs equal the oracle everywhere else (outside the last 16 bytes, or
   the last tile where a refused access was a bulk copy of a whole tile),
   and with receive buffers cut, their last 16 bytes keep their old
   contents.  Ring, tree, ReduceScatter and
   AllGather on the register path and the staged / TMA kernels.
No bad plan is ever given to a kernel.
"""

import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

from tests.conftest import ROOT  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA device", allow_module_level=True)

ENV = dict(os.environ, VR_BOUNDS_CHECKED="1")


def test_small_parity_cases_pass_under_bounds_checks():
    args = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "gpu",
            os.path.join("tests", "test_gpu_parity.py"), os.path.join("tests", "test_gpu_ablation.py"),
            os.path.join("tests", "test_gpu_jit.py"), os.path.join("tests", "test_gpu_failure.py"),
            os.path.join("tests", "test_zz_no_alloc.py"),
            "-k", "not full_size and not 2_pow_32 and not sweep_configuration and not allreduce_host "
                  "and not at_16_mib and not at_32_mib and not at_64_mib"]
    r = subprocess.run(args, cwd=ROOT, env=ENV, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "skipped" not in r.stdout.splitlines()[-1], r.stdout[-500:]


def test_drawn_tiles_pass_under_bounds_checks():
    """The staged kernels that draw their tiles (trees and rings, small and
    ragged messages, ring blocks far smaller than a tile) under the checks."""
    args = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "gpu",
            os.path.join("tests", "test_gpu_sched.py"), "-k", "small_and_ragged or many_blocks"]
    r = subprocess.run(args, cwd=ROOT, env=ENV, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "skipped" not in r.stdout.splitlines()[-1], r.stdout[-500:]


SHRINK = r"""
import numpy as np, torch, double_binary_tree_gb300 as vr, oracle, workloads
assert vr.vr_debug_bounds_checked()
st = torch.cuda.current_stream()
SENT = 0x7F
TAIL = 64 * 1024   # a refused bulk copy leaves its whole tile (at most 64 KB) unread

def run(coll, R, n, dtype, algo, path, which):
    vr.vr_set_option("VR_KERNEL_PATH", {"register": 1, "staged": 2}[path])
    inp = workloads.generate(R, (R * n) if coll == "rs" else n, dtype, "normal", 77)
    src = [t.cuda() for t in inp]
    nout = {"ar": n, "rs": n, "ag": R * n}[coll]
    E = vr.ELEM_SIZE[dtype]
    dst = [torch.full((nout * E,), SENT, dtype=torch.uint8, device="cuda").view(inp[0].dtype)
           for _ in range(R)]
    vr.vr_debug_shrink_next(16, which)
    if coll == "ar":
        vr.vr_allreduce(src, dst, R, n, dtype, 0, algo, 12, 1 << 16, st)
    elif coll == "rs":
        vr.vr_reduce_scatter(src, dst, R, n, dtype, 0, 0, 12, 1 << 16, st)
    else:
        vr.vr_allgather(src, dst, R, n, dtype, 0, 12, 1 << 16, st)
    status = vr.vr_stream_status(st)
    where = vr.vr_debug_bounds_fault()
    what = (coll, path, which)
    assert status == vr.VR_ERR_INTERNAL, (what, status)   # refused, not timed out
    bufs = dst if which == 2 else src
    # a refused bulk copy (staged loads, the TMA AllGather's stores) covers a
    # whole tile, so it reports the tile's start
    bulk = which == 1 or (coll == "ag" and path == "staged")
    span = TAIL if bulk else 16
    ends = [(b.data_ptr() + b.numel() * E - span, b.data_ptr() + b.numel() * E) for b in bufs]
    assert any(lo <= where < hi for lo, hi in ends), (what, hex(where))
    raws = [workloads.raw_numpy(t) for t in inp]
    if coll == "ar":
        want = oracle.allreduce(raws, dtype, 0, algo, 12, 1 << 16)
    elif coll == "rs":
        want = oracle.reduce_scatter(raws, dtype, 0)
    else:
        want = oracle.allgather(raws)
    for d, w in zip(dst, want):
        got = workloads.raw_numpy(d.cpu())
        k = span // E    # outputs exact before the refused span
        if coll == "ag" and which == 1:   # every source's tail feeds its own block
            for r in range(R):
                assert np.array_equal(got[r * n:(r + 1) * n - k], w[r * n:(r + 1) * n - k]), what
        else:
            assert np.array_equal(got[:-k], w[:-k]), what
        if which == 2:   # the refused stores were not made
            assert bool((d.view(torch.uint8)[-16:] == SENT).all()), what
    assert vr.vr_stream_status(st) == 0 and vr.vr_debug_bounds_fault() == 0

for path in ("register", "staged"):
    run("ar", 8, 1 << 20, vr.VR_FLOAT32, vr.VR_ALGO_RING, path, 2)
    run("ar", 8, 1 << 20, vr.VR_BFLOAT16, vr.VR_ALGO_TREE, path, 2)
    run("rs", 4, 1 << 18, vr.VR_FLOAT32, 0, path, 2)
    run("ag", 4, 1 << 18, vr.VR_FLOAT16, 0, path, 2)
    run("ar", 8, 1 << 20, vr.VR_FLOAT32, vr.VR_ALGO_RING, path, 1)
run("ag", 4, 1 << 18, vr.VR_FLOAT16, 0, "staged", 1)
print("refused and reported")
"""


def test_shortened_extents_are_refused_and_reported():
    r = subprocess.run([sys.executable, "-c", SHRINK], cwd=ROOT, env=ENV, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-3000:]
    assert "refused and reported" in r.stdout
