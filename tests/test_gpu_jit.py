"""Tree kernels specialised at run time (the straight-line folds compiled with
NVRTC) against the interpreting kernels and the oracle: both bit-exact on
the same inputs, on the register and the staged path."""


import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect these
    pytest.skip("needs a CUDA device", allow_module_level=True)

import double_binary_tree_gb300 as vr  # noqa: E402
from tests.options import options  # noqa: E402

TREE, RING = vr.VR_ALGO_TREE, vr.VR_ALGO_RING
F32, F16, BF16 = vr.VR_FLOAT32, vr.VR_FLOAT16, vr.VR_BFLOAT16
SUM = vr.VR_SUM


def _run(inp, dtype, op, nch, cb, L, jit, path):
    R, count = len(inp), inp[0].numel()
    with options(vr, VR_JIT=1 if jit else 0, VR_KERNEL_PATH=path):
        src = [t.cuda() for t in inp]
        dst = [torch.empty_like(s) for s in src]
        vr.vr_allreduce_ex(src, dst, R, count, dtype, op, TREE, nch, cb, L,
                           torch.cuda.current_stream())
        assert vr.vr_stream_status(torch.cuda.current_stream()) == 0
        return [workloads.raw_numpy(d.cpu()) for d in dst]


def test_specialisation_is_available():
    enabled, _, failed = vr.vr_jit_status()
    assert enabled, "NVRTC or the kernel sources beside the library were not found"
    assert failed == 0


@pytest.mark.parametrize("path", ["register", "staged"])
@pytest.mark.parametrize("nodes,L,dtype,op,count,nch", [
    (2, 1, vr.VR_FLOAT32, vr.VR_SUM, 10007, 2),
    (3, 1, vr.VR_BFLOAT16, vr.VR_SUM, 30011, 3),
    (7, 1, vr.VR_FLOAT16, vr.VR_MAX, 65539, 2),
    (8, 1, vr.VR_FLOAT32, vr.VR_MAX, 100003, 12),
    (16, 1, vr.VR_BFLOAT16, vr.VR_SUM, 20011, 4),
    (2, 4, vr.VR_FLOAT16, vr.VR_SUM, 9001, 5),
    (8, 8, vr.VR_BFLOAT16, vr.VR_SUM, 12345, 12),
])
def test_specialised_equals_interpreted_equals_oracle(nodes, L, dtype, op, count, nch, path):
    R = nodes * L
    inp = workloads.generate(R, count, dtype, "normal", 300 + R)
    want = oracle.allreduce([workloads.raw_numpy(t) for t in inp], dtype, op, TREE, nch, 1024,
                            local_ranks=L)
    _, compiled0, _ = vr.vr_jit_status()
    got_jit = _run(inp, dtype, op, nch, 1024, L, True, path)
    _, compiled1, failed = vr.vr_jit_status()
    got_int = _run(inp, dtype, op, nch, 1024, L, False, path)
    assert failed == 0
    assert compiled1 >= compiled0
    for r in range(R):
        assert np.array_equal(got_jit[r], want[r]), "specialised rank %d" % r
        assert np.array_equal(got_int[r], want[r]), "interpreted rank %d" % r


@pytest.mark.parametrize("path", ["register", "staged"])
@pytest.mark.parametrize("R,dtype,op,count,nch,cb", [
    (2, vr.VR_FLOAT32, vr.VR_SUM, 10007, 2, 64),
    (3, vr.VR_BFLOAT16, vr.VR_MAX, 30011, 3, 48),
    (4, vr.VR_FLOAT32, vr.VR_SUM, 65539, 12, 1024),
    (7, vr.VR_FLOAT16, vr.VR_SUM, 100003, 5, 160),
    (8, vr.VR_FLOAT32, vr.VR_SUM, 262147, 12, 4096),
    (16, vr.VR_BFLOAT16, vr.VR_SUM, 40009, 4, 256),
])
def test_specialised_ring_equals_oracle(R, dtype, op, count, nch, cb, path):
    """Ring folds specialised for R ranks (VR_JIT_RING=1) against the oracle:
    blocks cut units (small chunks), so the split and element paths run too."""
    inp = workloads.generate(R, count, dtype, "normal", 400 + R)
    want = oracle.allreduce([workloads.raw_numpy(t) for t in inp], dtype, op,
                            vr.VR_ALGO_RING, nch, cb)
    with options(vr, VR_JIT_RING=1, VR_KERNEL_PATH=path):
        src = [t.cuda() for t in inp]
        dst = [torch.empty_like(s) for s in src]
        vr.vr_allreduce(src, dst, R, count, dtype, op, vr.VR_ALGO_RING, nch, cb,
                        torch.cuda.current_stream())
        assert vr.vr_stream_status(torch.cuda.current_stream()) == 0
        got = [workloads.raw_numpy(d.cpu()) for d in dst]
    assert vr.vr_jit_status()[2] == 0
    for r in range(R):
        assert np.array_equal(got[r], want[r]), "rank %d" % r


@pytest.mark.parametrize("occ", ["0", "4"])
def test_four_ctas_per_sm_same_bits(occ):
    """The specialised register-path kernels compiled for four CTAs per SM
    (VR_JIT_OCC=4, rings included) give the oracle's bits, like those at
    their natural occupancy (VR_JIT_OCC=0)."""
    for R, dtype, algo, count in [(8, BF16, TREE, 300001), (7, BF16, TREE, 300001),
                                  (4, F32, TREE, 200003), (5, F16, RING, 300001),
                                  (8, F32, RING, 200003)]:
        inp = workloads.generate(R, count, dtype, "normal", 900 + R)
        raws = [workloads.raw_numpy(t) for t in inp]
        want = oracle.allreduce(raws, dtype, SUM, algo, 12, 4096)
        src = [t.cuda() for t in inp]
        dst = [torch.empty_like(t) for t in src]
        with options(vr, VR_JIT_OCC=int(occ)):
            vr.vr_allreduce(src, dst, R, count, dtype, SUM, algo, 12, 4096,
                            torch.cuda.current_stream())
        assert vr.vr_stream_status(torch.cuda.current_stream()) == 0
        for d, w in zip(dst, want):
            assert np.array_equal(workloads.raw_numpy(d), w), (R, dtype, algo)
