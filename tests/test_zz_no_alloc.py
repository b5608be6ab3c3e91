"""The entry point for callers that cannot allocate device memory.

vr_allreduce_ring_stepwise_noalloc runs the stepwise ring with its message
FIFO in a device array of the library instead of caller scratch, for
callers whose device memory belongs to another allocator or who may not
call cudaMalloc / cudaFree.  Its results must equal the allocating entry
point's, bit for bit (the parity bar of the other tests), on two calls in a
row; the second call must not depend on what the first left in the array.
This file is collected last, and passes alone or after the other tests.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA device", allow_module_level=True)

import double_binary_tree_gb300 as vr  # noqa: E402


def _run_reference(inp, dtype, op, nch, cb):
    R, count = len(inp), inp[0].numel()
    src = [t.cuda() for t in inp]
    dst = [torch.empty_like(s) for s in src]
    n = vr.vr_ring_stepwise_scratch_bytes(count, dtype)
    fifo = torch.empty(n, dtype=torch.uint8, device="cuda")
    vr.vr_allreduce_ring_stepwise(src, dst, R, count, dtype, op, nch, cb, fifo, n)
    assert vr.vr_stream_status() == vr.VR_SUCCESS
    return [workloads.raw_numpy(d.cpu()) for d in dst]


def _run_noalloc(inp, dtype, op, nch, cb):
    R, count = len(inp), inp[0].numel()
    src = [t.cuda() for t in inp]
    dst = [torch.empty_like(s) for s in src]
    vr.vr_allreduce_ring_stepwise_noalloc(src, dst, R, count, dtype, op, nch, cb)
    assert vr.vr_stream_status() == vr.VR_SUCCESS
    return [workloads.raw_numpy(d.cpu()) for d in dst]


@pytest.mark.parametrize("dtype", [vr.VR_FLOAT32, vr.VR_BFLOAT16])
def test_noalloc_matches_allocating_entry_point_twice(dtype):
    cases = [  # (R, count, channels, chunk bytes, seed): the second reuses the array
        (8, 1 << 20 if dtype == vr.VR_FLOAT32 else 3 << 20, 12, 512 * 1024, 1),
        (5, 100003, 3, 4096, 2),
    ]
    for R, count, nch, cb, seed in cases:
        inp = workloads.generate(R, count, dtype, "normal", 1300 + seed)
        want = _run_reference(inp, dtype, vr.VR_SUM, nch, cb)
        got = _run_noalloc(inp, dtype, vr.VR_SUM, nch, cb)
        for g, w in zip(got, want):
            assert np.array_equal(g, w)


def test_noalloc_rejects_sizes_beyond_its_array():
    E = 4
    count = vr.VR_NOALLOC_SCRATCH_BYTES // E + 1
    src = [torch.empty(count, device="cuda") for _ in range(2)]
    dst = [torch.empty_like(s) for s in src]
    before = vr.vr_launch_count()
    with pytest.raises(vr.VrError) as ei:
        vr.vr_allreduce_ring_stepwise_noalloc(src, dst, 2, count, vr.VR_FLOAT32, vr.VR_SUM, 1, 16)
    assert ei.value.code == vr.VR_ERR_UNSUPPORTED
    assert vr.vr_launch_count() == before


def test_noalloc_allocates_nothing():
    """After the first call on the device (which looks up the array and, with
    lazily loaded modules, brings it into being), further calls leave the
    device's free memory unchanged: no allocation by the library, by CUDA
    on its behalf, or by torch."""
    R, count, dtype = 8, 1 << 20, vr.VR_FLOAT32
    inp = workloads.generate(R, count, dtype, "normal", 1310)
    src = [t.cuda() for t in inp]
    dst = [torch.empty_like(s) for s in src]
    vr.vr_allreduce_ring_stepwise_noalloc(src, dst, R, count, dtype, vr.VR_SUM, 12, 512 * 1024)
    assert vr.vr_stream_status() == vr.VR_SUCCESS
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(4):
        vr.vr_allreduce_ring_stepwise_noalloc(src, dst, R, count, dtype, vr.VR_SUM, 12,
                                              512 * 1024)
    assert vr.vr_stream_status() == vr.VR_SUCCESS
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_empty_and_single_rank():
    """count == 0 launches nothing and leaves the outputs alone; R == 1 is the
    copy of the input (no ring step)."""
    src = [torch.arange(16, dtype=torch.float32, device="cuda") for _ in range(3)]
    dst = [torch.full_like(s, -1.0) for s in src]
    before = vr.vr_launch_count()
    vr.vr_allreduce_ring_stepwise_noalloc(src, dst, 3, 0, vr.VR_FLOAT32, vr.VR_SUM, 2, 64)
    assert vr.vr_launch_count() == before
    assert all(bool((d == -1.0).all()) for d in dst)
    inp = workloads.generate(1, 100003, vr.VR_BFLOAT16, "normal", 1320)
    for _ in range(2):
        got = _run_noalloc(inp, vr.VR_BFLOAT16, vr.VR_MAX, 3, 4096)
        assert np.array_equal(got[0], workloads.raw_numpy(inp[0]))
