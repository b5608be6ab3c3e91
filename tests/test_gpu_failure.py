"""Device-side failure detection without a GPU fault.

The staged kernels and the TMA AllGather bound every wait.  The library's
test hook makes the first CTA of the next such call skip the loads of one
tile, so the wait for
that tile runs out: the call must report VR_ERR_TIMEOUT through
vr_stream_status within about the wait limit (1 s), leave the context usable,
and the next call must be bit-exact again.  Nothing here traps, faults or
waits without a bound.
"""

import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA device", allow_module_level=True)

import double_binary_tree_gb300 as vr  # noqa: E402
from tests.options import options  # noqa: E402


@pytest.fixture(autouse=True)
def staged_path():
    """The bounded waits live in the shared-memory-staged kernels."""
    with options(vr, VR_KERNEL_PATH="staged"):
        yield


@pytest.mark.parametrize("algo", [vr.VR_ALGO_RING, vr.VR_ALGO_TREE])
def test_stalled_tile_reports_timeout_then_recovers(algo):
    R, count = 8, 1 << 20
    inp = workloads.generate(R, count, vr.VR_FLOAT32, "normal", 900)
    src = [t.cuda() for t in inp]
    dst = [torch.empty_like(s) for s in src]
    stream = torch.cuda.current_stream()
    assert vr.vr_stream_status(stream) == vr.VR_SUCCESS

    vr.vr_debug_stall_next(0)
    t0 = time.time()
    vr.vr_allreduce(src, dst, R, count, vr.VR_FLOAT32, vr.VR_SUM, algo, 12, 512 * 1024, stream)
    assert vr.vr_stream_status(stream) == vr.VR_ERR_TIMEOUT
    elapsed = time.time() - t0
    assert elapsed < 30.0, elapsed
    # the status word was cleared by the read
    assert vr.vr_stream_status(stream) == vr.VR_SUCCESS

    # the context is usable and the next call is exact
    vr.vr_allreduce(src, dst, R, count, vr.VR_FLOAT32, vr.VR_SUM, algo, 12, 512 * 1024, stream)
    assert vr.vr_stream_status(stream) == vr.VR_SUCCESS
    want = oracle.allreduce([workloads.raw_numpy(t) for t in inp], vr.VR_FLOAT32, vr.VR_SUM, algo,
                            12, 512 * 1024)
    for d, w in zip(dst, want):
        assert np.array_equal(workloads.raw_numpy(d.cpu()).view(np.uint32), w.view(np.uint32))


def test_stall_request_is_consumed_once_and_cancellable():
    R, count = 4, 4096
    src = [torch.ones(count, device="cuda") for _ in range(R)]
    dst = [torch.empty_like(s) for s in src]
    vr.vr_debug_stall_next(5)
    vr.vr_debug_stall_next(-1)          # cancelled before use
    vr.vr_allreduce(src, dst, R, count, vr.VR_FLOAT32, vr.VR_SUM, vr.VR_ALGO_RING, 1, 1024)
    assert vr.vr_stream_status() == vr.VR_SUCCESS
    assert all(bool((d == 4).all()) for d in dst)
    with pytest.raises(vr.VrError):
        vr.vr_debug_stall_next(-2)


@pytest.mark.parametrize("order", [1, 2])
def test_allgather_stalled_tile_times_out_and_recovers(order):
    """The TMA AllGather's waits are bounded too (source-major and
    destination-major kernels): CTA 0 skips the load of its first tile, the
    call reports VR_ERR_TIMEOUT, and the next call is exact."""
    R, sc = 4, 1 << 20
    src = [torch.full((sc,), float(r + 1), device="cuda") for r in range(R)]
    dst = [torch.zeros(R * sc, device="cuda") for _ in range(R)]
    stream = torch.cuda.current_stream()
    with options(vr, VR_AG_ORDER=order):
        vr.vr_debug_stall_next(0)
        t0 = time.time()
        vr.vr_allgather(src, dst, R, sc, vr.VR_FLOAT32, vr.VR_ALGO_RING, 12, 512 * 1024, stream)
        assert vr.vr_stream_status(stream) == vr.VR_ERR_TIMEOUT
        assert time.time() - t0 < 30
        vr.vr_allgather(src, dst, R, sc, vr.VR_FLOAT32, vr.VR_ALGO_RING, 12, 512 * 1024,
                        stream)
    assert vr.vr_stream_status(stream) == 0
    want = torch.cat(src)
    for d in dst:
        assert torch.equal(d, want)
