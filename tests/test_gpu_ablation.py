"""Parity of the non-fused variants with the oracle.

The two-phase tree reduces in the same order as the fused tree, so it must
give the oracle's tree bits.  The stepwise ring keeps partials in the element
type between hops, so it must give the oracle's ring with per-hop rounding
(identical to the fused ring for fp32 and for Max).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA device", allow_module_level=True)

import double_binary_tree_gb300 as vr  # noqa: E402

F32, F16, BF16 = vr.VR_FLOAT32, vr.VR_FLOAT16, vr.VR_BFLOAT16
SUM, MAX = vr.VR_SUM, vr.VR_MAX
TDT = workloads.TORCH_DTYPE


def _bits(t):
    return workloads.raw_numpy(t.cpu())


def _status_ok():
    st = vr.vr_stream_status()
    if st != 0:
        try:
            torch.cuda.synchronize()
            detail = "torch sees no CUDA error"
        except Exception as ex:  # the CUDA error text, for the report
            detail = repr(ex)[:300]
        raise AssertionError("status %d (%s): %s" % (st, vr.vr_get_error_string(st), detail))


def _check(got, want, what):
    for r, (g, w) in enumerate(zip(got, want)):
        assert np.array_equal(g, w), "%s: rank %d differs" % (what, r)


@pytest.mark.parametrize("dtype", [F32, F16, BF16])
@pytest.mark.parametrize("op", [SUM, MAX])
def test_tree_updown_matches_tree(dtype, op):
    for R, L, count, nch, cb, inplace, shift in [
            (2, 1, 1001, 2, 64, False, 0), (7, 1, 40003, 2, 1024, False, 0),
            (8, 1, 65536, 12, 4096, True, 0), (64, 8, 9001, 12, 512, False, 0),
            (5, 1, 777, 3, 16, False, 1)]:
        inp = workloads.generate(R, count, dtype, "normal", 1000 + R)
        want = oracle.allreduce([workloads.raw_numpy(t) for t in inp], dtype, op, 1, nch, cb,
                                local_ranks=L)
        if shift:
            bases = [torch.zeros(count + shift, dtype=TDT[dtype], device="cuda") for _ in inp]
            src = [b[shift:] for b in bases]
            for s, t in zip(src, inp):
                s.copy_(t)
        else:
            src = [t.cuda() for t in inp]
        dst = src if inplace else [torch.empty_like(s) for s in src]
        vr.vr_allreduce_tree_updown(src, dst, R, count, dtype, op, nch, cb, L)
        _status_ok()
        _check([_bits(d) for d in dst], want, "updown R=%d" % R)


@pytest.mark.parametrize("dtype", [F32, F16, BF16])
@pytest.mark.parametrize("op", [SUM, MAX])
def test_ring_stepwise_matches_hop_rounding(dtype, op):
    for R, count, nch, cb, inplace, shift in [
            (2, 999, 1, 64, False, 0), (3, 17, 2, 16, False, 0), (4, 1024, 1, 1024, False, 0),
            (7, 30011, 12, 1024, True, 0), (8, 65539, 12, 4096, False, 0),
            (16, 5000, 5, 160, False, 0), (5, 1001, 3, 48, False, 1)]:
        inp = workloads.generate(R, count, dtype, "normal", 1100 + R)
        raws = [workloads.raw_numpy(t) for t in inp]
        want = oracle.allreduce(raws, dtype, op, 0, nch, cb, hop_rounding=True)
        if shift:
            bases = [torch.zeros(count + shift, dtype=TDT[dtype], device="cuda") for _ in inp]
            src = [b[shift:] for b in bases]
            for s, t in zip(src, inp):
                s.copy_(t)
        else:
            src = [t.cuda() for t in inp]
        # outputs inside canary bytes (64 before, 64 after) that must survive
        E = vr.ELEM_SIZE[dtype]
        raw = [] if inplace else [torch.full(((count + 2 * 64) * E,), 0x5A, dtype=torch.uint8,
                                             device="cuda") for _ in src]
        dst = src if inplace else [b[64 * E:(64 + count) * E].view(TDT[dtype]) for b in raw]
        nbytes = vr.vr_ring_stepwise_scratch_bytes(count, dtype)
        scratch = torch.empty(nbytes + 16, dtype=torch.uint8, device="cuda")
        sptr = scratch.data_ptr() + (vr.ELEM_SIZE[dtype] if shift else 0)  # element-aligned
        before = vr.vr_launch_count()
        vr.vr_allreduce_ring_stepwise(src, dst, R, count, dtype, op, nch, cb, sptr, nbytes)
        _status_ok()
        assert vr.vr_launch_count() - before == 1 + 4 * (R - 1)
        for b in raw:   # nothing written past either end of an output
            assert bool((b[:64 * E] == 0x5A).all()) and bool((b[(64 + count) * E:] == 0x5A).all())
        _check([_bits(d) for d in dst], want, "stepwise R=%d" % R)
        if dtype == F32 or op == MAX:
            fused = oracle.allreduce(raws, dtype, op, 0, nch, cb)
            _check([_bits(d) for d in dst], fused, "stepwise == fused R=%d" % R)
