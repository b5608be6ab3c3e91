"""VR_DEBUG=GRAPH on collective calls: the first call of each plan prints a
header, the channels' trees in both log formats of the pages ([Course13]
"从 GRAPH 日志复原 active tree") or the ring order, and the channel partition;
every table equals the oracle's (trees, rings, channel ranges) line for line,
and a repeated call prints nothing more."""

import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

from oracle import partition, topology  # noqa: E402
from tests.conftest import ROOT  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA device", allow_module_level=True)

CODE = """
import torch, double_binary_tree_gb300 as vr
def bufs(R, n, dt):
    return ([torch.randn(n, device="cuda").to(dt) for _ in range(R)],
            [torch.empty(n, dtype=dt, device="cuda") for _ in range(R)])
s, d = bufs(8, 10007, torch.bfloat16)
vr.vr_allreduce_ex(s, d, 8, 10007, vr.VR_BFLOAT16, 0, vr.VR_ALGO_TREE, 3, 1024, 2, None)
s, d = bufs(5, 1000, torch.float32)
for _ in range(2):
    vr.vr_allreduce(s, d, 5, 1000, vr.VR_FLOAT32, 0, vr.VR_ALGO_RING, 2, 64, None)
s, d = bufs(4, 4 * 64, torch.float16)
vr.vr_reduce_scatter(s, [x[:64] for x in d], 4, 64, vr.VR_FLOAT16, 0, 0, 2, 64, None)
assert vr.vr_stream_status(None) == 0
"""


def _ring_lines(R, nch):
    nxt, _ = topology.build_ring(R, nch)
    out = []
    for c in range(nch):
        order, v = [], 0
        for _ in range(R):
            order.append(v)
            v = nxt[c][v]
        out.append("Ring %d : %s" % (c, " ".join(map(str, order))))
    return out


def test_plan_log_equals_the_oracle_tables():
    env = dict(os.environ, VR_DEBUG="GRAPH")
    r = subprocess.run([sys.executable, "-c", CODE], cwd=ROOT, env=env, check=True,
                       capture_output=True, text=True)
    lines = [ln for ln in r.stderr.splitlines() if ln.split(" ", 1)[0] in
             ("vr", "Tree", "Trees", "Ring", "Part")]
    want = ["vr plan: allreduce tree R=8 localRanks=2 count=10007 dtype=2 nChannels=3 "
            "chunkBytes=1024"]
    for c, tr in enumerate(topology.build_dtree(4, 2, 3)):
        want += topology.format_tree_log(tr, c, "arrow") + topology.format_tree_log(tr, c, "b")
    want += ["Part %d : offset %d count %d" % (c, s, n)
             for c, (s, n) in enumerate(partition.channel_ranges(10007, 2, 3))]
    want += ["vr plan: allreduce ring R=5 localRanks=1 count=1000 dtype=0 nChannels=2 "
             "chunkBytes=64"] + _ring_lines(5, 2)
    want += ["Part %d : offset %d count %d" % (c, s, n)
             for c, (s, n) in enumerate(partition.channel_ranges(1000, 4, 2))]
    want += ["vr plan: reduce_scatter ring R=4 localRanks=1 count=64 dtype=1 nChannels=2 "
             "chunkBytes=64"] + _ring_lines(4, 2)
    assert lines == want
