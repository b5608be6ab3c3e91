"""CPU oracle for the emulated Ring / Double-Binary-Tree AllReduce.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, links or
runs this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It
shares no code, table or helper with the CUDA path: the two meet only on the
seeded inputs built by ``workloads.py``.

It is deliberately plain and slow: pure-Python integer code for topology and
partition, and numpy float32 element-wise arithmetic (IEEE round-to-nearest-
even, no flush-to-zero) for the literal message-passing simulations of the
ring and tree schedules.  An fp64 brute-force sum gives the plain definition
the schedules must approach.

Sources (web pages), cited in every module as ``[tag] section``:

* [Course13]  "NCCL 专家课程 13：Tree、双树、层次化连接与真实交叉区间"
              (blog.cptz.space) -- ncclTree, ncclTopoPreset, connectTrees,
              ncclGetBtree, ncclGetDtree, runTreeSplit, the Dtree probe table.
* [Internals] "NCCL 内部机制：一次 AllReduce 如何变成拓扑图、Channel 与 GPU
              Kernel" (charlestar.github.io) -- API contract, chunk/slice/step,
              the Ring AllReduce step structure, algbw/busbw.
* [CodeNotes] "NCCL代码分析" (jianzi123.github.io) -- algorithm support table
              (tree is AllReduce-only).
* [Interview] "all-reduce 每张卡要发多少数据? ring 和 tree 有什么区别?"
              (charliedreemur.github.io) -- definitions, the 2-rank example,
              Figure 1 (4-rank ring trace), closed forms, the NumPy ring
              simulation, busbw.

Where the pages are silent the module that takes a reading says so in its
docstring; every such reading is also listed in the design notes.
"""

from . import numerics, topology, partition, schedules, sample, api  # noqa: F401
from .api import allreduce, reduce_scatter, allgather, fp64_sum, fp64_max  # noqa: F401
