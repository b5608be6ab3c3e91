"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the collectives: it only draws numbers.
Both the CUDA path and the CPU oracle take their inputs from here, so the
two sides see the same bits.  Draws are rank-major from one CPU generator
(``torch.Generator('cpu').manual_seed(seed)``): rank 0's values first.

Workloads (R virtual ranks, elements per rank):

* ``small_ring``   R=4, 1024 fp32, integers uniform in [-8, 8], seed 0,
                   1 channel, chunk = count/R elements (the small ring case);
* ``two_rank``     R=2, the (1, 2), (3, 4) example;
* ``ring_64mib``   R=8, 16 777 216 fp32 (64 MiB), N(0, 1), seed 1, 12 channels,
                   512 KiB chunks;
* ``tree_4mib``    R=8 (even: mirror) and R=7 (odd: shift), 2 097 152 bf16
                   (4 MiB), N(0, 1) drawn in fp32 then rounded to bf16, seed 2,
                   2 channels (one per tree) or 12, 512 KiB chunks;
* ``sweep``        R=4, 8 B .. 256 MiB per rank (powers of two), fp32 uniform in
                   [-1, 1), seed 3, 12 channels, 512 KiB chunks;
* ``hier_16mib``   R=64 = 8 nodes x 8 local ranks, 8 388 608 fp16 (16 MiB),
                   uniform in [-1, 1) drawn in fp32 then rounded to fp16, seed 4,
                   12 channels, 512 KiB chunks, Sum and Max; also
                   ReduceScatter and AllGather alone.
"""

import torch

FLOAT32, FLOAT16, BFLOAT16 = 0, 1, 2
TORCH_DTYPE = {FLOAT32: torch.float32, FLOAT16: torch.float16, BFLOAT16: torch.bfloat16}

WORKLOADS = {
    "small_ring": dict(R=4, count=1024, dtype=FLOAT32, dist="int8", seed=0,
                       n_channels=1, chunk_bytes=256 * 4, local_ranks=1),
    "ring_64mib": dict(R=8, count=16 * 1024 * 1024, dtype=FLOAT32, dist="normal", seed=1,
                       n_channels=12, chunk_bytes=512 * 1024, local_ranks=1),
    "tree_4mib_r8": dict(R=8, count=2 * 1024 * 1024, dtype=BFLOAT16, dist="normal", seed=2,
                         n_channels=2, chunk_bytes=512 * 1024, local_ranks=1),
    "tree_4mib_r7": dict(R=7, count=2 * 1024 * 1024, dtype=BFLOAT16, dist="normal", seed=2,
                         n_channels=2, chunk_bytes=512 * 1024, local_ranks=1),
    "hier_16mib": dict(R=64, count=8 * 1024 * 1024, dtype=FLOAT16, dist="uniform", seed=4,
                       n_channels=12, chunk_bytes=512 * 1024, local_ranks=8),
}


def generate(R, count, dtype, dist, seed):
    """R CPU tensors of ``count`` elements of ``dtype``.

    dist: "normal" N(0, 1); "uniform" [-1, 1); "int8" integers in [-8, 8];
    16-bit types are drawn in fp32 and rounded by torch's conversion."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if dist == "normal":
        x = torch.randn(R, count, generator=g, dtype=torch.float32)
    elif dist == "uniform":
        x = torch.rand(R, count, generator=g, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "int8":
        x = torch.randint(-8, 9, (R, count), generator=g).to(torch.float32)
    elif dist == "pow2":
        # rank r holds 2**r everywhere: every result is the bitmask of the
        # ranks that contributed to it
        x = torch.stack([torch.full((count,), float(2 ** r)) for r in range(R)])
    else:
        raise ValueError("unknown distribution %r" % (dist,))
    x = x.to(TORCH_DTYPE[dtype])
    return [x[r].clone() for r in range(R)]


def two_rank():
    """The two-rank example: rank 0 holds (1, 2), rank 1 holds (3, 4)."""
    return [torch.tensor([1.0, 2.0]), torch.tensor([3.0, 4.0])]


def workload(name):
    w = dict(WORKLOADS[name])
    w["inputs"] = generate(w["R"], w["count"], w["dtype"], w["dist"], w["seed"])
    return w


def raw_numpy(t):
    """Storage view for the oracle: float32 as is, 16-bit types as uint16."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view("uint16")
