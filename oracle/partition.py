"""Channel, loop and block partition of a message.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).  Pure-Python integers.

Sources:
* [Course13] section "前置知识": a channel is an independent topology plus a
  share of the work; channels process different ranges of the message, not
  copies of it.  Section "runTreeSplit 如何流水": a tree channel walks its range
  in chunks of chunkCount elements.
* [Internals] section "Chunk、slice、step 是三个尺度": the tensor is first
  partitioned over channels, then cut into chunks that travel the ring or
  tree.
* [Interview] section "手撕代码(NumPy 模拟 ring all-reduce)": a rank's data is
  cut into n blocks with numpy ``array_split`` semantics (the first L mod n
  blocks are one element longer).

Reading (the per-channel formula is not on the pages): channels split the
message in 16-byte grains with ``array_split`` semantics over grains; the
ring then walks a channel in loops of R*C elements (C = chunkBytes / E), the
last loop shorter, and cuts each loop into R blocks with ``array_split``
semantics.  The partition changes only which block an element falls in (its
ring fold order), never the set of elements.
"""

GRAIN_BYTES = 16


def split_sizes(total, parts):
    """``array_split`` sizes: the first total % parts pieces get one more."""
    q, m = divmod(total, parts)
    return [q + (1 if i < m else 0) for i in range(parts)]


def split_ranges(total, parts):
    """``array_split`` as (start, length) pairs."""
    out, s = [], 0
    for n in split_sizes(total, parts):
        out.append((s, n))
        s += n
    return out


def channel_ranges(count, elem_size, n_channels):
    """Element range [start, start+len) of every channel: grains of 16 bytes
    split over channels, clipped at ``count``."""
    if GRAIN_BYTES % elem_size:
        raise ValueError("element size must divide 16")
    U = GRAIN_BYTES // elem_size
    grains = -(-count // U)
    out = []
    for gs, gn in split_ranges(grains, n_channels):
        s = min(count, gs * U)
        e = min(count, (gs + gn) * U)
        out.append((s, e - s))
    return out


def ring_blocks(ch_start, ch_len, R, chunk_elems):
    """The ring's blocks inside one channel: loops of R*C elements (the last
    loop shorter), each loop cut into R blocks.  Returns a list of loops; each
    loop is a list of R (start, length) pairs in absolute element offsets,
    indexed by block number j."""
    if chunk_elems < 1:
        raise ValueError("chunk must hold at least one element")
    loops = []
    step = R * chunk_elems
    off = 0
    while off < ch_len:
        L = min(step, ch_len - off)
        loops.append([(ch_start + off + s, n) for s, n in split_ranges(L, R)])
        off += L
    return loops


def tree_chunks(ch_start, ch_len, chunk_elems):
    """A tree channel's chunks of C elements (the last one shorter)."""
    out, off = [], 0
    while off < ch_len:
        n = min(chunk_elems, ch_len - off)
        out.append((ch_start + off, n))
        off += n
    return out
