"""Python binding of libvr.so (include/vr.h): argument marshalling only.

Every function keeps the C name and argument order.  Buffer arguments take
sequences of device pointers (ints) or of torch tensors (their data_ptr() is
passed); streams take a cudaStream_t as an int, a torch.cuda.Stream, or None
for the legacy default stream.  A non-zero result code raises VrError.

The compute path is the CUDA library only: the first call loads libvr.so
and fails loudly (ImportError) when it has not been built for this machine
(build it with ``python -m double_binary_tree_gb300.build`` or
``__graft_entry__.build()``).  With VR_BOUNDS_CHECKED=1 in the environment
it loads the bounds-checked build libvr_debug.so instead (built by
``build(debug=True)``), in which every kernel access is checked against its
call's buffers.
"""

import ctypes
import os

from .build import LIB, LIB_DEBUG, is_fresh

VR_SUCCESS, VR_ERR_INVALID_ARGUMENT, VR_ERR_UNSUPPORTED = 0, 1, 2
VR_ERR_CUDA, VR_ERR_TIMEOUT, VR_ERR_INTERNAL = 3, 4, 5
VR_FLOAT32, VR_FLOAT16, VR_BFLOAT16 = 0, 1, 2
VR_SUM, VR_MAX = 0, 1
VR_ALGO_RING, VR_ALGO_TREE, VR_ALGO_AUTO = 0, 1, 2
VR_PATTERN_TREE, VR_PATTERN_SPLIT_TREE, VR_PATTERN_BALANCED_TREE = 0, 1, 2
VR_MAX_RANKS = 64
VR_MAX_CHANNELS = 64
VR_NOALLOC_SCRATCH_BYTES = 8 << 20
VR_HOST_PIECE_BYTES = 8 << 20
ELEM_SIZE = {VR_FLOAT32: 4, VR_FLOAT16: 2, VR_BFLOAT16: 2}


class VrError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s: %s (%d)" % (where, vr_get_error_string(code), code))


class vr_cost_model_t(ctypes.Structure):
    _fields_ = [("alphaUs", ctypes.c_double * 2), ("usPerByte", ctypes.c_double * 2)]


class vr_tree_t(ctypes.Structure):
    _fields_ = [("depth", ctypes.c_int), ("up", ctypes.c_int), ("down", ctypes.c_int * 3)]


P, I, S, VP = ctypes.POINTER, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
PP = P(VP)
_SIGNATURES = {
    "vr_build_ring": (I, [I, I, P(I), P(I)]),
    "vr_build_dtree": (I, [I, I, I, P(vr_tree_t)]),
    "vr_build_dtree_ex": (I, [I, I, I, I, P(I), P(vr_tree_t)]),
    "vr_partition": (I, [S, I, I, I, P(S), P(S)]),
    "vr_ring_block": (I, [S, I, I, I, S, S, P(I), P(I)]),
    "vr_allreduce": (I, [PP, PP, I, S, I, I, I, I, S, VP]),
    "vr_allreduce_ex": (I, [PP, PP, I, S, I, I, I, I, S, I, VP]),
    "vr_allreduce_host": (I, [PP, PP, I, S, I, I, I, I, S, I, PP, S, VP]),
    "vr_allreduce_trees": (I, [PP, PP, I, S, I, I, I, S, P(vr_tree_t), VP]),
    "vr_reduce_scatter": (I, [PP, PP, I, S, I, I, I, I, S, VP]),
    "vr_allgather": (I, [PP, PP, I, S, I, I, I, S, VP]),
    "vr_allreduce_tree_updown": (I, [PP, PP, I, S, I, I, I, S, I, VP]),
    "vr_ring_stepwise_scratch_bytes": (S, [S, I]),
    "vr_allreduce_ring_stepwise": (I, [PP, PP, I, S, I, I, I, S, VP, S, VP]),
    "vr_allreduce_ring_stepwise_noalloc": (I, [PP, PP, I, S, I, I, I, S, VP]),
    "vr_predict_us": (I, [I, I, I, S, P(vr_cost_model_t), P(ctypes.c_double)]),
    "vr_select_algo": (I, [I, I, S, P(vr_cost_model_t), P(I)]),
    "vr_set_cost_model": (I, [P(vr_cost_model_t)]),
    "vr_fit_cost_model": (I, [I, P(I), P(I), P(S), P(ctypes.c_double), P(ctypes.c_double),
                              P(vr_cost_model_t)]),
    "vr_crossover_bytes": (I, [I, I, P(vr_cost_model_t), P(ctypes.c_double)]),
    "vr_jit_status": (I, [P(I), P(ctypes.c_longlong), P(ctypes.c_longlong)]),
    "vr_jit_compile_dtree": (I, [I, I, I, I, I, P(S), ctypes.c_char_p, S]),
    "vr_jit_compile_ring": (I, [I, I, I, I, P(S), ctypes.c_char_p, S]),
    "vr_stream_status": (I, [VP]),
    "vr_launch_count": (ctypes.c_ulonglong, []),
    "vr_debug_stall_next": (I, [ctypes.c_longlong]),
    "vr_debug_sched_slot": (I, [VP, P(ctypes.c_ulonglong), I]),
    "vr_set_option": (I, [ctypes.c_char_p, ctypes.c_longlong]),
    "vr_debug_bounds_checked": (I, []),
    "vr_debug_shrink_next": (I, [ctypes.c_longlong, I]),
    "vr_debug_bounds_fault": (I, [P(ctypes.c_ulonglong)]),
    "vr_debug_access_ok": (I, [PP, P(ctypes.c_ulonglong), P(I), I, VP, ctypes.c_ulonglong, I]),
    "vr_get_option": (I, [ctypes.c_char_p, P(ctypes.c_longlong)]),
    "vr_get_error_string": (ctypes.c_char_p, [I]),
    "vr_finalize": (None, []),
}
EXPORTED = tuple(_SIGNATURES)
_lib = None


def library_path():
    """The library this process loads: libvr.so, or libvr_debug.so when
    VR_BOUNDS_CHECKED=1."""
    return LIB_DEBUG if os.environ.get("VR_BOUNDS_CHECKED") == "1" else LIB


def _load():
    path = library_path()
    debug = path == LIB_DEBUG
    name = os.path.basename(path)
    how = "python -m double_binary_tree_gb300.build" + (" --debug" if debug else "")
    if not os.path.exists(path):
        raise ImportError("%s is not built: run %s" % (name, how))
    if not is_fresh(debug):
        raise ImportError("%s is older than its sources or built for another machine: "
                          "run %s" % (name, how))
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def _L():
    """The loaded library (loaded on first use)."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def _check(code, where):
    if code != VR_SUCCESS:
        raise VrError(code, where)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _ptrs(bufs):
    if bufs is None:
        return None
    return (ctypes.c_void_p * len(bufs))(*[_ptr(b) for b in bufs])


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ------------------------------------------------------------- topology
def vr_build_ring(R, nChannels):
    """Returns (next, prev) as lists of nChannels*R ints."""
    n = (ctypes.c_int * (R * nChannels))() if R > 0 and nChannels > 0 else None
    p = (ctypes.c_int * (R * nChannels))() if R > 0 and nChannels > 0 else None
    _check(_L().vr_build_ring(R, nChannels, n, p), "vr_build_ring")
    return list(n), list(p)


def vr_build_dtree(nNodes, localRanks, nChannels):
    """Returns nChannels*nNodes*localRanks vr_tree_t records, [c*R + r]."""
    R = nNodes * localRanks
    size = max(R * nChannels, 1)
    out = (vr_tree_t * size)()
    _check(_L().vr_build_dtree(nNodes, localRanks, nChannels, out), "vr_build_dtree")
    return list(out)[:R * nChannels]


def vr_build_dtree_ex(nNodes, localRanks, nChannels, pattern=VR_PATTERN_TREE, intraOrders=None):
    """intraOrders: None or nChannels rows of localRanks ints."""
    R = nNodes * localRanks
    out = (vr_tree_t * max(R * nChannels, 1))()
    orders = None
    if intraOrders is not None:
        flat = [int(x) for row in intraOrders for x in row]
        orders = (ctypes.c_int * max(len(flat), 1))(*flat)
    _check(_L().vr_build_dtree_ex(nNodes, localRanks, nChannels, pattern, orders, out),
           "vr_build_dtree_ex")
    return list(out)[:R * nChannels]


def vr_partition(count, dtype, nChannels, channel):
    """Returns (offset, channelCount)."""
    off, n = ctypes.c_size_t(), ctypes.c_size_t()
    _check(_L().vr_partition(count, dtype, nChannels, channel, ctypes.byref(off), ctypes.byref(n)),
           "vr_partition")
    return off.value, n.value


def vr_ring_block(count, dtype, R, nChannels, chunkBytes, elem):
    """Returns (channel, block) of element `elem`."""
    c, b = ctypes.c_int(), ctypes.c_int()
    _check(_L().vr_ring_block(count, dtype, R, nChannels, chunkBytes, elem, ctypes.byref(c),
                              ctypes.byref(b)), "vr_ring_block")
    return c.value, b.value


# ---------------------------------------------------------- collectives
def vr_allreduce(sendbufs, recvbufs, R, count, dtype, op, algo, nChannels, chunkBytes,
                 stream=None):
    _check(_L().vr_allreduce(_ptrs(sendbufs), _ptrs(recvbufs), R, count, dtype, op, algo,
                             nChannels, chunkBytes, _stream(stream)), "vr_allreduce")


def vr_allreduce_ex(sendbufs, recvbufs, R, count, dtype, op, algo, nChannels, chunkBytes,
                    localRanks, stream=None):
    _check(_L().vr_allreduce_ex(_ptrs(sendbufs), _ptrs(recvbufs), R, count, dtype, op, algo,
                                nChannels, chunkBytes, localRanks, _stream(stream)),
           "vr_allreduce_ex")


def vr_allreduce_host(sendbufs, recvbufs, R, count, dtype, op, algo, nChannels, chunkBytes,
                      localRanks, workbufs, pieceBytes=0, stream=None):
    """sendbufs / recvbufs: host tensors (pinned for overlap); workbufs:
    device tensors of count elements each."""
    _check(_L().vr_allreduce_host(_ptrs(sendbufs), _ptrs(recvbufs), R, count, dtype, op, algo,
                                  nChannels, chunkBytes, localRanks, _ptrs(workbufs),
                                  pieceBytes, _stream(stream)),
           "vr_allreduce_host")


def vr_allreduce_trees(sendbufs, recvbufs, R, count, dtype, op, nChannels, chunkBytes, trees,
                       stream=None):
    """trees: nChannels*R vr_tree_t records (as vr_build_dtree_ex returns)."""
    arr = (vr_tree_t * max(len(trees), 1))(*trees) if trees is not None else None
    _check(_L().vr_allreduce_trees(_ptrs(sendbufs), _ptrs(recvbufs), R, count, dtype, op,
                                   nChannels, chunkBytes, arr, _stream(stream)),
           "vr_allreduce_trees")


def vr_reduce_scatter(sendbufs, recvbufs, R, recvcount, dtype, op, algo, nChannels, chunkBytes,
                      stream=None):
    _check(_L().vr_reduce_scatter(_ptrs(sendbufs), _ptrs(recvbufs), R, recvcount, dtype, op,
                                  algo, nChannels, chunkBytes, _stream(stream)),
           "vr_reduce_scatter")


def vr_allgather(sendbufs, recvbufs, R, sendcount, dtype, algo, nChannels, chunkBytes,
                 stream=None):
    _check(_L().vr_allgather(_ptrs(sendbufs), _ptrs(recvbufs), R, sendcount, dtype, algo,
                             nChannels, chunkBytes, _stream(stream)), "vr_allgather")


def vr_allreduce_tree_updown(sendbufs, recvbufs, R, count, dtype, op, nChannels, chunkBytes,
                             localRanks, stream=None):
    _check(_L().vr_allreduce_tree_updown(_ptrs(sendbufs), _ptrs(recvbufs), R, count, dtype, op,
                                         nChannels, chunkBytes, localRanks, _stream(stream)),
           "vr_allreduce_tree_updown")


def vr_ring_stepwise_scratch_bytes(count, dtype):
    return _L().vr_ring_stepwise_scratch_bytes(count, dtype)


def vr_allreduce_ring_stepwise(sendbufs, recvbufs, R, count, dtype, op, nChannels, chunkBytes,
                               scratch, scratchBytes, stream=None):
    _check(_L().vr_allreduce_ring_stepwise(_ptrs(sendbufs), _ptrs(recvbufs), R, count, dtype, op,
                                           nChannels, chunkBytes, _ptr(scratch), scratchBytes,
                                           _stream(stream)), "vr_allreduce_ring_stepwise")


def vr_allreduce_ring_stepwise_noalloc(sendbufs, recvbufs, R, count, dtype, op, nChannels,
                                       chunkBytes, stream=None):
    """vr_allreduce_ring_stepwise without caller scratch: for callers that
    cannot allocate device memory (see include/vr.h)."""
    _check(_L().vr_allreduce_ring_stepwise_noalloc(_ptrs(sendbufs), _ptrs(recvbufs), R, count,
                                                   dtype, op, nChannels, chunkBytes,
                                                   _stream(stream)),
           "vr_allreduce_ring_stepwise_noalloc")


def _model(m):
    """None, a vr_cost_model_t, or ((alpha_ring, alpha_tree), (b_ring, b_tree))."""
    if m is None or isinstance(m, vr_cost_model_t):
        return m
    (a0, a1), (b0, b1) = m
    return vr_cost_model_t((ctypes.c_double * 2)(a0, a1), (ctypes.c_double * 2)(b0, b1))


def vr_predict_us(algo, R, localRanks, bytesPerRank, model=None):
    out = ctypes.c_double()
    m = _model(model)
    _check(_L().vr_predict_us(algo, R, localRanks, bytesPerRank,
                              ctypes.byref(m) if m is not None else None, ctypes.byref(out)),
           "vr_predict_us")
    return out.value


def vr_select_algo(R, localRanks, bytesPerRank, model=None):
    out = ctypes.c_int()
    m = _model(model)
    _check(_L().vr_select_algo(R, localRanks, bytesPerRank,
                               ctypes.byref(m) if m is not None else None, ctypes.byref(out)),
           "vr_select_algo")
    return out.value


def vr_fit_cost_model(R, localRanks, bytesPerRank, ringUs, treeUs):
    """Sequences of equal length; returns ((alpha_ring, alpha_tree),
    (per_byte_ring, per_byte_tree))."""
    n = len(R)
    D = ctypes.c_double
    out = vr_cost_model_t()
    _check(_L().vr_fit_cost_model(n, (I * n)(*R), (I * n)(*localRanks), (S * n)(*bytesPerRank),
                                  (D * n)(*ringUs), (D * n)(*treeUs), ctypes.byref(out)),
           "vr_fit_cost_model")
    return (tuple(out.alphaUs), tuple(out.usPerByte))


def vr_crossover_bytes(R, localRanks, model=None):
    """Bytes per rank where ring and tree predictions meet, or None."""
    out = ctypes.c_double()
    m = _model(model)
    _check(_L().vr_crossover_bytes(R, localRanks, ctypes.byref(m) if m is not None else None,
                                   ctypes.byref(out)), "vr_crossover_bytes")
    return None if out.value < 0 else out.value


def vr_set_cost_model(model=None):
    m = _model(model)
    _check(_L().vr_set_cost_model(ctypes.byref(m) if m is not None else None),
           "vr_set_cost_model")


def vr_jit_status():
    """(enabled, kernel sets compiled, failed) of the run-time specialised trees."""
    en, comp, fail = ctypes.c_int(), ctypes.c_longlong(), ctypes.c_longlong()
    _check(_L().vr_jit_status(ctypes.byref(en), ctypes.byref(comp), ctypes.byref(fail)),
           "vr_jit_status")
    return bool(en.value), comp.value, fail.value


def vr_jit_compile_dtree(nNodes, localRanks, dtype, op, smArch=103):
    """Compile-only: CUBIN bytes of the specialised kernels of the double
    binary tree of (nNodes, localRanks); raises VrError with the log."""
    size = ctypes.c_size_t()
    log = ctypes.create_string_buffer(8192)
    code = _L().vr_jit_compile_dtree(nNodes, localRanks, dtype, op, smArch, ctypes.byref(size),
                                     log, len(log))
    if code != 0:
        raise VrError(code, "vr_jit_compile_dtree: " + log.value.decode(errors="replace")[:2000])
    return size.value


def vr_jit_compile_ring(R, dtype, op, smArch=103):
    """Compile-only: CUBIN bytes of the specialised ring kernels for R ranks."""
    size = ctypes.c_size_t()
    log = ctypes.create_string_buffer(8192)
    code = _L().vr_jit_compile_ring(R, dtype, op, smArch, ctypes.byref(size), log, len(log))
    if code != 0:
        raise VrError(code, "vr_jit_compile_ring: " + log.value.decode(errors="replace")[:2000])
    return size.value


def vr_stream_status(stream=None):
    """Synchronises the stream and returns the device status code (0 = ok)."""
    return _L().vr_stream_status(_stream(stream))


def vr_launch_count():
    return _L().vr_launch_count()


def vr_debug_stall_next(tile):
    _check(_L().vr_debug_stall_next(tile), "vr_debug_stall_next")


def vr_debug_sched_slot(stream=None, words=None):
    """The four words of the tile scheduler slot of calls on ``stream``:
    returned when ``words`` is None, else written (four integers)."""
    buf = (ctypes.c_ulonglong * 4)(*(words or (0, 0, 0, 0)))
    _check(_L().vr_debug_sched_slot(_stream(stream), buf, 0 if words is None else 1),
           "vr_debug_sched_slot")
    return tuple(buf)


def vr_set_option(name, value):
    _check(_L().vr_set_option(name.encode(), int(value)), "vr_set_option")


def vr_get_option(name):
    v = ctypes.c_longlong()
    _check(_L().vr_get_option(name.encode(), ctypes.byref(v)), "vr_get_option")
    return v.value


def vr_get_error_string(code):
    return _L().vr_get_error_string(code).decode()


def vr_finalize():
    _L().vr_finalize()


def vr_debug_bounds_checked():
    return bool(_L().vr_debug_bounds_checked())


def vr_debug_shrink_next(nbytes, which=3):
    _check(_L().vr_debug_shrink_next(nbytes, which), "vr_debug_shrink_next")


def vr_debug_bounds_fault():
    v = ctypes.c_ulonglong()
    _check(_L().vr_debug_bounds_fault(ctypes.byref(v)), "vr_debug_bounds_fault")
    return v.value


def vr_debug_access_ok(extents, p, size, store):
    """extents: (lo, bytes, writable) triples; returns the C result (1, 0, -1)."""
    n = len(extents)
    lo = (VP * max(n, 1))(*[e[0] for e in extents])
    by = (ctypes.c_ulonglong * max(n, 1))(*[e[1] for e in extents])
    wr = (I * max(n, 1))(*[int(e[2]) for e in extents])
    return _L().vr_debug_access_ok(lo, by, wr, n, p, size, int(store))
