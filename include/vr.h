/*
 * vr.h -- emulated Ring / Double-Binary-Tree AllReduce on one GPU.
 *
 * R "virtual ranks" are R device buffers in one GPU's memory.  The library
 * computes what an AllReduce (ReduceScatter, AllGather) over R ranks
 * computes, following the ring and double-binary-tree schedules, and writes
 * every rank's result buffer.  Each fused collective call is one kernel
 * launch on the caller's stream (the host-buffer and non-fused variants
 * enqueue several); nothing crosses a GPU or process boundary.
 *
 * Sources (web pages), cited below as [tag] "section":
 *   [Course13]  "NCCL 专家课程 13：Tree、双树、层次化连接与真实交叉区间" (blog.cptz.space)
 *   [Internals] "NCCL 内部机制：一次 AllReduce 如何变成拓扑图、Channel 与 GPU Kernel"
 *               (charlestar.github.io)
 *   [CodeNotes] "NCCL代码分析" (jianzi123.github.io)
 *   [Interview] "all-reduce 每张卡要发多少数据? ring 和 tree 有什么区别?"
 *               (charliedreemur.github.io)
 *
 * Conventions shared by every call
 *   - All functions are thread-safe.  They return VR_SUCCESS or an error code;
 *     argument errors are detected on the host before anything is enqueued.
 *   - Buffers are owned by the caller.  The pointer arrays are read during the
 *     call only (their contents are passed to the kernel by value), so the
 *     caller may reuse or free the arrays as soon as the call returns.
 *   - Collective calls are asynchronous on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream): returning means enqueued, not completed
 *     ([Internals] "API 返回只意味着提交边界，不意味着数据已经可读").  Read the
 *     result only after synchronising the stream or through a stream-ordered
 *     dependency.
 *   - The library allocates no device buffers at run time.  Its own device
 *     state is static: one status word and one bounds word per device and
 *     the 8 MiB FIFO of vr_allreduce_ring_stepwise_noalloc (__device__
 *     variables), plus the code
 *     of kernels compiled at run time (vr_jit_status) and, once
 *     vr_allreduce_host has run on a device, two streams and four events
 *     there.  vr_finalize releases what is not static.
 *   - Reductions accumulate in fp32 for every dtype and narrow to the element
 *     type once, round-to-nearest-even.  Sum is IEEE fp32 addition in the
 *     schedule's order; Max returns the larger value, with +0 above -0.
 *   - Results are deterministic: the same call on the same inputs gives the
 *     same bits, and every rank's output is bit-identical.
 *
 * Options, for tests and tuning (no option changes a result, only which
 * kernel computes it, or what the library prints).  Each is read from the
 * environment once, at the first call that needs an option, and changed
 * afterwards only through vr_set_option (same names and values):
 *   VR_KERNEL_PATH=staged|register  force the shared-memory-staged or the
 *                                   register-path AllReduce / ReduceScatter
 *                                   kernel (aligned buffers); vr_set_option
 *                                   takes 2 or 1 (0: automatic)
 *   VR_JIT=0                        interpreting tree / ring folds only
 *   VR_JIT_RING=0|1                 ring folds specialised: never / also on
 *                                   the staged kernel
 *   VR_SMALL_RANKS=0                no few-rank register-path variant
 *   VR_SPREAD=0                     256-thread CTAs even when a small call
 *                                   would leave SMs idle
 *   VR_JIT_OCC=0|4                  specialised register-path kernels at
 *                                   four CTAs per SM: never / always (by
 *                                   default a tree call takes them when
 *                                   each thread folds at most three units
 *                                   and the larger grid saves every thread
 *                                   one)
 *   VR_PDL=0                        launch without programmatic stream
 *                                   serialisation (by default a kernel may
 *                                   start while the previous one on the
 *                                   stream drains; it waits for it before
 *                                   touching memory)
 *   VR_STAGED_MIN_BYTES=n           staged kernel from n bytes per rank
 *                                   (default 16 MiB; 2-7 ranks: from the
 *                                   larger of n and 32 MiB; trees that draw
 *                                   their tiles (VR_SCHED): above 8 ranks
 *                                   from n / 2, 5-7 ranks from the larger
 *                                   of n and 24 MiB)
 *   VR_STAGED_TILE_BYTES, VR_STAGED_STAGES, VR_STAGED_MIN_STAGES
 *                                   staged geometry: bytes per rank per
 *                                   tile, most stages, fewest stages
 *   VR_AG_TILE, VR_AG_STAGES, VR_AG_CTAS
 *                                   TMA AllGather geometry (pairs of tile
 *                                   and stages that are compiled: 8192/4,
 *                                   8192/8, 16384/4, 16384/6, 32768/3,
 *                                   4096/8; others are INVALID_ARGUMENT)
 *   VR_AG_ORDER=1|2                 TMA AllGather tile order: source-major
 *                                   (each loaded tile stored to all R
 *                                   outputs) / destination-major (each
 *                                   output written in long runs, sources
 *                                   re-read from L2); by default
 *                                   destination-major when the R sources
 *                                   take at most a quarter of L2
 *   VR_SCHED=0|1|2                  staged AllReduce: 0 every CTA takes a
 *                                   fixed run of tiles; 1 (default) the
 *                                   CTAs draw tiles at run time where that
 *                                   measured faster (trees of 4 or more
 *                                   ranks, 8 excepted; rings of 16 or
 *                                   more, and fp32 rings of 4 and of 9
 *                                   or more);
 *                                   2 always drawn.
 *                                   Drawing uses a scheduler slot in
 *                                   device memory per stream, and one per
 *                                   launch captured into a graph: launches
 *                                   on one stream, and the replays of one
 *                                   instantiated graph, run one after
 *                                   another.  Two instances of one captured
 *                                   graph running at the same time share
 *                                   the captured launch's slot; the later
 *                                   one's CTAs wait (bounded) and report
 *                                   VR_ERR_TIMEOUT if it stays held (a
 *                                   slot so left held fails later drawing
 *                                   calls on it the same way until
 *                                   vr_debug_sched_slot frees it).
 *                                   Slots per device: 1024 streams and
 *                                   3072 captured launches; past them,
 *                                   fixed runs.  The same bits either way.
 *   VR_DEBUG=GRAPH                  print every tree set, ring and channel
 *                                   partition a call plans to stderr, in
 *                                   the log formats of [Course13] "从 GRAPH
 *                                   日志复原 active tree" (vr_set_option
 *                                   takes 1)
 * Read once at first use, not changeable:
 *   VR_WAIT_TIMEOUT_NS=n            limit of every bounded wait
 *                                   (default 1 s)
 *   VR_VALIDATE_POINTERS=1          check that every buffer is reachable
 *                                   from the current device
 */
#ifndef VR_H
#define VR_H

#ifndef __CUDACC_RTC__
#include <stddef.h>
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  VR_SUCCESS = 0,
  VR_ERR_INVALID_ARGUMENT = 1, /* bad size, pointer, overlap or enum value */
  VR_ERR_UNSUPPORTED = 2,      /* valid arguments, combination not offered  */
  VR_ERR_CUDA = 3,             /* a CUDA runtime call failed                */
  VR_ERR_TIMEOUT = 4,          /* a bounded device-side wait ran out        */
  VR_ERR_INTERNAL = 5          /* a library invariant failed (bounds fault) */
} vr_result_t;

typedef enum { VR_FLOAT32 = 0, VR_FLOAT16 = 1, VR_BFLOAT16 = 2 } vr_dtype_t;
typedef enum { VR_SUM = 0, VR_MAX = 1 } vr_op_t;
/* VR_ALGO_AUTO (AllReduce only): ring or tree, whichever the cost model
 * (vr_select_algo) predicts faster. */
typedef enum { VR_ALGO_RING = 0, VR_ALGO_TREE = 1, VR_ALGO_AUTO = 2 } vr_algo_t;

#define VR_MAX_RANKS 64
#define VR_MAX_CHANNELS 64

/* One rank's view of one tree: the ncclTree record of [Course13]
 * "数据结构不是纯二叉树".  up = parent rank (-1 at the root); down[] = child
 * ranks, present children first, empty slots -1; depth = the approximation
 * localRanks - 1 + floor(log2(nNodes)) of [Course13] "节点间连接". */
typedef struct {
  int depth;
  int up;
  int down[3];
} vr_tree_t;

/* ------------------------------------------------------------ topology */

/* Identity ring of every channel ([Interview] "先弄清楚": each rank sends to
 * its right-hand neighbour).  next[c*R + r] = (r+1) mod R and
 * prev[c*R + r] = (r-1) mod R for c < nChannels.  `next` and `prev` are
 * caller-owned host arrays of nChannels*R ints.
 * Errors: VR_ERR_INVALID_ARGUMENT for R outside [1, VR_MAX_RANKS], nChannels
 * outside [1, VR_MAX_CHANNELS] or a NULL array. */
vr_result_t vr_build_ring(int R, int nChannels, int* next, int* prev);

/* Hierarchical double binary tree over R = nNodes*localRanks ranks
 * ([Course13] "节点内先形成链", "节点间连接", "Btree 的 bit 构造",
 * "双树：偶数 mirror，奇数 shift").  Within a node the ranks k*L .. k*L+L-1
 * form a chain (up = previous, down[0] = next).  Over node indices, tree 0 is
 * the bit-trick binary tree and tree 1 its mirror (even nNodes) or its
 * one-step shift (odd nNodes); the head k*L of node k takes up = head of its
 * parent node and appends the heads of its child nodes to down[].
 * Channels [0, ceil(nChannels/2)) carry tree 0, the others tree 1.
 * `trees` is a caller-owned host array of nChannels*R records,
 * trees[c*R + r].  localRanks = 1 gives the flat double binary tree.
 * Errors: VR_ERR_INVALID_ARGUMENT for R outside [1, VR_MAX_RANKS], nNodes or
 * localRanks < 1, nChannels outside [1, VR_MAX_CHANNELS], NULL `trees`. */
vr_result_t vr_build_dtree(int nNodes, int localRanks, int nChannels, vr_tree_t* trees);

/* Which rank of a node's intra order joins the node-level tree
 * ([Course13] "节点内先形成链"): the parent head is always the first; the
 * heads that take child nodes d0 / d1 are the first / first (TREE), the
 * second / second (SPLIT_TREE) or the second / first (BALANCED_TREE). */
typedef enum {
  VR_PATTERN_TREE = 0,
  VR_PATTERN_SPLIT_TREE = 1,
  VR_PATTERN_BALANCED_TREE = 2
} vr_tree_pattern_t;

/* vr_build_dtree with a head pattern and per-channel intra-node orders
 * ([Course13] "节点内先形成链": the chain follows treeIntra, which a topology
 * search may order differently per channel; "本机真实树形" shows such
 * channels).  intraOrders: NULL (identity) or nChannels*localRanks ints, row
 * c a permutation of 0..localRanks-1 giving channel c's chain order inside
 * every node.  The parent head of node k takes up = the child0 or child1
 * head of its parent node (by k's parentChildType in the node-level tree);
 * the child0 head appends child node d0's parent head, then the child1 head
 * appends d1's.  Errors: those of vr_build_dtree, plus
 * VR_ERR_INVALID_ARGUMENT for a bad pattern, SPLIT_TREE / BALANCED_TREE
 * with one local rank, or a row that is not a permutation. */
vr_result_t vr_build_dtree_ex(int nNodes, int localRanks, int nChannels,
                              vr_tree_pattern_t pattern, const int* intraOrders,
                              vr_tree_t* trees);

/* Channel c's element range of a message of `count` elements ([Course13]
 * "前置知识": channels take different ranges of one message).  The message
 * is cut into 16-byte grains, split over channels so that the first
 * (grains mod nChannels) channels get one more grain, and clipped at count.
 * Writes *offset and *channelCount (elements).
 * Errors: VR_ERR_INVALID_ARGUMENT for a bad dtype, nChannels outside
 * [1, VR_MAX_CHANNELS], channel outside [0, nChannels) or NULL outputs. */
vr_result_t vr_partition(size_t count, vr_dtype_t dtype, int nChannels, int channel,
                         size_t* offset, size_t* channelCount);

/* Ring block of element `elem` in the ring AllReduce partition, which fixes
 * the order in which the element is reduced ([Interview] "手撕代码": the
 * block leaves rank j first and each later rank adds its copy).  A channel is
 * walked in loops of R*C elements (C = chunkBytes / element size), the last
 * loop shorter; each loop is cut into R blocks, the first (loop mod R) one
 * element longer.  Writes *channel and *block (the block number j).
 * Errors: VR_ERR_INVALID_ARGUMENT for elem >= count or the argument errors
 * of vr_allreduce. */
vr_result_t vr_ring_block(size_t count, vr_dtype_t dtype, int R, int nChannels,
                          size_t chunkBytes, size_t elem, int* channel, int* block);

/* --------------------------------------------------------- collectives */

/* AllReduce: every recvbufs[r] (count elements) receives the reduction over
 * r' < R of sendbufs[r'] ([Internals] "从 API 调用到可调度任务": two buffers,
 * count, dtype, op, communicator and stream).
 *   RING ([Interview] "手撕代码", [Internals] "Ring：带宽友好"): an element in
 *        block j of its ring loop is reduced over ranks j, j+1, ..., j+R-1
 *        (mod R), left to right -- reduce-scatter followed by all-gather.
 *   TREE ([Course13] "先固定方向", "runTreeSplit 如何流水", "每种 rank 的操作"):
 *        on the channel's tree every rank folds its local input with its
 *        children's partials in down[] order and passes the result up; the
 *        root's value is broadcast down to all ranks.  localRanks = 1 here.
 *   AUTO the one of the two that vr_select_algo predicts faster.
 * nChannels in [1, VR_MAX_CHANNELS] splits the message (vr_partition);
 * chunkBytes (a positive multiple of 16) is the per-rank chunk C of a ring
 * loop and the chunk of a tree channel.
 * In place: sendbufs[r] == recvbufs[r] is allowed.
 * Buffers: any alignment.  16-byte aligned buffers run 16-byte units: from
 * 16 MiB per rank the ring and the tree with 8..64 ranks (the tree with
 * 9..64 ranks from 8 MiB), and from 32 MiB per rank those with 2..7 ranks
 * (the tree with 5..7 from 24 MiB; not the ring of 6), run on a kernel that
 * stages each tile of all R ranks in shared memory with bulk asynchronous
 * copies (the tree's fold specialised at run time, see vr_jit_status),
 * everything else on a kernel that loads the ranks' units into registers
 * (rings of at most 64 Ki elements per rank: one element per thread).  The
 * ring of two ranks runs the tree kernels (two operands fold to the same bits
 * in either order).  The option VR_KERNEL_PATH (staged|register; see the top
 * of this header) forces one of the two for testing and tuning; results are
 * identical.  Unaligned buffers run element units on the register kernel.
 * Errors (nothing enqueued): VR_ERR_INVALID_ARGUMENT for R outside
 * [1, VR_MAX_RANKS], NULL arrays, a NULL buffer with count > 0, a buffer not
 * aligned to the element size, a bad enum, bad nChannels or chunkBytes, or a
 * recv buffer that overlaps another rank's send or recv buffer or partly
 * overlaps its own send buffer.
 * count == 0 enqueues nothing.  R == 1 copies (or leaves in place). */
vr_result_t vr_allreduce(const void* const* sendbufs, void* const* recvbufs, int R,
                         size_t count, vr_dtype_t dtype, vr_op_t op, vr_algo_t algo,
                         int nChannels, size_t chunkBytes, void* stream);

/* vr_allreduce with a hierarchical rank layout: R = nNodes * localRanks,
 * node k holding ranks k*localRanks .. (k+1)*localRanks - 1.  TREE uses the
 * trees of vr_build_dtree(R / localRanks, localRanks, nChannels); RING is the
 * same as vr_allreduce.  Extra error: localRanks < 1 or not dividing R. */
vr_result_t vr_allreduce_ex(const void* const* sendbufs, void* const* recvbufs, int R,
                            size_t count, vr_dtype_t dtype, vr_op_t op, vr_algo_t algo,
                            int nChannels, size_t chunkBytes, int localRanks, void* stream);

/* vr_allreduce_ex on HOST buffers, pipelined through a device workspace.
 * [Internals] "API 返回只意味着提交边界": the call enqueues and returns; here
 * the enqueued work also moves the data in and out.  The message is cut into
 * pieces of pieceBytes per rank (0: VR_HOST_PIECE_BYTES; else a multiple of
 * 16).  Piece p is copied in to workbufs on one internal stream, folded in
 * place there on `stream`, and copied out to recvbufs on another internal
 * stream, so copies in both directions overlap the fold of other pieces.
 * The result equals vr_allreduce_ex's bit for bit: an element's fold reads
 * only that element of each rank, in the order the whole message's
 * partition gives it.
 *   sendbufs[r], recvbufs[r]: host memory, count elements; page-locked for
 *     the copies to overlap (pageable memory works, serialised); in place
 *     (recvbufs[r] == sendbufs[r]) allowed.  They must stay valid, and
 *     sendbufs unchanged, until `stream` has passed this call.
 *     recvbufs[r] may be NULL: rank r's result is then not copied out and
 *     stays in workbufs[r] only (every rank's result is the same vector, so
 *     a caller that needs one copy on the host names one receive buffer).
 *   workbufs[r]: device memory of the current device, count elements each,
 *     owned by the caller; overwritten.
 *   stream: nothing is copied in before the caller's earlier work on it is
 *     done, and work the caller enqueues on it after this call waits for the
 *     last copy out.
 * The internal streams and events are created per device on first use and
 * destroyed by vr_finalize.  Calls from several threads are serialised on
 * the host.  Errors as vr_allreduce_ex, plus VR_ERR_INVALID_ARGUMENT for a
 * NULL workbufs, a pieceBytes not a multiple of 16, a workspace buffer that
 * is not device memory of the current device, or a host buffer that is
 * device memory. */
#define VR_HOST_PIECE_BYTES ((size_t)8 << 20)
vr_result_t vr_allreduce_host(const void* const* sendbufs, void* const* recvbufs, int R,
                              size_t count, vr_dtype_t dtype, vr_op_t op, vr_algo_t algo,
                              int nChannels, size_t chunkBytes, int localRanks,
                              void* const* workbufs, size_t pieceBytes, void* stream);

/* Tree AllReduce over caller-given trees: channel c folds every element over
 * trees[c*R .. c*R + R-1] (vr_tree_t records, e.g. from vr_build_dtree_ex)
 * in the order of vr_allreduce's TREE: each rank folds its local input with
 * its children's partials in down[] order, the root's value goes to every
 * rank.  Each channel's records must form one tree over the R ranks: up and
 * down[] agree both ways, down[] has its present children first, one root,
 * every rank reaches it.  At most 16 distinct trees per call.  Host-side
 * errors: those of vr_allreduce, VR_ERR_INVALID_ARGUMENT for a NULL or
 * invalid tree, VR_ERR_UNSUPPORTED for more than 16 distinct trees or a tree
 * whose fold keeps more than 8 partials live. */
vr_result_t vr_allreduce_trees(const void* const* sendbufs, void* const* recvbufs, int R,
                               size_t count, vr_dtype_t dtype, vr_op_t op, int nChannels,
                               size_t chunkBytes, const vr_tree_t* trees, void* stream);

/* ReduceScatter ([Interview] "先弄清楚": each rank keeps the reduced 1/n
 * segment it is responsible for): sendbufs[r] holds R*recvcount elements;
 * recvbufs[b] (recvcount elements) receives block b = elements
 * [b*recvcount, (b+1)*recvcount) reduced over all ranks, in ring order
 * b+1, b+2, ..., b (mod R).  Only VR_ALGO_RING: tree implements AllReduce
 * only ([CodeNotes] "通讯时如何选择Channel"), so VR_ALGO_TREE returns
 * VR_ERR_UNSUPPORTED.  In place: recvbufs[r] == sendbufs[r] + r*recvcount
 * (in elements).  fp32 with 2..8 ranks from 16 MiB sent per rank runs the
 * shared-memory-staged kernel (64 KB stages), everything else the register
 * kernel.  Other errors as vr_allreduce. */
vr_result_t vr_reduce_scatter(const void* const* sendbufs, void* const* recvbufs, int R,
                              size_t recvcount, vr_dtype_t dtype, vr_op_t op,
                              vr_algo_t algo, int nChannels, size_t chunkBytes,
                              void* stream);

/* AllGather ([Interview] "先弄清楚": the segments are concatenated back):
 * recvbufs[q] (R*sendcount elements) receives sendbufs[r] (sendcount
 * elements) at elements [r*sendcount, (r+1)*sendcount) for every r -- an exact
 * copy.  Only VR_ALGO_RING (VR_ALGO_TREE: VR_ERR_UNSUPPORTED).  In place:
 * sendbufs[r] == recvbufs[r] + r*sendcount.  Other errors as vr_allreduce. */
vr_result_t vr_allgather(const void* const* sendbufs, void* const* recvbufs, int R,
                         size_t sendcount, vr_dtype_t dtype, vr_algo_t algo,
                         int nChannels, size_t chunkBytes, void* stream);

/* ------------------------------------------------ non-fused variants
 * Same results as the fused calls above, computed the way a schedule that
 * moves messages between ranks does, to measure what fusion buys. */

/* Two-phase tree AllReduce ([Course13] "当前环境命中哪个 device 实现":
 * runTreeUpDown reduces the whole message up the tree before broadcasting it
 * down; runTreeSplit overlaps the two).  First launch: every unit is folded
 * over its channel's tree and stored to the tree root's receive buffer only;
 * second launch: copied from there to every other rank.  Same arguments,
 * errors and bits as vr_allreduce_ex with VR_ALGO_TREE; one more read and
 * write of the message.  Two kernel launches. */
vr_result_t vr_allreduce_tree_updown(const void* const* sendbufs, void* const* recvbufs, int R,
                                     size_t count, vr_dtype_t dtype, vr_op_t op, int nChannels,
                                     size_t chunkBytes, int localRanks, void* stream);

/* Bytes of device scratch vr_allreduce_ring_stepwise needs: count elements
 * of dtype, rounded up to 16 (0 for a bad dtype). */
size_t vr_ring_stepwise_scratch_bytes(size_t count, vr_dtype_t dtype);

/* Stepwise ring AllReduce ([Interview] "手撕代码"; [Internals] "Ring：带宽友好"):
 * the ring's 2(R-1) steps run one after the other, each as two launches, and
 * every message crosses device memory: each step first copies every rank's
 * outgoing block (of every loop) into the caller's scratch FIFO, then folds
 * the FIFO into the receiving rank's block (reduce-scatter half) or
 * overwrites it (all-gather half).  recvbufs[r] is rank r's working copy
 * (first set to sendbufs[r]) and keeps partials in the element type, so
 * 16-bit partials are rounded (RNE) at every hop, as messages that travel in
 * that type are; for fp32 and for Max the bits equal vr_allreduce's RING.
 * `scratch` is caller-owned device memory of at least
 * vr_ring_stepwise_scratch_bytes(count, dtype) bytes, aligned to the element
 * size, that overlaps no buffer; its contents are overwritten.  Launches 1 + 4(R-1) kernels.
 * Errors: those of vr_allreduce, plus VR_ERR_INVALID_ARGUMENT for a NULL,
 * short, misaligned or overlapping scratch. */
vr_result_t vr_allreduce_ring_stepwise(const void* const* sendbufs, void* const* recvbufs, int R,
                                       size_t count, vr_dtype_t dtype, vr_op_t op,
                                       int nChannels, size_t chunkBytes, void* scratch,
                                       size_t scratchBytes, void* stream);

/* Size of the device array that vr_allreduce_ring_stepwise_noalloc uses as
 * its message FIFO: 8 MiB per GPU that loads the library. */
#define VR_NOALLOC_SCRATCH_BYTES (8u << 20)

/* vr_allreduce_ring_stepwise for callers that cannot allocate device memory
 * (no counterpart in the pages: it exists for the callers, not the method).
 * A runtime that has given all of the GPU's memory to its own allocator, or
 * code on a latency-critical path that may not call cudaMalloc / cudaFree
 * (both can synchronise the device), cannot supply the scratch FIFO; this
 * entry point uses a file-scope device array of VR_NOALLOC_SCRATCH_BYTES
 * bytes instead, which every GPU that loads the library holds until the
 * process exits.  It allocates nothing, and calls neither cudaMalloc nor
 * cudaFree nor any allocating library routine.
 * Arguments, results and errors are those of vr_allreduce_ring_stepwise
 * without scratch/scratchBytes, plus VR_ERR_UNSUPPORTED when count elements
 * of dtype exceed VR_NOALLOC_SCRATCH_BYTES (2 Mi fp32 or 4 Mi 16-bit
 * elements per rank at most).
 * Arguments are checked first (VR_ERR_INVALID_ARGUMENT as for the other
 * entry point), the size limit after them.
 * Set-up: the first call on a device looks up the array's device address on
 * that device (the device current at the call).  CUDA loads modules lazily,
 * so that first call is also when the device's copy of the array is
 * created: make it before any stream capture, and before the caller's own
 * allocator takes the device's memory (else it can fail with
 * VR_ERR_CUDA).  A call with count == 0 does nothing, set-up included.
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents; nothing in it needs to start at zero (each step writes
 * every message before it is read).  Calls whose executions overlap on the
 * GPU (different streams, or different host threads) race on the array:
 * order them. */
vr_result_t vr_allreduce_ring_stepwise_noalloc(const void* const* sendbufs, void* const* recvbufs,
                                               int R, size_t count, vr_dtype_t dtype, vr_op_t op,
                                               int nChannels, size_t chunkBytes, void* stream);

/* ---------------------------------------------------------- cost model
 * The pages' alpha-beta model ([Course13] "理想成本模型"; [Interview]
 * "推导 / 关键公式"), with N ranks, tree depth D (the deeper of the two
 * trees, edges from root to deepest leaf) and M bytes per rank:
 *   T_ring = 2(N-1) * alpha[0] + 2(N-1)/N * M * usPerByte[0]
 *   T_tree = 2D     * alpha[1] + 2 M       * usPerByte[1]
 * in microseconds.  The built-in model is fitted (least squares of relative
 * error) to the ring and tree times this library measures on GB300 for
 * 4 ranks, 8 B .. 256 MiB per rank. */
typedef struct {
  double alphaUs[2];    /* per dependent stage: [0] ring, [1] tree */
  double usPerByte[2];  /* per byte of the traffic term: [0] ring, [1] tree */
} vr_cost_model_t;

/* Predicted time of an AllReduce (algo RING or TREE) over R ranks in nodes of
 * localRanks, bytesPerRank each, under `model` (NULL: the current model).
 * Errors: VR_ERR_INVALID_ARGUMENT for a bad algo, R, localRanks or NULL us. */
vr_result_t vr_predict_us(vr_algo_t algo, int R, int localRanks, size_t bytesPerRank,
                          const vr_cost_model_t* model, double* us);

/* The algorithm with the smaller prediction (RING on a tie); what
 * VR_ALGO_AUTO uses with model NULL.  Errors as vr_predict_us. */
vr_result_t vr_select_algo(int R, int localRanks, size_t bytesPerRank,
                           const vr_cost_model_t* model, vr_algo_t* algo);

/* Fits the model to measured AllReduce times: sample i ran R[i] ranks in
 * nodes of localRanks[i], bytesPerRank[i] each, in ringUs[i] and treeUs[i]
 * microseconds (a value <= 0 leaves that algorithm's sample out).  For each
 * algorithm, (alphaUs, usPerByte) minimises the sum of squared relative
 * errors (predicted / measured - 1)^2, so that short and long messages count
 * alike -- the pages give the model's form, not its constants.  On noisy data
 * a fitted parameter can come out negative (vr_set_cost_model refuses it).
 * Errors: VR_ERR_INVALID_ARGUMENT for n < 2, NULL arrays, a bad R /
 * localRanks, or fewer than two usable samples (or a singular system) for an
 * algorithm. */
vr_result_t vr_fit_cost_model(int n, const int* R, const int* localRanks,
                              const size_t* bytesPerRank, const double* ringUs,
                              const double* treeUs, vr_cost_model_t* out);

/* The message size per rank at which the ring and tree predictions are equal
 * under `model` (NULL: the current model), from the closed form of the two
 * lines; *bytes = -1 when they do not cross at a positive size.  Errors as
 * vr_predict_us. */
vr_result_t vr_crossover_bytes(int R, int localRanks, const vr_cost_model_t* model,
                               double* bytes);

/* Installs `model` as the current model for this process (NULL restores the
 * built-in one), e.g. one fitted to other hardware.  Errors:
 * VR_ERR_INVALID_ARGUMENT for negative or non-finite entries. */
vr_result_t vr_set_cost_model(const vr_cost_model_t* model);

/* ------------------------------------------ run-time specialised trees
 * Tree AllReduce on 16-byte aligned buffers runs kernels compiled at run time
 * (NVRTC, opened with dlopen) for the call's trees: the fold program of each
 * tree ([Course13] "每种 rank 的操作", post-order) becomes straight-line code
 * instead of an interpreted control stream, with the same operations in the
 * same order, so results are unchanged.  Kernels are cached per architecture,
 * element type, op and set of trees; the first call with new trees compiles
 * them (about a second).  Without NVRTC, without the kernel sources beside
 * the library, or with the option VR_JIT=0 (see the top of this header), the
 * built-in interpreting kernels run. */

/* Whether specialised trees are in use, and how many kernel sets were
 * compiled and failed to compile or load so far.  Errors:
 * VR_ERR_INVALID_ARGUMENT for a NULL output. */
vr_result_t vr_jit_status(int* enabled, long long* compiled, long long* failed);

/* Compiles, without loading or touching a device, the specialised kernels of
 * vr_build_dtree(nNodes, localRanks, 2)'s two trees for sm_<smArch>a (e.g.
 * 103) -- register path, staged, staged drawing its tiles (VR_SCHED) -- and
 * returns their total CUBIN size; the compiler log, if any, goes to `log`
 * (logBytes, NUL-terminated, may be NULL / 0).  Errors:
 * VR_ERR_INVALID_ARGUMENT for bad sizes, dtype, op or smArch < 90;
 * VR_ERR_UNSUPPORTED when NVRTC or the kernel sources are not found;
 * VR_ERR_INTERNAL when the compilation fails. */
vr_result_t vr_jit_compile_dtree(int nNodes, int localRanks, vr_dtype_t dtype, vr_op_t op,
                                 int smArch, size_t* cubinBytes, char* log, size_t logBytes);

/* The same for the ring fold of R ranks (register-path and staged kernels):
 * the R ranks' units loaded in rank order, block j's rotation folded from
 * them ([Interview] "手撕代码": block j starts at rank j), one straight-line
 * case per j.  Register-path ring kernels of 16-byte aligned buffers with
 * 3 <= R <= 16 use it (measured 6-12% faster; neutral on the staged kernel,
 * which keeps the loop); the environment variable VR_JIT_RING=0 (read per
 * call) turns it off, VR_JIT_RING=1 also applies it to the staged kernel.
 * Errors as
 * vr_jit_compile_dtree (R outside [1, VR_MAX_RANKS]: invalid). */
vr_result_t vr_jit_compile_ring(int R, vr_dtype_t dtype, vr_op_t op, int smArch,
                                size_t* cubinBytes, char* log, size_t logBytes);

/* ------------------------------------------------------------- status */

/* Synchronises `stream`, then returns and clears the current device's status
 * word: VR_SUCCESS, or the first device-side error any kernel of this library
 * recorded since the last call (VR_ERR_TIMEOUT for a bounded wait that ran
 * out, VR_ERR_INTERNAL for a broken invariant: in the bounds-checked build,
 * an access outside the call's buffers, refused), or VR_ERR_CUDA when the
 * synchronisation itself fails.  The word is per device, not per stream. */
vr_result_t vr_stream_status(void* stream);

/* Number of kernels this library has launched in this process (all devices,
 * all threads). */
unsigned long long vr_launch_count(void);

/* Test hook for the device-side failure path.  The next collective call
 * that runs a shared-memory-staged kernel (16-byte aligned AllReduce or
 * ReduceScatter) or the TMA AllGather makes its first CTA skip the loads of
 * its tile number
 * `tile`, so the wait for that tile runs out after the bounded-wait limit
 * (1 s, or VR_WAIT_TIMEOUT_NS nanoseconds from the environment at first
 * use): that call's results are incomplete and vr_stream_status reports
 * VR_ERR_TIMEOUT; the stream and the context stay usable.  -1 cancels a
 * pending request.  Errors: VR_ERR_INVALID_ARGUMENT for tile < -1. */
vr_result_t vr_debug_stall_next(long long tile);

/* Test hook for the tile scheduler of the staged AllReduce kernels (see
 * VR_SCHED): reads (write = 0) or writes (write != 0) the four words of the
 * scheduler slot that calls on `stream` use -- owner (0 when free), next
 * tile, and the CTAs that joined (low 32 bits) and left (high 32 bits) --
 * through a copy on `stream`, which is then synchronised.  A slot whose owner
 * is set to a value no launch has makes the next call's CTAs wait for it
 * (bounded) and report VR_ERR_TIMEOUT; writing four zeros frees it.
 * `words` is host memory of 4 elements.  Errors: VR_ERR_INVALID_ARGUMENT
 * (null words, or a stream being captured), VR_ERR_UNSUPPORTED (no slot
 * left for a new stream), VR_ERR_CUDA. */
vr_result_t vr_debug_sched_slot(void* stream, unsigned long long* words, int write);

/* Sets one of the options listed at the top of this header for the rest of
 * the process (all threads, all devices); value -1 restores the built-in
 * default.  Calls already enqueued are not affected.  Meant for tests and
 * tuning: options choose among kernels that compute the same bits.
 * Errors: VR_ERR_INVALID_ARGUMENT for an unknown name or value < -1. */
vr_result_t vr_set_option(const char* name, long long value);

/* The current value of an option (-1: the call site's built-in default).
 * Errors: VR_ERR_INVALID_ARGUMENT for an unknown name or NULL value. */
vr_result_t vr_get_option(const char* name, long long* value);

/* ------------------------------------------------ bounds-checked build
 * The library's calls return at enqueue, so a kernel's fault would surface
 * later and asynchronously ([Internals] "API 返回只意味着提交边界").  The
 * bounds-checked build of this library (libvr_debug.so, built by
 * double_binary_tree_gb300.build with debug=True; loaded by the Python
 * binding when VR_BOUNDS_CHECKED=1) compiles every global-memory access of
 * every kernel with a check against the buffers of its call: the send and
 * receive buffers (count elements, or the collective's sizes) and the
 * stepwise ring's FIFO.  An access outside them (a store outside the
 * receive buffers and the FIFO) is skipped, VR_ERR_INTERNAL is recorded in
 * the status word (vr_stream_status) and the first such address in a second
 * device word.  Results and performance of the normal build are unchanged:
 * there the checks compile to nothing. */

/* 1 in the bounds-checked build, 0 in the normal one. */
int vr_debug_bounds_checked(void);

/* The first address the bounds-checked build refused on the current device
 * since the last call (0: none), then cleared.  Errors: VR_ERR_INVALID_ARGUMENT
 * for NULL address, VR_ERR_CUDA when the device cannot be read. */
vr_result_t vr_debug_bounds_fault(unsigned long long* address);

/* Test hook of the bounds-checked build: the next kernel launch records some
 * of its buffers as ending `bytes` earlier than they do (`which`: 1 the
 * send buffers, 2 the receive buffers, 4 the FIFO, or a sum), so the checks
 * refuse its last accesses to them while every access still lies inside
 * real memory: refused loads read zeros (a refused bulk copy into shared
 * memory completes its barrier without copying), refused stores are not
 * made, and vr_stream_status reports VR_ERR_INTERNAL.  No effect in the
 * normal build.  bytes == 0 cancels a pending request.
 * Errors: VR_ERR_INVALID_ARGUMENT for bytes < 0 or which outside 0..7. */
vr_result_t vr_debug_shrink_next(long long bytes, int which);

/* The bounds predicate of the device checks, run on the host (for tests):
 * 1 when [p, p + size) lies inside one of the n extents [lo[i], lo[i] +
 * bytes[i]) -- a writable one (writable[i] != 0) when store != 0 -- else 0;
 * -1 for bad arguments (n < 0, n > 129, NULL arrays with n > 0).  NULL
 * extents never match.  Touches no memory at p. */
int vr_debug_access_ok(const void* const* lo, const unsigned long long* bytes,
                       const int* writable, int n, const void* p, unsigned long long size,
                       int store);

/* Static English text for a result code ("unknown result" for others). */
const char* vr_get_error_string(vr_result_t result);

/* Releases host-side caches (tree programs, device properties).  Optional;
 * the library stays usable afterwards. */
void vr_finalize(void);

#ifdef __cplusplus
}
#endif

#endif /* VR_H */
