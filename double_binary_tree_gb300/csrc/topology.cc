// Ring and double-binary-tree topology of the emulated ranks, and the fold
// programs the tree kernel executes.
//
// Sources (web pages):
//   [Course13] "NCCL 专家课程 13：Tree、双树、层次化连接与真实交叉区间" (blog.cptz.space),
//     sections "数据结构不是纯二叉树" (ncclTree record), "节点内先形成链"
//     (ncclTopoPreset: intra-node chain, head ranks, channel duplication),
//     "节点间连接" (connectTrees: the double tree is built over node indices
//     and attached to the heads; depth approximation), "Btree 的 bit 构造"
//     (ncclGetBtree), "双树：偶数 mirror，奇数 shift" (ncclGetDtree),
//     "先固定方向" (reduce: receive from down[], reduce the local input, send up).
//   [Interview] "all-reduce 每张卡要发多少数据? ring 和 tree 有什么区别?",
//     section "先弄清楚:每个概念是什么" (ring neighbours; two trees, half the
//     data each).
#include <cstring>

#include "common.h"
#include "host.h"

namespace vr {

// The identity ring of every channel: next = r + 1, prev = r - 1 (mod R)
// ([Interview] "先弄清楚": each rank sends to its right-hand neighbour).
void build_ring(int R, int nCh, int* next, int* prev) {
  for (int c = 0; c < nCh; ++c)
    for (int r = 0; r < R; ++r) {
      next[c * R + r] = (r + 1) % R;
      prev[c * R + r] = (r + R - 1) % R;
    }
}

// The largest power of two not above x (x >= 1).
static int bit_floor(int x) {
  int p = 1;
  while (p <= x / 2) p <<= 1;
  return p;
}

// Node r of the bit-trick binary tree over n nodes ([Course13] "Btree 的 bit
// 构造"), in closed form.  A node's level is its lowest set bit b.  Its
// parent is one of r - b and r + b, the one whose own lowest set bit is 2b
// -- r + b exactly when bit 2b of r is clear -- and r - b when r + b is not
// a node.  Its lower child is r - b/2; its upper child r + o for the largest
// power of two o <= b/2 that is still a node (none for the last node).  Node
// 0 is the root, whose only child is the largest power of two below n.
// childType: 0 when r is below its parent, else 1 (-1 for the root).
void btree(int n, int r, int* up, int* d0, int* d1, int* childType) {
  if (r == 0) {
    *up = -1;
    *d0 = -1;
    *d1 = n > 1 ? bit_floor(n - 1) : -1;
    *childType = -1;
    return;
  }
  const int b = r & -r;
  const bool above = (r & (b << 1)) == 0 && r + b < n;
  *up = above ? r + b : r - b;
  *childType = above ? 0 : 1;
  const int half = b >> 1, room = n - 1 - r;
  *d0 = half ? r - half : -1;
  *d1 = half && room > 0 ? r + bit_floor(half < room ? half : room) : -1;
}

// Node r's place in both trees: tree 0 is btree; tree 1 runs btree on a
// relabelled node (mirror n-1-r for even n, shift r-1 mod n for odd n) and
// maps parent and children back with the inverse relabelling.
void dtree(int n, int r, int t[2][4]) {
  btree(n, r, &t[0][0], &t[0][1], &t[0][2], &t[0][3]);
  int u, a, b, ct;
  if (n & 1) {
    btree(n, (r - 1 + n) % n, &u, &a, &b, &ct);
    auto back = [n](int x) { return x < 0 ? -1 : (x + 1) % n; };
    t[1][0] = back(u); t[1][1] = back(a); t[1][2] = back(b);
  } else {
    btree(n, n - 1 - r, &u, &a, &b, &ct);
    auto back = [n](int x) { return x < 0 ? -1 : n - 1 - x; };
    t[1][0] = back(u); t[1][1] = back(a); t[1][2] = back(b);
  }
  t[1][3] = ct;
}

static int floor_log2(int n) {
  int k = 0;
  while (n > 1) { n >>= 1; ++k; }
  return k;
}

int channel_tree(int c, int nCh) { return c < (nCh + 1) / 2 ? 0 : 1; }

// Append `child` to the first free down[] slot; -1 adds nothing.
static bool add_child(vr_tree_t* t, int child) {
  if (child < 0) return true;
  for (int s = 0; s < 3; ++s)
    if (t->down[s] < 0) { t->down[s] = child; return true; }
  return false;
}

// Positions, in a node's intra order, of its parent head and its child0 and
// child1 heads ([Course13] "节点内先形成链": TREE 0/0/0, SPLIT_TREE 0/1/1,
// any other pattern 0/1/0).
static void head_positions(int pattern, int* p, int* c0, int* c1) {
  *p = 0;
  *c0 = pattern == VR_PATTERN_TREE ? 0 : 1;
  *c1 = pattern == VR_PATTERN_SPLIT_TREE ? 1 : 0;
}

vr_result_t build_dtree_ex(int nNodes, int L, int nCh, int pattern, const int* orders,
                           vr_tree_t* out) {
  const int R = nNodes * L;
  const int depth = L - 1 + floor_log2(nNodes);
  int pi, c0i, c1i;
  head_positions(pattern, &pi, &c0i, &c1i);
  if (c0i >= L || c1i >= L) return VR_ERR_INVALID_ARGUMENT;
  int nodeTree[kMaxRanks][2][4];
  for (int k = 0; k < nNodes; ++k) dtree(nNodes, k, nodeTree[k]);
  for (int c = 0; c < nCh; ++c) {
    const int t = channel_tree(c, nCh);
    // the channel's intra order: a permutation of the local ranks
    int order[kMaxRanks];
    unsigned long long seen = 0;
    for (int i = 0; i < L; ++i) {
      order[i] = orders ? orders[(size_t)c * L + i] : i;
      if (order[i] < 0 || order[i] >= L || (seen >> order[i] & 1)) return VR_ERR_INVALID_ARGUMENT;
      seen |= 1ull << order[i];
    }
    vr_tree_t* tc = out + (size_t)c * R;
    // preset: each node's chain in intra order
    for (int k = 0; k < nNodes; ++k)
      for (int i = 0; i < L; ++i) {
        vr_tree_t* x = &tc[k * L + order[i]];
        x->depth = depth;
        x->up = i == 0 ? -1 : k * L + order[i - 1];
        x->down[0] = i == L - 1 ? -1 : k * L + order[i + 1];
        x->down[1] = x->down[2] = -1;
      }
    // connect: the node-level tree t attached at the heads
    for (int k = 0; k < nNodes; ++k) {
      const int u = nodeTree[k][t][0], d0 = nodeTree[k][t][1], d1 = nodeTree[k][t][2];
      const int type = nodeTree[k][t][3];
      if (u >= 0) tc[k * L + order[pi]].up = u * L + order[type == 0 ? c0i : c1i];
      if (!add_child(&tc[k * L + order[c0i]], d0 < 0 ? -1 : d0 * L + order[pi]))
        return VR_ERR_INTERNAL;
      if (!add_child(&tc[k * L + order[c1i]], d1 < 0 ? -1 : d1 * L + order[pi]))
        return VR_ERR_INTERNAL;
    }
  }
  return VR_SUCCESS;
}

vr_result_t build_dtree(int nNodes, int L, int nCh, vr_tree_t* out) {
  return build_dtree_ex(nNodes, L, nCh, VR_PATTERN_TREE, nullptr, out);
}

// A caller's tree over R ranks: up/down agree both ways, down[] is compacted,
// exactly one root, every rank reaches it (hence R-1 edges and no cycle).
bool valid_tree(const vr_tree_t* tr, int R) {
  int roots = 0;
  for (int r = 0; r < R; ++r) {
    const vr_tree_t& t = tr[r];
    if (t.up < -1 || t.up >= R || t.up == r) return false;
    if (t.up < 0) ++roots;
    else {
      const int* d = tr[t.up].down;
      if (d[0] != r && d[1] != r && d[2] != r) return false;
    }
    bool gap = false;
    for (int s = 0; s < 3; ++s) {
      const int c = t.down[s];
      if (c < -1 || c >= R) return false;
      if (c < 0) { gap = true; continue; }
      if (gap || tr[c].up != r) return false;
      for (int q = 0; q < s; ++q)
        if (t.down[q] == c) return false;
    }
  }
  if (roots != 1) return false;
  for (int r = 0; r < R; ++r) {
    int v = r, steps = 0;
    while (tr[v].up >= 0) {
      v = tr[v].up;
      if (++steps > R) return false;
    }
  }
  return true;
}

// ------------------------------------------------------------ fold program
// A rank's partial is its local input folded with each child's partial in
// down[] order.  Emitted as: the first child's partial (recursively), then
// the local input folded into it (the two-operand fold commutes bit-for-bit),
// then each further child's partial pushed and popped into it.  A chain thus
// needs a single live partial.
namespace {
struct Emitter {
  const vr_tree_t* tr;
  FoldProg* p;
  int slot = 0, pendingPops = 0, sp = 0, maxSp = 0;
  bool ok = true;

  void load(int rank, bool push) {
    if (slot >= kMaxRanks || pendingPops > 15) { ok = false; return; }
    p->rank[slot] = (uint8_t)rank;
    p->ctl[slot] = (uint8_t)(pendingPops | (push ? 16 : 0));
    sp -= pendingPops;
    pendingPops = 0;
    if (push) { ++sp; if (sp > maxSp) maxSp = sp; }
    ++slot;
  }
  void emit(int v, int guard) {
    if (guard > kMaxRanks) { ok = false; return; }
    const int* d = tr[v].down;
    if (d[0] < 0) { load(v, true); return; }
    emit(d[0], guard + 1);
    load(v, false);
    for (int s = 1; s < 3; ++s) {
      if (d[s] < 0) continue;
      emit(d[s], guard + 1);
      ++pendingPops;
    }
  }
};
}  // namespace

vr_result_t compile_fold(const vr_tree_t* tr, int R, FoldProg* p) {
  std::memset(p, 0, sizeof(*p));
  int root = -1;
  for (int r = 0; r < R; ++r)
    if (tr[r].up < 0) { if (root >= 0) return VR_ERR_INTERNAL; root = r; }
  if (root < 0) return VR_ERR_INTERNAL;
  Emitter e{tr, p};
  e.emit(root, 0);
  if (!e.ok || e.slot != R || e.pendingPops > 15) return VR_ERR_INTERNAL;
  p->n = (uint8_t)R;
  p->root = (uint8_t)root;
  p->tail = (uint8_t)e.pendingPops;
  p->depth = (uint8_t)e.maxSp;
  if (e.sp - e.pendingPops != 1 || e.maxSp > kMaxStack) return VR_ERR_INTERNAL;
  // every rank loaded exactly once
  uint64_t seen = 0;
  for (int i = 0; i < R; ++i) seen |= 1ull << p->rank[i];
  if (seen != (R == 64 ? ~0ull : ((1ull << R) - 1))) return VR_ERR_INTERNAL;
  return VR_SUCCESS;
}

// The two fold programs of the double binary tree of (nNodes, localRanks):
// tree 0 and tree 1 as channel 0 and channel 1 of vr_build_dtree see them.
vr_result_t dtree_programs(int nNodes, int L, FoldProg out[2]) {
  if (nNodes < 1 || L < 1 || nNodes * L > kMaxRanks) return VR_ERR_INVALID_ARGUMENT;
  const int R = nNodes * L;
  vr_tree_t trees[2 * kMaxRanks];
  vr_result_t e = build_dtree(nNodes, L, 2, trees);
  for (int t = 0; e == VR_SUCCESS && t < 2; ++t) e = compile_fold(trees + t * R, R, &out[t]);
  return e;
}

}  // namespace vr
