// The option VR_DEBUG=GRAPH: the library prints the topology and partition
// it plans to stderr.
//
// Trees use the two log formats of [Course13] "从 GRAPH 日志复原 active tree"
// and "先固定方向": "Tree c : up -> rank -> d0/d1/d2" (one line per rank,
// read as: on channel c, `rank` has parent `up` and children d0, d1, d2) and
// "Trees [c] d0/d1/d2->rank->up" (the same record, children first).  The
// pages print no ring or partition lines; this library's own are
//   Ring c : r0 r1 ... r(R-1)        the ranks in ring order from rank 0
//   Part c : offset o count n        channel c's elements [o, o + n)
// A collective call prints its plan the first time the process sees that
// plan (kind, algorithm, R, local ranks, count, element size, channels,
// chunk bytes, tree set), after a header line "vr plan: ...".
#include <cstdio>
#include <mutex>
#include <set>
#include <string>

#include "host.h"

namespace vr {
namespace {

std::mutex g_logMu;
std::set<std::string> g_printed;

void tree_lines(const vr_tree_t* trees, int R, int nCh) {
  for (int c = 0; c < nCh; ++c) {
    const vr_tree_t* t = trees + (size_t)c * R;
    for (int r = 0; r < R; ++r)
      std::fprintf(stderr, "Tree %d : %d -> %d -> %d/%d/%d\n", c, t[r].up, r, t[r].down[0],
                   t[r].down[1], t[r].down[2]);
    for (int r = 0; r < R; ++r)
      std::fprintf(stderr, "Trees [%d] %d/%d/%d->%d->%d\n", c, t[r].down[0], t[r].down[1],
                   t[r].down[2], r, t[r].up);
  }
}

void ring_lines(const int* next, int R, int nCh) {
  for (int c = 0; c < nCh; ++c) {
    std::fprintf(stderr, "Ring %d :", c);
    int v = 0;
    for (int i = 0; i < R; ++i) {
      std::fprintf(stderr, " %d", v);
      v = next[(size_t)c * R + v];
    }
    std::fprintf(stderr, "\n");
  }
}

}  // namespace

bool graph_logging() { return (option(kOptDebug) & kDebugGraph) != 0; }

void log_trees(const vr_tree_t* trees, int R, int nCh) {
  if (!graph_logging()) return;
  std::lock_guard<std::mutex> g(g_logMu);
  tree_lines(trees, R, nCh);
  std::fflush(stderr);
}

void log_ring(const int* next, int R, int nCh) {
  if (!graph_logging()) return;
  std::lock_guard<std::mutex> g(g_logMu);
  ring_lines(next, R, nCh);
  std::fflush(stderr);
}

void log_plan(const char* kind, int algo, int R, int L, size_t count, int dtype, int nCh,
              size_t chunkBytes, const vr_tree_t* trees, bool partitioned) {
  if (!graph_logging()) return;
  char head[256];
  std::snprintf(head, sizeof(head),
                "vr plan: %s %s R=%d localRanks=%d count=%zu dtype=%d nChannels=%d "
                "chunkBytes=%zu",
                kind, algo == VR_ALGO_TREE ? "tree" : "ring", R, L, count, dtype, nCh,
                chunkBytes);
  std::string key(head);
  if (trees)
    key.append(reinterpret_cast<const char*>(trees), sizeof(vr_tree_t) * (size_t)R * nCh);
  std::lock_guard<std::mutex> g(g_logMu);
  if (!g_printed.insert(key).second) return;
  std::fprintf(stderr, "%s\n", head);
  if (trees) {
    tree_lines(trees, R, nCh);
  } else {
    static int next[kMaxRanks * kMaxChannels], prev[kMaxRanks * kMaxChannels];  // under g_logMu
    build_ring(R, nCh, next, prev);
    ring_lines(next, R, nCh);
  }
  for (int c = 0; partitioned && c < nCh; ++c) {
    size_t off = 0, n = 0;
    if (vr_partition(count, (vr_dtype_t)dtype, nCh, c, &off, &n) != VR_SUCCESS) return;
    std::fprintf(stderr, "Part %d : offset %zu count %zu\n", c, off, n);
  }
  std::fflush(stderr);
}

}  // namespace vr
