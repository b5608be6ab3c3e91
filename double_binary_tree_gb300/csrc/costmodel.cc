// The pages' alpha-beta cost model ([Course13] "理想成本模型"; [Interview]
// "推导 / 关键公式"): ring and tree predictions, selection, crossover, and a
// relative least-squares fit to measured times.
#include <algorithm>
#include <cmath>
#include <map>
#include <mutex>
#include <utility>

#include "host.h"

namespace vr {
namespace {

std::mutex g_modelMu;

// The alpha-beta cost model: built-in constants fitted on GB300 with
// vr_fit_cost_model to the measured times of 4 ranks, 8 B .. 256 MiB per rank
// (bench.py --sweep); replaceable through vr_set_cost_model.
const vr_cost_model_t kBuiltinModel = {{0.343939, 0.473172}, {8.66964e-7, 6.13639e-7}};
vr_cost_model_t g_model = kBuiltinModel;

// Exact depth (edges from the root to the deepest leaf) of one tree.
int exact_depth(const vr_tree_t* tr, int R) {
  int worst = 0;
  for (int r = 0; r < R; ++r) {
    int d = 0;
    for (int v = r; tr[v].up >= 0 && d <= R; v = tr[v].up) ++d;
    worst = std::max(worst, d);
  }
  return worst;
}

}  // namespace
}  // namespace vr

using namespace vr;

extern "C" {

vr_result_t vr_predict_us(vr_algo_t algo, int R, int localRanks, size_t bytesPerRank,
                          const vr_cost_model_t* model, double* us) {
  if ((algo != VR_ALGO_RING && algo != VR_ALGO_TREE) || R < 1 || R > kMaxRanks ||
      localRanks < 1 || R % localRanks || !us)
    return VR_ERR_INVALID_ARGUMENT;
  vr_cost_model_t m;
  {
    std::lock_guard<std::mutex> g(g_modelMu);
    m = model ? *model : g_model;
  }
  const double M = (double)bytesPerRank, N = (double)R;
  if (algo == VR_ALGO_RING) {
    *us = 2.0 * (N - 1) * m.alphaUs[0] + (2.0 * (N - 1) / N * M) * m.usPerByte[0];
    return VR_SUCCESS;
  }
  int D = 0;
  {
    static std::map<std::pair<int, int>, int> depths;  // (R, localRanks) -> D
    std::lock_guard<std::mutex> g(g_modelMu);
    auto it = depths.find(std::make_pair(R, localRanks));
    if (it == depths.end()) {
      vr_tree_t trees[2 * kMaxRanks];
      const vr_result_t e = build_dtree(R / localRanks, localRanks, 2, trees);
      if (e != VR_SUCCESS) return e;
      it = depths.emplace(std::make_pair(R, localRanks),
                          std::max(exact_depth(trees, R), exact_depth(trees + R, R)))
               .first;
    }
    D = it->second;
  }
  *us = 2.0 * D * m.alphaUs[1] + (2.0 * M) * m.usPerByte[1];
  return VR_SUCCESS;
}

vr_result_t vr_select_algo(int R, int localRanks, size_t bytesPerRank,
                           const vr_cost_model_t* model, vr_algo_t* algo) {
  if (!algo) return VR_ERR_INVALID_ARGUMENT;
  double tr = 0, tt = 0;
  vr_result_t e = vr_predict_us(VR_ALGO_RING, R, localRanks, bytesPerRank, model, &tr);
  if (e == VR_SUCCESS) e = vr_predict_us(VR_ALGO_TREE, R, localRanks, bytesPerRank, model, &tt);
  if (e != VR_SUCCESS) return e;
  *algo = tr <= tt ? VR_ALGO_RING : VR_ALGO_TREE;
  return VR_SUCCESS;
}

vr_result_t vr_fit_cost_model(int n, const int* R, const int* localRanks,
                              const size_t* bytesPerRank, const double* ringUs,
                              const double* treeUs, vr_cost_model_t* out) {
  if (n < 2 || !R || !localRanks || !bytesPerRank || !ringUs || !treeUs || !out)
    return VR_ERR_INVALID_ARGUMENT;
  // Each sample's prediction is alpha * stages + perByte * traffic, linear in
  // the two unknowns: the model with alpha = 1, perByte = 0 gives `stages`,
  // the one with alpha = 0, perByte = 1 gives `traffic`.
  const vr_cost_model_t unitA = {{1.0, 1.0}, {0.0, 0.0}};
  const vr_cost_model_t unitB = {{0.0, 0.0}, {1.0, 1.0}};
  vr_cost_model_t m;
  for (int alg = 0; alg < 2; ++alg) {
    const double* t = alg == 0 ? ringUs : treeUs;
    double ss = 0, sb = 0, bb = 0, s1 = 0, b1 = 0;
    int used = 0;
    for (int i = 0; i < n; ++i) {
      if (!(t[i] > 0)) continue;
      double st = 0, tr = 0;
      vr_result_t e = vr_predict_us((vr_algo_t)alg, R[i], localRanks[i], bytesPerRank[i], &unitA,
                                    &st);
      if (e == VR_SUCCESS)
        e = vr_predict_us((vr_algo_t)alg, R[i], localRanks[i], bytesPerRank[i], &unitB, &tr);
      if (e != VR_SUCCESS) return e;
      // relative error: divide the row and its target (the time) by the time
      const double x = st / t[i], y = tr / t[i];
      ss += x * x; sb += x * y; bb += y * y; s1 += x; b1 += y;
      ++used;
    }
    const double det = ss * bb - sb * sb;
    if (used < 2 || !(std::fabs(det) > 1e-300 * (ss * bb + 1e-300)) || !std::isfinite(det))
      return VR_ERR_INVALID_ARGUMENT;
    m.alphaUs[alg] = (s1 * bb - b1 * sb) / det;
    m.usPerByte[alg] = (ss * b1 - sb * s1) / det;
  }
  *out = m;
  return VR_SUCCESS;
}

vr_result_t vr_crossover_bytes(int R, int localRanks, const vr_cost_model_t* model,
                               double* bytes) {
  if (!bytes) return VR_ERR_INVALID_ARGUMENT;
  // Both predictions are lines in the message size M: evaluate each at M = 0
  // and M = 1 GiB (far apart, so the slopes lose no precision) and intersect.
  const size_t far = (size_t)1 << 30;
  double r0 = 0, r1 = 0, t0 = 0, t1 = 0;
  vr_result_t e = vr_predict_us(VR_ALGO_RING, R, localRanks, 0, model, &r0);
  if (e == VR_SUCCESS) e = vr_predict_us(VR_ALGO_RING, R, localRanks, far, model, &r1);
  if (e == VR_SUCCESS) e = vr_predict_us(VR_ALGO_TREE, R, localRanks, 0, model, &t0);
  if (e == VR_SUCCESS) e = vr_predict_us(VR_ALGO_TREE, R, localRanks, far, model, &t1);
  if (e != VR_SUCCESS) return e;
  const double slope = ((r1 - r0) - (t1 - t0)) / (double)far;
  const double m = slope != 0 ? (t0 - r0) / slope : -1.0;
  *bytes = m > 0 && std::isfinite(m) ? m : -1.0;
  return VR_SUCCESS;
}

vr_result_t vr_set_cost_model(const vr_cost_model_t* model) {
  if (model)
    for (int i = 0; i < 2; ++i)
      if (!(model->alphaUs[i] >= 0 && model->usPerByte[i] >= 0) ||
          !std::isfinite(model->alphaUs[i]) || !std::isfinite(model->usPerByte[i]))
        return VR_ERR_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> g(g_modelMu);
  g_model = model ? *model : kBuiltinModel;
  return VR_SUCCESS;
}

}  // extern "C"
