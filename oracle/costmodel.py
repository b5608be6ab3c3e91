"""The pages' alpha-beta cost model of ring and tree AllReduce.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources:
* [Course13] section "理想成本模型": with N ranks, tree depth D, M bytes per
  rank, a fixed cost alpha per dependent stage and an effective bandwidth B,
  T_tree ~ 2 D alpha + 2 M / B_tree and
  T_ring ~ 2 (N-1) alpha + 2 (N-1)/N * M / B_ring; the formulas are meant for
  falsifiable predictions, not to replace measurement.
* [Interview] section "推导 / 关键公式": ring latency term 2(n-1) alpha, per-card
  traffic 2(n-1)/n * S; tree latency ~ 2 log2(n) alpha, traffic ~ 2S.

Readings: the model's two terms are fitted per algorithm by least squares to
measured times (alpha in microseconds per stage, 1/B in microseconds per
byte of the model's traffic term); the predicted crossover is where the two
lines meet.  The pages give the model's form, not how to fit it.  Measured
times span several decades (8 B to 256 MiB messages), so the fit that sets
the model's constants weighs every sample by its own size: it minimises the
sum of squared relative errors (prediction - t) / t (``fit_relative``), and a
sample whose time is not positive carries no information and is left out.
``fit`` is the plain (absolute) least-squares fit of the same model.
"""

import numpy as np


def ring_terms(N, M):
    """(stages, traffic bytes) of the ring: 2(N-1) and 2(N-1)/N * M."""
    return 2 * (N - 1), 2.0 * (N - 1) / N * M


def tree_terms(D, M):
    """(stages, traffic bytes) of the tree: 2D and 2M."""
    return 2 * D, 2.0 * M


def predict(stages, traffic, alpha, inv_bw):
    return stages * alpha + traffic * inv_bw


def t_ring(N, M, alpha, inv_bw):
    s, b = ring_terms(N, M)
    return predict(s, b, alpha, inv_bw)


def t_tree(D, M, alpha, inv_bw):
    s, b = tree_terms(D, M)
    return predict(s, b, alpha, inv_bw)


def crossover(N, D, ring, tree):
    """Message size M at which the ring and tree predictions are equal, or
    None when the lines do not cross at a positive size.  ring / tree are
    (alpha, inv_bw) pairs."""
    (ar, br), (at, bt) = ring, tree
    num = 2 * D * at - 2 * (N - 1) * ar
    den = 2.0 * (N - 1) / N * br - 2.0 * bt
    if den == 0:
        return None
    m = num / den
    return m if m > 0 else None


def fit(stages, traffic, times):
    """Least-squares (alpha, inv_bw) for times ~ alpha*stages + inv_bw*traffic."""
    A = np.stack([np.asarray(stages, float), np.asarray(traffic, float)], axis=1)
    sol, *_ = np.linalg.lstsq(A, np.asarray(times, float), rcond=None)
    return float(sol[0]), float(sol[1])


def fit_relative(stages, traffic, times):
    """(alpha, inv_bw) minimising sum over samples with t > 0 of
    ((alpha*stages + inv_bw*traffic - t) / t)**2: least squares of the rows
    (stages/t, traffic/t) against 1."""
    keep = [i for i, t in enumerate(times) if t > 0]
    t = np.asarray([times[i] for i in keep], float)
    A = np.stack([np.asarray([stages[i] for i in keep], float) / t,
                  np.asarray([traffic[i] for i in keep], float) / t], axis=1)
    sol, *_ = np.linalg.lstsq(A, np.ones(len(keep)), rcond=None)
    return float(sol[0]), float(sol[1])


def select(N, D, M, ring, tree):
    """"ring" when its prediction is not above the tree's, else "tree"."""
    return "ring" if t_ring(N, M, *ring) <= t_tree(D, M, *tree) else "tree"
