"""Error bounds of the fp32-accumulated reductions against the fp64 sum.

Any summation order of R terms in fp32 (unit roundoff u = 2**-24) satisfies
|y - s| <= gamma_{R-1} * sum|x|, gamma_k = k u / (1 - k u) (the classical
recursive-summation bound, Higham, "Accuracy and Stability of Numerical
Algorithms", section 4.2).  A 16-bit output adds one final rounding of
relative size u_T (bf16: 2**-8, fp16: 2**-11) plus, for fp16, half the
smallest subnormal.  The norm-wise acceptance bounds are the ones the method
is specified to: 1e-5 relative for fp32 results, 1e-2 for 16-bit outputs.
"""

import numpy as np

U32 = 2.0 ** -24
U_T = {0: 0.0, 1: 2.0 ** -11, 2: 2.0 ** -8}
ABS_MIN = {0: 0.0, 1: 2.0 ** -25, 2: 0.0}
NORM_TOL = {0: 1e-5, 1: 1e-2, 2: 1e-2}


def gamma(k):
    return k * U32 / (1.0 - k * U32)


def elementwise_bound(abs_sum, s, R, dtype):
    g = gamma(max(R - 1, 0)) * abs_sum
    uT = U_T[dtype]
    return g * (1.0 + uT) + uT * np.abs(s) * (1.0 + 1e-12) + ABS_MIN[dtype] + 1e-300


def check_against_fp64(y, s, abs_sum, R, dtype):
    """Raise AssertionError with a short report when y (fp64 view of the
    results) breaks either bound against the fp64 sum s."""
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - s)
    bound = elementwise_bound(abs_sum, s, R, dtype)
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, "elementwise bound broken at %s: y=%r s=%r bound=%r" % (
        bad[:5], y[bad[:5]], s[bad[:5]], bound[bad[:5]])
    ns = np.linalg.norm(s)
    if ns > 0:
        rel = np.linalg.norm(y - s) / ns
        assert rel <= NORM_TOL[dtype], "norm-wise relative error %g > %g" % (rel, NORM_TOL[dtype])
