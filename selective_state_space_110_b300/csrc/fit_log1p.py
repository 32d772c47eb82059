"""Coefficients of the polynomial P(w) ~ log1p(w) / w on [0, 1] used by the scan kernel's softplus.

The kernel evaluates softplus(x) = max(x, 0) + w * P(w) with w = exp(-|x|) in (0, 1], so that
one SFU exp2 and a short Horner chain replace the log1p(exp(x)) of the library. P is fitted by
weighted least squares on Chebyshev nodes of [0, 1], weighted so that the error of w * P(w) is
measured relative to log1p(w), then checked on a dense grid in float64.

python -m selective_state_space_110_b300.csrc.fit_log1p   (prints the C initialiser)
"""
from __future__ import annotations

import numpy as np

DEGREE = 6


def fit(degree: int = DEGREE, nodes: int = 400):
    k = np.arange(nodes)
    w = 0.5 - 0.5 * np.cos((2 * k + 1) * np.pi / (2 * nodes))  # Chebyshev nodes on [0, 1]
    w = np.concatenate([[0.0], w, [1.0]])
    target = np.where(w > 0, np.log1p(w) / np.where(w > 0, w, 1.0), 1.0)
    V = np.vander(w, degree + 1, increasing=True)
    coef, *_ = np.linalg.lstsq(V, target, rcond=None)
    return coef


def max_rel_error(coef, n: int = 200001) -> float:
    w = np.linspace(0.0, 1.0, n)[1:]
    p = np.polynomial.polynomial.polyval(w, coef)
    return float(np.max(np.abs(w * p - np.log1p(w)) / np.log1p(w)))


if __name__ == "__main__":
    c = fit()
    c32 = c.astype(np.float32).astype(np.float64)
    print("// max relative error of w*P(w) vs log1p(w) on (0,1]: %.2e (float32 coefficients: %.2e)"
          % (max_rel_error(c), max_rel_error(c32)))
    print("{" + ", ".join("%.9ef" % v for v in c.astype(np.float32)) + "}")
