"""Accuracy of a collective's result against the plain definition in fp64.

Two measures of the same error d = |y - y64|:
- normwise: ||d||_2 / ||y64||_2, the form in which the 1e-2 (bf16) and 1e-5
  (fp32) relative tolerances are checked, since elementwise relative error is
  unbounded where the sum cancels;
- elementwise: max_e d_e / max(|y64_e|, S_e), with S_e = sum_r |x_r,e| (divided
  by N for AVG), the condition scale of the sum.  Recursive summation with a
  rounding after each of the N-1 hops bounds it by (N-1+[AVG]) * u, where
  u = 2^-8 + 2^-24 for bf16 and 2^-24 for fp32.
"""
import numpy as np


def error_figures(y, y64, absum):
    y = np.asarray(y, dtype=np.float64)
    d = np.abs(y - y64)
    scale = np.maximum(np.abs(y64), absum)
    nz = scale > 0
    assert np.all(d[~nz] == 0)
    n64 = np.linalg.norm(y64)
    return {"normwise": float(np.linalg.norm(d) / n64) if n64 > 0 else 0.0,
            "elementwise": float(np.max(d[nz] / scale[nz])) if nz.any() else 0.0}


def report(tag, fig):
    print("ACCURACY %s normwise=%.4g elementwise=%.4g" % (tag, fig["normwise"], fig["elementwise"]))
