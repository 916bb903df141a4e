"""Dense float64 products from decoded weights.  Test infrastructure.

[QMoE] "The GPU Decoding Kernel": the fused kernel computes y = W x for one
token (one dot product per row); "Per-Layer Kernel Performance" / the
limitations section propose an inner loop over tokens for experts that
receive several tokens, i.e. Y = X W^T.  Here the product is formed plainly in
float64 from the decoded matrix; ``ternary_dot`` restates one row in the form
s * (sum of x over +1 positions - sum of x over -1 positions).
"""
from __future__ import annotations

import numpy as np


def matmul_xwt(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Y[T, rows] = X[T, cols] . W[rows, cols]^T in float64."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    if x.ndim == 1:
        x = x[None, :]
    if x.shape[1] != w.shape[1]:
        raise ValueError("inner dimensions differ")
    return x @ w.T


def ternary_dot(tern_row: np.ndarray, scale: float, x: np.ndarray) -> float:
    """One output of a ternary row: s * (sum_{w=+1} x - sum_{w=-1} x)."""
    t = np.asarray(tern_row)
    x = np.asarray(x, dtype=np.float64)
    return float(scale) * (float(x[t == 1].sum()) - float(x[t == -1].sum()))


def normwise_rel_err(y: np.ndarray, ref: np.ndarray) -> float:
    """max_i |y_i - ref_i| / max_i |ref_i| (0 when both are all zero)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(y - ref))) if ref.size else 0.0
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den
