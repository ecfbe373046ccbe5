"""CPU oracle of the post-scale W8A8 linear operator (TurboT2VA, section 6.2 of the
robotworld.top/zh reading, "shape-aware post-scale W8A8 linear operator"; section 6 of
the robotworld.top/en summary).

TEST INFRASTRUCTURE ONLY. Nothing in the library imports this module; only tests/,
__graft_entry__.smoke() and bench.py's CPU legs may call it.

What the pages fix:
  * activations are quantised per row, dynamically: s_i^x = max(||x_i||_inf, eps) / 127,
    x_hat_i = clip(round(x_i / s_i^x), -127, 127);
  * weights are quantised the same way per output channel (row j of W, [N, K]), once;
  * y_ij = s_i^x s_j^w sum_k x_hat_ik w_hat_jk + b_j, the sum accumulated exactly in
    INT32 over the whole K and both scales applied once, after the sum;
  * eps = 1e-4.

Readings (the pages leave these open):
  * the rounding is round-half-to-even;
  * a quantised code is an integer decided in floating point, so the oracle takes that
    decision in the precision the kernel uses: the scale is max(amax, eps) / 127 in
    float32 (IEEE division), and the code is rint(x / s) of the float32 quotient;
  * y is evaluated exactly (float64 of the integer sum and the float32 scales); the
    kernel's float32 epilogue is compared against it within a stated bound.
"""

from __future__ import annotations

from typing import Optional, Tuple

import numpy as np

EPS = 1e-4


def row_scales(x: np.ndarray, eps: float = EPS) -> np.ndarray:
    """s_i = max(||x_i||_inf, eps) / 127 per row, in float32 (IEEE division)."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=1) if x32.shape[1] > 0 else np.zeros(x32.shape[0], np.float32)
    return (np.maximum(amax, np.float32(eps)) / np.float32(127.0)).astype(np.float32)


def quantize_rows(x: np.ndarray, eps: float = EPS) -> Tuple[np.ndarray, np.ndarray]:
    """x_hat = clip(round(x / s), -127, 127) per row, s = row_scales(x); returns
    (int8 codes [M, K], float32 scales [M])."""
    x32 = np.asarray(x, dtype=np.float32)
    s = row_scales(x32, eps)
    q = np.rint(x32 / s[:, None])           # float32 quotient, round half to even
    q = np.clip(q, -127, 127)
    return q.astype(np.int8), s


def int_dot(xq: np.ndarray, wq: np.ndarray) -> np.ndarray:
    """acc_ij = sum_k x_hat_ik w_hat_jk, exact (int64)."""
    return np.asarray(xq, np.int64) @ np.asarray(wq, np.int64).T


def w8a8_linear(xq: np.ndarray, sx: np.ndarray, wq: np.ndarray, sw: np.ndarray,
                bias: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
    """y_ij = s_i^x s_j^w acc_ij + b_j with the exact integer sum; returns (acc int64
    [M, N], y float64 [M, N])."""
    acc = int_dot(xq, wq)
    y = (np.asarray(sx, np.float64)[:, None] * np.asarray(sw, np.float64)[None, :]) * acc
    if bias is not None:
        y = y + np.asarray(bias, np.float64)[None, :]
    return acc, y


def w8a8_forward(x: np.ndarray, wq: np.ndarray, sw: np.ndarray,
                 bias: Optional[np.ndarray] = None, eps: float = EPS):
    """The whole operator for activations x [M, K] and pre-quantised weights: quantise
    x per row, then w8a8_linear. Returns (xq, sx, acc, y)."""
    xq, sx = quantize_rows(x, eps)
    acc, y = w8a8_linear(xq, sx, wq, sw, bias)
    return xq, sx, acc, y
