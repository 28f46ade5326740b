"""W8A8 rollout linear (INT8 or FP8 E4M3 weights and activations) -- CPU oracle (test
infrastructure only).

Source: "QuRL: Low-Precision Reinforcement Learning for Efficient Reasoning"
(papernotes.org reading notes): before each rollout the full-precision actor is
quantised, theta_hat = Q(theta, b), weights with one scale per output channel and
activations with one scale per token, in INT8 or FP8, and the rollout runs on INT8 /
FP8 matrix products; the quantisation error is about |theta| / 2^b.

Readings taken here (the notes give no formula for Q):
* symmetric absmax scales, no zero point: INT8 s = fp32(amax / 127), q = clip(RNE(fp32(v / s)),
  -127, 127); FP8 s = fp32(amax / 448), code = E4M3 of fp32(v / s) (round to nearest, ties
  to even, saturating at 448; sign bit separate, +0 for zero); s = 1 for an all-zero row;
* weight rows = output channels; activation rows = tokens, quantised after the
  RMSNorm-AQN prologue (the same h as the NVFP4 path);
* y[m, o] = s_x[m] s_w[o] sum_k q_x[m, k] q_w[o, k] (exact: integer sum for INT8, FP64 for
  FP8), plus the adapter term lambda B (A h) on the unquantised h, as on the NVFP4 path.
"""

from __future__ import annotations

import numpy as np

from .linear import rmsnorm_aqn
from .nvfp4 import E4M3_MAX, E4M3_TABLE, e4m3_encode

INT8_MAX = 127


def _row_scale(X: np.ndarray, top: float) -> np.ndarray:
    amax = np.max(np.abs(X.astype(np.float32)), axis=-1)
    s = (amax / np.float32(top)).astype(np.float32)
    return np.where(amax > 0, s, np.float32(1.0)).astype(np.float32)


def quantize_int8_rows(X):
    """(q int8 [R, C], s float32 [R]): symmetric absmax, round to nearest even."""
    X32 = np.asarray(X, dtype=np.float32)
    s = _row_scale(X32, INT8_MAX)
    v = (X32 / s[:, None]).astype(np.float32)
    q = np.clip(np.rint(v), -INT8_MAX, INT8_MAX).astype(np.int8)
    return q, s


def e4m3_encode_signed(v) -> np.ndarray:
    """E4M3 codes of finite FP32 values: sign bit | nearest-even magnitude code, saturating."""
    v = np.asarray(v, dtype=np.float32)
    mag = e4m3_encode(np.abs(v))
    sign = np.where((v < 0) & (mag != 0), 0x80, 0).astype(np.uint8)
    return (mag.astype(np.uint8) | sign).astype(np.uint8)


def quantize_fp8_rows(X):
    """(codes uint8 [R, C] E4M3, s float32 [R]): symmetric absmax onto E4M3's 448."""
    X32 = np.asarray(X, dtype=np.float32)
    s = _row_scale(X32, E4M3_MAX)
    v = (X32 / s[:, None]).astype(np.float32)
    return e4m3_encode_signed(v), s


def dequant_rows(q, s, fmt: str) -> np.ndarray:
    """FP64 reconstruction s[r] * value(q[r, c])."""
    vals = q.astype(np.float64) if fmt == "int8" else E4M3_TABLE[q]
    return vals * np.asarray(s, dtype=np.float64)[:, None]


def w8a8_linear(x, Wq, s_w, fmt: str, A=None, B=None, lam=0.0, w_norm=None, z=None, eps=1e-6):
    """y [M, d_o] in FP64 for quantised weights (Wq [d_o, d_i], s_w [d_o]) of format fmt."""
    x = np.asarray(x, dtype=np.float64)
    h = rmsnorm_aqn(x, w_norm, z, eps) if w_norm is not None else x
    h32 = h.astype(np.float32)
    if fmt == "int8":
        qx, s_x = quantize_int8_rows(h32)
        acc = qx.astype(np.int64) @ Wq.astype(np.int64).T  # exact integer sum
        y = acc.astype(np.float64)
    elif fmt == "fp8":
        qx, s_x = quantize_fp8_rows(h32)
        y = E4M3_TABLE[qx] @ E4M3_TABLE[Wq].T  # products of E4M3 values, FP64 sum
    else:
        raise ValueError(fmt)
    y = y * np.asarray(s_x, np.float64)[:, None] * np.asarray(s_w, np.float64)[None, :]
    if A is not None and B is not None and np.asarray(A).shape[0] > 0:
        y = y + float(lam) * ((h @ np.asarray(A, np.float64).T) @ np.asarray(B, np.float64).T)
    return y
