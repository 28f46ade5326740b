"""Backward of the frozen-backbone LoRA linear with its RMSNorm-AQN prologue -- CPU
oracle (test infrastructure only).  FP64 throughout.

Source: "QeRL: When Quantized Weights Help Reinforcement Learning, and Where the
Evidence Stops" (zhongzhuzhou.org), section 2.1 "Weight storage and trainable state
are different budgets": the forward map is y = W_hat x + lambda B (A x) with
W_hat = Q(W) frozen; the gradients update A and B only, but they still have to pass
through the frozen projection to reach the layers (and adapters) before it.  The
prologue is section 5.1's h = u (.) (w + z), u = x / sqrt(mean(x^2) + delta), with w
and z not trained.

In the row-vector form of the forward oracle (h [M, d_i], y = h W_hat^T + lambda
(h A^T) B^T), for an upstream gradient g = dL/dy [M, d_o]:

* dh = g W_hat + lambda (g B) A                  [M, d_i]
* dA = lambda (g B)^T h                          [r, d_i]
* dB = lambda g^T (h A^T)                        [d_o, r]
* with rho = (mean_j x_j^2 + delta)^(-1/2) per row and s = w + z:
  dx = rho s (.) dh - rho^3 x (sum_j x_j s_j dh_j) / d

These are the chain rule written out (the derivative of h_j = x_j rho s_j is
rho s_j [j == i] - x_j s_j rho^3 x_i / d); nothing is blocked, fused or reordered.
"""

from __future__ import annotations

import numpy as np

from .linear import rms_factor, rmsnorm_aqn
from .nvfp4 import dequantize


def lora_backward_input(g, W_hat, A=None, B=None, lam=0.0) -> np.ndarray:
    """dh = g W_hat + lam (g B) A: the gradient that passes through the frozen backbone."""
    g = np.asarray(g, dtype=np.float64)
    dh = g @ np.asarray(W_hat, dtype=np.float64)
    if A is not None and B is not None and np.asarray(A).shape[0] > 0:
        gb = g @ np.asarray(B, dtype=np.float64)  # [M, r]
        dh = dh + float(lam) * (gb @ np.asarray(A, dtype=np.float64))
    return dh


def lora_adapter_grads(h, g, A, B, lam):
    """(dA, dB) = (lam (g B)^T h, lam g^T (h A^T)), the adapter's parameter gradients."""
    h = np.asarray(h, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    dA = float(lam) * ((g @ B).T @ h)
    dB = float(lam) * (g.T @ (h @ A.T))
    return dA, dB


def rmsnorm_aqn_backward(x, w_norm, z, eps, dh) -> np.ndarray:
    """dx of h = u (.) (w + z), u = x rho: rho s (.) dh - rho^3 x (sum_j x_j s_j dh_j) / d."""
    x = np.asarray(x, dtype=np.float64)
    dh = np.asarray(dh, dtype=np.float64)
    s = np.asarray(w_norm, dtype=np.float64)
    if z is not None:
        s = s + np.asarray(z, dtype=np.float64)
    d = x.shape[-1]
    rho = rms_factor(x, eps)[..., None]
    proj = np.sum(x * s * dh, axis=-1, keepdims=True) / d
    return rho * s * dh - rho ** 3 * x * proj


def nvfp4_lora_linear_backward(x, g, packed, sb_codes, s_g, A=None, B=None, lam=0.0, w_norm=None, z=None,
                               eps=1e-6):
    """The whole path's backward: (dx, dA, dB) for the forward of oracle.linear.nvfp4_lora_linear.
    dA and dB are None without an adapter."""
    x = np.asarray(x, dtype=np.float64)
    h = rmsnorm_aqn(x, w_norm, z, eps) if w_norm is not None else x
    W_hat = dequantize(packed, sb_codes, s_g)
    dh = lora_backward_input(g, W_hat, A, B, lam)
    dx = rmsnorm_aqn_backward(x, w_norm, z, eps, dh) if w_norm is not None else dh
    if A is not None and B is not None and np.asarray(A).shape[0] > 0:
        dA, dB = lora_adapter_grads(h, g, A, B, lam)
    else:
        dA = dB = None
    return dx, dA, dB
