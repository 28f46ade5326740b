"""RMSNorm with AQN noise, LoRA forward on the NVFP4 backbone -- CPU oracle (test
infrastructure only).  FP64 throughout.

Sources ("QeRL: When Quantized Weights Help Reinforcement Learning, and Where the
Evidence Stops", zhongzhuzhou.org):

* section 2.1 "Weight storage and trainable state are different budgets",
  forward map:  y = W_hat x + lambda * B (A x),  W_hat = Q(W),
  A in R^{r x d_i},  B in R^{d_o x r};  its worked count 32(4096+4096) = 262,144.
* section 5.1 "Deriving the RMSNorm identity":
  u = x / sqrt(d^-1 sum_j x_j^2 + delta),  h = u (.) w,  h_z = u (.) (w + z),
  and h_z W = h diag(1 + z/w) W  when every w_j != 0.

Readings taken here: the adapter acts on the same normalised, noised
input h_z as the backbone; delta is a caller argument (1e-6 in the workloads);
w + z is formed before the product, never by dividing by w.
"""

from __future__ import annotations

import numpy as np

from .nvfp4 import dequantize


def rms_factor(x: np.ndarray, eps: float) -> np.ndarray:
    """1 / sqrt(mean_j x_j^2 + eps) per row, FP64, shape [M]."""
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / np.sqrt(np.mean(x * x, axis=-1) + float(eps))


def rmsnorm_aqn(x: np.ndarray, w_norm: np.ndarray, z: np.ndarray | None, eps: float) -> np.ndarray:
    """h_z = u (.) (w + z) with u = x / sqrt(mean(x^2) + eps); z None means no noise."""
    x = np.asarray(x, dtype=np.float64)
    scale = np.asarray(w_norm, dtype=np.float64)
    if z is not None:
        scale = scale + np.asarray(z, dtype=np.float64)
    u = x * rms_factor(x, eps)[..., None]
    return u * scale


def lora_linear_dense(h: np.ndarray, W_hat: np.ndarray, A: np.ndarray | None,
                      B: np.ndarray | None, lam: float) -> np.ndarray:
    """Row-vector form of the forward map for a batch h [M, d_i]:
    y = h W_hat^T + lam * (h A^T) B^T, FP64, shape [M, d_o]."""
    h = np.asarray(h, dtype=np.float64)
    y = h @ np.asarray(W_hat, dtype=np.float64).T
    if A is not None and B is not None and A.shape[0] > 0:
        t = h @ np.asarray(A, dtype=np.float64).T
        y = y + float(lam) * (t @ np.asarray(B, dtype=np.float64).T)
    return y


def nvfp4_lora_linear(x, packed, sb_codes, s_g, A=None, B=None, lam=0.0,
                      w_norm=None, z=None, eps=1e-6) -> np.ndarray:
    """The whole path: optional RMSNorm-AQN prologue, dequantised backbone, LoRA.
    x [M, d_i] (BF16 values as FP32/FP64), packed [d_o, d_i/2], sb_codes
    [d_o, d_i/16], A [r, d_i], B [d_o, r].  Returns y [M, d_o] in FP64."""
    x = np.asarray(x, dtype=np.float64)
    h = rmsnorm_aqn(x, w_norm, z, eps) if w_norm is not None else x
    W_hat = dequantize(packed, sb_codes, s_g)
    return lora_linear_dense(h, W_hat, A, B, lam)


def lora_param_count(d_i: int, d_o: int, r: int) -> int:
    """Trainable adapter parameters r * (d_i + d_o) of one projection."""
    return r * (d_i + d_o)
