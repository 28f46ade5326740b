"""Update-aware quantisation (invariant scaling) folded into the NVFP4 backbone and the
RMSNorm in front of it -- CPU oracle (test infrastructure only).

Source: "QuRL: Low-Precision Reinforcement Learning for Efficient Reasoning"
(papernotes.org reading notes), section 3 "更新感知量化 UAQ": a linear layer is
invariant under W X = (W / s)(s X); the factor on the activations is absorbed by the
normalisation before it; the method picks s > 1 on purpose (s = 1.5 in its runs), once,
before training, so that a weight update grows by s relative to the quantisation step.

Readings taken here: the fold divides the weight in FP32, W' = fp32(W / s),
before the fixed-scale quantiser of oracle.nvfp4, and multiplies the FP32 norm weight,
w' = fp32(w * s); the AQN noise is drawn on the folded scale as before, h = u (.) (w' + z).
"""

from __future__ import annotations

import numpy as np

from .nvfp4 import quantize

UAQ_S = 1.5  # the factor of the QuRL runs


def fold(W, w_norm, s: float = UAQ_S):
    """(W' = fp32(W / s), w' = fp32(w_norm * s)): the folded weight and norm scale."""
    s32 = np.float32(s)
    W32 = np.asarray(W, dtype=np.float32)
    Wf = (W32 / s32).astype(np.float32)
    wf = (np.asarray(w_norm, dtype=np.float32) * s32).astype(np.float32)
    return Wf, wf


def quantize_folded(W, s: float = UAQ_S):
    """NVFP4 encoding (packed codes, scale codes, s_g) of the folded weight fp32(W / s)."""
    Wf, _ = fold(W, np.ones(np.asarray(W).shape[-1], np.float32), s)
    return quantize(Wf)
