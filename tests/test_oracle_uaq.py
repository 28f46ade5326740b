"""Pins of the UAQ fold (oracle/uaq.py): the invariance W X = (W / s)(s X) in FP64; for
a power-of-two s the fixed-scale NVFP4 quantiser is exactly scale-equivariant (same
codes and block scales, s_g divided by s), so the folded layer's output equals the
unfolded one bit for bit; for the pages' s = 1.5 the folded layer stays within the
NVFP4 error of the unfolded one."""

import numpy as np
import pytest

from oracle import linear as olin
from oracle import nvfp4 as onv
from oracle import uaq


def _case(d_o=64, d_i=128, M=6, seed=0):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((d_o, d_i)) * 0.02).astype(np.float32)
    x = rng.standard_normal((M, d_i))
    w = (1 + 0.1 * rng.standard_normal(d_i)).astype(np.float32)
    z = (1e-2 * rng.standard_normal(d_i)).astype(np.float32)
    return W, x, w, z


@pytest.mark.parametrize("s", [1.5, 2.0, 0.75])
def test_invariance_in_fp64(s):
    W, x, _, _ = _case()
    W64 = W.astype(np.float64)
    y = x @ W64.T
    y_s = (s * x) @ (W64 / s).T
    assert np.max(np.abs(y - y_s)) <= 1e-14 * np.max(np.abs(y))


@pytest.mark.parametrize("s", [2.0, 4.0, 0.5])
def test_power_of_two_fold_is_exact_through_the_quantiser(s):
    W, x, w, _ = _case(seed=1)
    packed, sb, s_g = onv.quantize(W)
    pf, sbf, s_gf = uaq.quantize_folded(W, s)
    assert np.array_equal(pf, packed) and np.array_equal(sbf, sb)
    assert np.float32(s_gf) == np.float32(np.float32(s_g) / np.float32(s))
    Wf, wf = uaq.fold(W, w, s)
    assert np.array_equal(wf, (w * np.float32(s)).astype(np.float32))
    # the folded layer (norm scale times s, backbone over s) gives the same y exactly
    y = olin.nvfp4_lora_linear(x, packed, sb, s_g, w_norm=w, eps=1e-6)
    yf = olin.nvfp4_lora_linear(x, pf, sbf, s_gf, w_norm=wf, eps=1e-6)
    assert np.array_equal(y, yf)


def test_uaq_factor_stays_within_the_nvfp4_error():
    W, x, w, z = _case(d_o=128, d_i=256, seed=2)
    packed, sb, s_g = onv.quantize(W)
    pf, sbf, s_gf = uaq.quantize_folded(W, uaq.UAQ_S)
    Wf, wf = uaq.fold(W, w, uaq.UAQ_S)
    ref = olin.nvfp4_lora_linear(x, packed, sb, s_g, w_norm=w, z=None, eps=1e-6)
    yf = olin.nvfp4_lora_linear(x, pf, sbf, s_gf, w_norm=wf, z=None, eps=1e-6)
    exact = olin.rmsnorm_aqn(x, w, None, 1e-6) @ W.astype(np.float64).T
    rms = np.sqrt(np.mean(exact ** 2))
    # both are NVFP4 approximations of the same exact product: each within the format's
    # error, so their difference is within twice the larger of the two
    e_ref, e_f = np.max(np.abs(ref - exact)), np.max(np.abs(yf - exact))
    assert e_f <= 2 * max(e_ref, 1e-3 * rms)
    assert np.max(np.abs(yf - ref)) <= e_ref + e_f
    # and the folded weight reconstructs W / s within the format's bound: per block of 16,
    # |w / s - w_hat| <= S = s_g s_b (the largest half-gap of the E2M1 grid is 1, 4 to 6)
    Wh = onv.dequantize(pf, sbf, s_gf)
    S = float(s_gf) * np.repeat(onv.E4M3_TABLE[sbf], onv.BLOCK, axis=1)
    assert np.all(np.abs(Wf.astype(np.float64) - Wh) <= S * (1 + 1e-6))
