"""Pins of the backward oracle (oracle/backward.py) to the forward oracle, which is
itself pinned: the adjoint identity of the linear map, central finite differences of
the whole path (RMSNorm-AQN + NVFP4 backbone + LoRA), exact differences in the adapter
parameters (the loss is linear in A for fixed B and in B for fixed A), and the
degenerate cases (no adapter, lambda = 0, no norm)."""

import numpy as np
import pytest

from oracle import backward as obw
from oracle import linear as olin
from oracle import nvfp4 as onv


def _case(d_o=48, d_i=64, M=5, r=4, seed=0, norm=True):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((d_o, d_i)) * 0.02).astype(np.float32)
    packed, sb, s_g = onv.quantize(W)
    x = rng.standard_normal((M, d_i))
    A = rng.standard_normal((r, d_i)) * 0.05
    B = rng.standard_normal((d_o, r)) * 0.05
    w = 1 + 0.1 * rng.standard_normal(d_i) if norm else None
    z = 1e-2 * rng.standard_normal(d_i) if norm else None
    g = rng.standard_normal((M, d_o))
    return dict(x=x, packed=packed, sb=sb, s_g=s_g, A=A, B=B, w=w, z=z, g=g, W_hat=onv.dequantize(packed, sb, s_g))


def _loss(c, x=None, A=None, B=None, lam=2.0):
    y = olin.nvfp4_lora_linear(c["x"] if x is None else x, c["packed"], c["sb"], c["s_g"],
                               c["A"] if A is None else A, c["B"] if B is None else B, lam, c["w"], c["z"], 1e-6)
    return float(np.sum(c["g"] * y))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_adjoint_identity_of_the_linear_map(seed):
    c = _case(seed=seed, norm=False)
    rng = np.random.default_rng(100 + seed)
    h = rng.standard_normal(c["x"].shape)
    y = olin.lora_linear_dense(h, c["W_hat"], c["A"], c["B"], 2.0)
    dh = obw.lora_backward_input(c["g"], c["W_hat"], c["A"], c["B"], 2.0)
    lhs, rhs = float(np.sum(c["g"] * y)), float(np.sum(dh * h))
    assert abs(lhs - rhs) <= 1e-12 * (abs(lhs) + 1.0)
    assert dh.shape == h.shape


@pytest.mark.parametrize("seed", [0, 1])
def test_input_gradient_matches_central_differences_through_the_norm(seed):
    c = _case(seed=seed)
    dx, _, _ = obw.nvfp4_lora_linear_backward(c["x"], c["g"], c["packed"], c["sb"], c["s_g"], c["A"], c["B"], 2.0,
                                              c["w"], c["z"], 1e-6)
    rng = np.random.default_rng(50 + seed)
    for _ in range(4):
        v = rng.standard_normal(c["x"].shape)
        eps = 1e-5
        fd = (_loss(c, x=c["x"] + eps * v) - _loss(c, x=c["x"] - eps * v)) / (2 * eps)
        an = float(np.sum(dx * v))
        assert abs(fd - an) <= 1e-7 * (abs(an) + 1e-3), (fd, an)
    # one coordinate at a time on a few entries: catches a mis-indexed row or channel
    for m, k in ((0, 0), (2, 17), (4, 63)):
        e = np.zeros_like(c["x"])
        e[m, k] = 1.0
        fd = (_loss(c, x=c["x"] + 1e-5 * e) - _loss(c, x=c["x"] - 1e-5 * e)) / 2e-5
        assert abs(fd - dx[m, k]) <= 1e-7 * (abs(dx[m, k]) + 1e-3)


def test_adapter_gradients_are_exact_differences():
    c = _case(seed=3)
    h = olin.rmsnorm_aqn(c["x"], c["w"], c["z"], 1e-6)
    dA, dB = obw.lora_adapter_grads(h, c["g"], c["A"], c["B"], 2.0)
    rng = np.random.default_rng(9)
    E = rng.standard_normal(c["A"].shape)
    F = rng.standard_normal(c["B"].shape)
    base = _loss(c)
    assert abs((_loss(c, A=c["A"] + E) - base) - float(np.sum(dA * E))) <= 1e-11 * (abs(base) + 1)
    assert abs((_loss(c, B=c["B"] + F) - base) - float(np.sum(dB * F))) <= 1e-11 * (abs(base) + 1)
    assert dA.shape == c["A"].shape and dB.shape == c["B"].shape


def test_degenerate_cases():
    c = _case(seed=4, norm=False)
    gw = c["g"] @ c["W_hat"]
    assert np.array_equal(obw.lora_backward_input(c["g"], c["W_hat"]), gw)  # no adapter
    assert np.allclose(obw.lora_backward_input(c["g"], c["W_hat"], c["A"], c["B"], 0.0), gw, rtol=0, atol=0)
    dx, dA, dB = obw.nvfp4_lora_linear_backward(c["x"], c["g"], c["packed"], c["sb"], c["s_g"])
    assert np.allclose(dx, gw, rtol=1e-15, atol=0) and dA is None and dB is None
    h = c["x"]
    dA0, dB0 = obw.lora_adapter_grads(h, c["g"], c["A"], c["B"], 0.0)
    assert not dA0.any() and not dB0.any()


def test_norm_backward_is_orthogonal_to_the_row_for_unit_scale():
    # with s = 1 and delta -> 0 the norm is scale invariant along x, so dx . x = 0
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 32))
    dh = rng.standard_normal((3, 32))
    dx = obw.rmsnorm_aqn_backward(x, np.ones(32), None, 0.0, dh)
    assert np.max(np.abs(np.sum(dx * x, axis=-1))) <= 1e-12
