"""Frozen-backbone backward (pl_nvfp4_lora_linear_backward) against the FP64 oracle
(oracle/backward.py; "QeRL: When Quantized Weights Help Reinforcement Learning, and Where
the Evidence Stops", section 2.1: the gradients train A and B and pass through the frozen
quantised projection; section 5.1's RMSNorm-AQN prologue is differentiated in x).

Bound, for each of dx, dA and dB: |d - d_ref| <= 1e-2 rms(d_ref) + e, e an element-wise
bound of the kernels' arithmetic computed from the oracle's FP64 intermediates.  The kernels
feed the tensor cores BF16 operands: W_hat (exact in BF16) and g (given in BF16) carry no
rounding; h, u = lambda g B and lambda h A^T are rounded once to BF16 (relative 2^-9 each,
after FP32 sums of d terms, n 2^-24 of the absolute terms), and every contraction
accumulates in FP32 (again n 2^-24 of its absolute terms).  With few tokens (M = 4) the
rounding of u and h does not average out, and e is what admits it; a wrong index, sign or
operand breaks both terms by orders of magnitude."""

import numpy as np
import pytest
import torch

from oracle import backward as obw
from precision_linear_gb300 import binding as pl
from precision_linear_gb300 import synthetic
from tests.gpu_cases import DEV, LINEAR_TOL, make_case, np32, oracle_quantize_cached, to_dev_nvfp4

pytestmark = pytest.mark.gpu


def _grad(M, d_o, seed):
    g = torch.randn(M, d_o, generator=torch.Generator().manual_seed(seed))
    return g.to(torch.bfloat16)


U_BF16 = 2.0 ** -9   # unit roundoff of BF16
U_F32 = 2.0 ** -24


def _bounds(x, g, W_hat, A, B, lam, w, z, eps):
    """Element-wise error bounds (dx, dA, dB) of the kernels' arithmetic, in FP64."""
    from oracle import backward as ob
    from oracle import linear as ol
    M, d_i = x.shape
    d_o = g.shape[1]
    h = ol.rmsnorm_aqn(x, w, z, eps) if w is not None else x
    ag, ah = np.abs(g), np.abs(h)
    b_dh = d_o * U_F32 * (ag @ np.abs(W_hat))
    b_dA = b_dB = None
    if A is not None:
        r = A.shape[0]
        u = lam * (g @ B)
        au = np.abs(u) + lam * d_o * U_F32 * (ag @ np.abs(B))  # |u| with its FP32 sum error
        lt = lam * np.abs(h) @ np.abs(A).T                      # |lambda t| terms
        at = np.abs(lam * (h @ A.T)) + d_i * U_F32 * lt
        b_dh = b_dh + (U_BF16 + r * U_F32) * (au @ np.abs(A))
        b_dA = (2 * U_BF16 + M * U_F32) * (au.T @ ah)
        b_dB = (2 * U_BF16 + M * U_F32) * (ag.T @ at)
    if w is None:
        return b_dh, b_dA, b_dB
    s = w + (z if z is not None else 0.0)
    rho = ol.rms_factor(x, eps)[:, None]
    proj = np.abs(x * s) @ np.ones((d_i, 1))
    b_dx = rho * np.abs(s) * b_dh + rho ** 3 * np.abs(x) * ((np.abs(x * s) * b_dh).sum(axis=1, keepdims=True)) / d_i
    dh = ob.lora_backward_input(g, W_hat, A, B, lam)
    b_dx = b_dx + 8 * U_F32 * (rho * np.abs(s) * np.abs(dh) + rho ** 3 * np.abs(x) * proj * np.abs(dh).max() / d_i)
    return b_dx, b_dA, b_dB


def _close(got, ref, what, bound=None):
    assert got is not None and ref is not None, what
    d = np32(got).astype(np.float64)
    assert d.shape == ref.shape and np.all(np.isfinite(d)), what
    rms = float(np.sqrt(np.mean(ref * ref)))
    lim = LINEAR_TOL * rms + (bound if bound is not None else 0.0)
    excess = np.abs(d - ref) - lim
    assert float(excess.max()) <= 0.0, (f"{what}: max err {np.abs(d - ref).max():.3e}, "
                                        f"{LINEAR_TOL} * rms {LINEAR_TOL * rms:.3e} + element bound")


def _check(d_o, d_i, M, r, seed=0, norm=True, noise=True, lora=True, z_rows=False, rows=None):
    case = make_case(d_o, d_i, M, r, 1e-2, seed)
    packed, sb, s_g = oracle_quantize_cached(("bwd", d_o, d_i, seed), case["W"])
    codes, scales, sg = to_dev_nvfp4(packed, sb, s_g)
    g = _grad(M, d_o, seed + 1)
    z = None
    if norm and noise:
        z = case["z"]
        if z_rows:
            z = (torch.randn(M, d_i, generator=torch.Generator().manual_seed(seed + 2)) * 1e-2).to(DEV)
    dx, dA, dB = pl.nvfp4_lora_linear_backward(g.to(DEV), case["x"], codes, scales, sg,
                                               case["A"] if lora else None, case["B"] if lora else None, 2.0,
                                               case["w_norm"] if norm else None, z, synthetic.EPS)
    f = lambda t: np32(t).astype(np.float64)
    rdx, rdA, rdB = obw.nvfp4_lora_linear_backward(f(case["x"]), f(g), packed, sb, s_g,
                                                   f(case["A"]) if lora else None, f(case["B"]) if lora else None,
                                                   2.0, f(case["w_norm"]) if norm else None,
                                                   f(z) if z is not None else None, synthetic.EPS)
    what = f"backward d_o={d_o} d_i={d_i} M={M} r={r} norm={norm} noise={noise} lora={lora}"
    from oracle import nvfp4 as onv
    bx, bA, bB = _bounds(f(case["x"]), f(g), onv.dequantize(packed, sb, s_g), f(case["A"]) if lora else None,
                         f(case["B"]) if lora else None, 2.0, f(case["w_norm"]) if norm else None,
                         f(z) if z is not None else None, synthetic.EPS)
    if rows is None:
        _close(dx, rdx, what + " dx", bx)
    else:
        _close(dx[torch.from_numpy(rows).to(DEV)], rdx[rows], what + " dx (sampled rows)", bx[rows])
    if lora:
        _close(dA, rdA, what + " dA", bA)
        _close(dB, rdB, what + " dB", bB)
    else:
        assert dA is None and dB is None
    assert pl.last_device_status() == 0


def test_backward_tiny(cuda_ok):
    _check(256, 256, 4, 8)


@pytest.mark.parametrize("d_o,d_i", [(3584, 3584), (18944, 3584), (3584, 18944), (512, 3584)])
def test_backward_7b_shapes_m64(cuda_ok, d_o, d_i):
    _check(d_o, d_i, 64, 32, seed=d_o + d_i)


@pytest.mark.parametrize("kw", [dict(norm=False), dict(lora=False), dict(noise=False), dict(z_rows=True)])
def test_backward_variants(cuda_ok, kw):
    _check(1024, 2048, 40, 16, seed=7, **kw)


@pytest.mark.parametrize("d_o,d_i,M,r", [(200, 512, 300, 5), (136, 256, 129, 64), (1000, 1280, 1, 1)])
def test_backward_ragged(cuda_ok, d_o, d_i, M, r):
    _check(d_o, d_i, M, r, seed=d_o + M)


def test_backward_m4096_q_projection(cuda_ok):
    """The 7B q projection at M = 4096: dA, dB in full, dx on two full 128-token tiles and a
    spread of rows."""
    rows = np.unique(np.concatenate([np.arange(0, 128), np.arange(1920, 2048),
                                     np.random.default_rng(2).choice(4096, 32, replace=False)]))
    _check(3584, 3584, 4096, 32, seed=11, rows=rows)


def test_backward_repeatable_bitwise(cuda_ok):
    case = make_case(512, 1024, 100, 32, 1e-2, 3)
    codes, scales, sg = pl.nvfp4_quantize(case["W"])
    g = _grad(100, 512, 4).to(DEV)
    outs = [pl.nvfp4_lora_linear_backward(g, case["x"], codes, scales, sg, case["A"], case["B"], 2.0, case["w_norm"],
                                          case["z"], synthetic.EPS) for _ in range(3)]
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    for a, b in zip(outs[0], outs[2]):
        assert torch.equal(a, b)
