"""W8A8 rollout linear (FP8 E4M3, per-channel weight and per-token activation scales)
against the oracle (oracle/w8a8.py, "QuRL: Low-Precision Reinforcement Learning for
Efficient Reasoning", reading notes, method / overall framework).

The weight quantiser must be bit-exact (codes and FP32 scales).  The linear is compared
on FP32 output with |y - y_ref| <= 1e-2 rms(y_ref) + allowance.  The activation codes are
an integer decision taken on FP32 values of h: where the exact quotient h / s_x lies
within a few FP32 ulps of a midpoint between two E4M3 values, either code is a correct
result (the kernel's FP32 h and the oracle's FP32 rounding of its FP64 h may differ by an
ulp).  For those elements only, the allowance admits the other code: one E4M3 step times
s_x s_w |q_w| per output.  The test also requires such elements to be rare (<= 1e-3)."""

import numpy as np
import pytest
import torch

from oracle import linear as olin
from oracle import w8a8
from oracle.nvfp4 import E4M3_TABLE
from precision_linear_gb300 import binding as pl
from precision_linear_gb300 import synthetic
from tests.gpu_cases import DEV, LINEAR_TOL, assert_bf16_is_rounded_f32, np32

pytestmark = pytest.mark.gpu


def _quant_check(W):
    codes, s_w = pl.w8a8_quantize_weight(W.to(DEV))
    q_ref, s_ref = w8a8.quantize_fp8_rows(np32(W))
    assert np.array_equal(s_w.cpu().numpy().view(np.uint32), s_ref.view(np.uint32)), "s_w differs"
    got = codes.cpu().numpy()
    bad = int((got != q_ref).sum())
    assert bad == 0, f"{bad} codes differ"
    return codes, s_w, q_ref, s_ref


@pytest.mark.parametrize("d_o,d_i,outliers", [(3584, 3584, 1e-3), (18944, 3584, 0.0), (512, 3584, 0.0),
                                              (37, 272, 0.0), (3, 16, 0.0)])
def test_weight_quantiser_bit_exact(cuda_ok, d_o, d_i, outliers):
    _quant_check(synthetic.weight(d_o, d_i, seed=d_o + d_i, outlier_frac=outliers))


def test_weight_quantiser_edge_rows(cuda_ok):
    rng = np.random.default_rng(5)
    W = rng.standard_normal((8, 64)).astype(np.float32) * 0.02
    W[0] = 0.0                                   # zero row: s = 1, codes +0
    W[1, :] = -0.0
    W[2, 0] = 448.0                              # s = 1 exactly: codes are E4M3 of the values
    W[3] = np.linspace(-1e-30, 1e-30, 64)         # tiny values that round to zero keep no sign
    W[3, 5] = 1e-3
    W[4, 1] = -3e4                               # large magnitudes
    W[5] = 2.0 ** np.arange(-20, 44)[:64] * 1e-9  # a wide dynamic range in one row
    Wb = torch.from_numpy(W).to(torch.bfloat16)
    codes, s_w, _, _ = _quant_check(Wb)
    assert float(s_w[0]) == 1.0 and int(codes[0].max()) == 0 and int(codes[1].max()) == 0


def _case(d_o, d_i, M, r, seed, outliers=0.0):
    c = synthetic.projection_case(d_o, d_i, M, r, 1e-2, seed, outliers)
    return {k: v.to(DEV) for k, v in c.items()}, c


_E4M3_POS = np.unique(np.abs(E4M3_TABLE[np.isfinite(E4M3_TABLE)]))  # 0 .. 448, ascending
_MIDS = (_E4M3_POS[:-1] + _E4M3_POS[1:]) / 2
_AMBIG_REL = 2.0 ** -19  # 16 FP32 ulps of the quotient


def _allowance(h, q_ref, s_ref):
    """Per output [M, d_o]: one E4M3 step s_x s_w |q_w| summed over the activations whose exact
    quotient 448 h / max|h| sits within _AMBIG_REL of a rounding midpoint; and their fraction."""
    amax = np.max(np.abs(h), axis=1, keepdims=True)
    amax = np.where(amax > 0, amax, 1.0)
    v = np.abs(448.0 * h / amax)
    i = np.clip(np.searchsorted(_MIDS, v), 1, len(_MIDS) - 1)
    near = np.where(np.abs(v - _MIDS[i - 1]) < np.abs(v - _MIDS[i]), i - 1, i)
    amb = np.abs(v - _MIDS[near]) <= _AMBIG_REL * np.maximum(v, 1e-30)
    step = np.where(amb, _E4M3_POS[near + 1] - _E4M3_POS[near], 0.0)
    s_x = amax[:, 0] / 448.0
    wq = np.abs(E4M3_TABLE[q_ref]) * s_ref[:, None].astype(np.float64)
    return (step * s_x[:, None]) @ wq.T, float(amb.mean())


def _oracle(c_cpu, q_ref, s_ref, lam, norm=True, noise=True, lora=True, rows=None, z=None):
    x = np32(c_cpu["x"]).astype(np.float64)
    if rows is not None:
        x = x[rows]
        if z is not None and z.ndim == 2:
            z = z[rows]
    zz = z if z is not None else (np32(c_cpu["z"]) if noise else None)
    w = np32(c_cpu["w_norm"]) if norm else None
    y = w8a8.w8a8_linear(x, q_ref, s_ref, "fp8", np32(c_cpu["A"]) if lora else None,
                         np32(c_cpu["B"]) if lora else None, lam, w, zz if norm else None, synthetic.EPS)
    if not norm:
        # without the norm both sides quantise the same FP32 values (h = x, BF16) with the same
        # FP32 operations: the codes are unique and no allowance applies
        return y, np.zeros_like(y)
    h = olin.rmsnorm_aqn(x, w, zz, synthetic.EPS)
    allow, frac = _allowance(h, q_ref, s_ref)
    assert frac <= 1e-3, f"{frac:.2e} of the activations sit at an FP32-ambiguous rounding midpoint"
    return y, allow


def _assert_close(y_gpu, ref, what):
    y_ref, allow = ref
    y = np32(y_gpu).astype(np.float64)
    assert y.shape == y_ref.shape and np.all(np.isfinite(y)), what
    rms = float(np.sqrt(np.mean(y_ref * y_ref)))
    excess = np.abs(y - y_ref) - (LINEAR_TOL * rms + allow)
    assert float(excess.max()) <= 0.0, (f"{what}: max |y - y_ref| {np.abs(y - y_ref).max():.3e}, "
                                         f"bound {LINEAR_TOL} * rms {rms:.3e} + allowance")


@pytest.mark.parametrize("d_o,d_i,M", [(3584, 3584, 1), (3584, 3584, 8), (3584, 3584, 64), (512, 3584, 16),
                                       (18944, 3584, 8), (3584, 18944, 32), (300, 384, 5), (1000, 1024, 300)])
def test_w8a8_linear_matches_oracle(cuda_ok, d_o, d_i, M):
    g, c = _case(d_o, d_i, M, 32, seed=d_o + M, outliers=1e-3)
    codes, s_w, q_ref, s_ref = _quant_check(c["W"])
    args = (g["x"], codes, s_w, g["A"], g["B"], 2.0, g["w_norm"], g["z"], synthetic.EPS)
    y = pl.w8a8_lora_linear(*args, out_dtype=torch.float32)
    yb = pl.w8a8_lora_linear(*args)
    assert_bf16_is_rounded_f32(yb, y, f"w8a8 {d_o}x{d_i} M={M}")
    _assert_close(y, _oracle(c, q_ref, s_ref, 2.0), f"w8a8 {d_o}x{d_i} M={M}")


@pytest.mark.parametrize("kw", [dict(lora=False), dict(norm=False), dict(noise=False)])
def test_w8a8_variants(cuda_ok, kw):
    d_o, d_i, M = 1024, 3584, 24
    g, c = _case(d_o, d_i, M, 16, seed=9)
    codes, s_w, q_ref, s_ref = _quant_check(c["W"])
    lora, norm, noise = kw.get("lora", True), kw.get("norm", True), kw.get("noise", True)
    y = pl.w8a8_lora_linear(g["x"], codes, s_w, g["A"] if lora else None, g["B"] if lora else None, 2.0,
                            g["w_norm"] if norm else None, g["z"] if (norm and noise) else None, synthetic.EPS,
                            out_dtype=torch.float32)
    _assert_close(y, _oracle(c, q_ref, s_ref, 2.0, norm, noise, lora), f"w8a8 {kw}")


def test_w8a8_per_token_states_and_odd_rank(cuda_ok):
    d_o, d_i, M = 640, 1024, 12
    g, c = _case(d_o, d_i, M, 5, seed=4)
    codes, s_w, q_ref, s_ref = _quant_check(c["W"])
    z = (torch.randn(M, d_i, generator=torch.Generator().manual_seed(1)) * 1e-2)
    y = pl.w8a8_lora_linear(g["x"], codes, s_w, g["A"], g["B"], 2.0, g["w_norm"], z.to(DEV), synthetic.EPS,
                            out_dtype=torch.float32)
    _assert_close(y, _oracle(c, q_ref, s_ref, 2.0, z=np32(z)), "w8a8 per-token states")


def test_w8a8_m4096_sampled_rows(cuda_ok):
    """The 7B q projection at M = 4096: one full 128-token tile and a spread of rows."""
    d_o, d_i, M = 3584, 3584, 4096
    g, c = _case(d_o, d_i, M, 32, seed=44)
    codes, s_w, q_ref, s_ref = _quant_check(c["W"])
    y = pl.w8a8_lora_linear(g["x"], codes, s_w, g["A"], g["B"], 2.0, g["w_norm"], g["z"], synthetic.EPS,
                            out_dtype=torch.float32)
    rows = np.unique(np.concatenate([np.arange(256, 384), np.random.default_rng(3).choice(M, 32, replace=False)]))
    _assert_close(y[torch.from_numpy(rows).to(DEV)], _oracle(c, q_ref, s_ref, 2.0, rows=rows), "w8a8 M=4096")
    assert pl.last_device_status() == 0


@pytest.mark.parametrize("kw", [dict(lora=False), dict(norm=False), dict(rows=True)])
def test_w8a8_large_m_variants(cuda_ok, kw):
    """M > 64 (the persistent kernel, ragged last token and weight tiles): no adapter, no norm,
    and per-token states with an odd rank."""
    d_o, d_i, M = 640, 1024, 300
    r = 5 if kw.get("rows") else 16
    g, c = _case(d_o, d_i, M, r, seed=31)
    codes, s_w, q_ref, s_ref = _quant_check(c["W"])
    lora, norm = kw.get("lora", True), kw.get("norm", True)
    z, z_ref = g["z"], None
    if kw.get("rows"):
        zt = torch.randn(M, d_i, generator=torch.Generator().manual_seed(3)) * 1e-2
        z, z_ref = zt.to(DEV), np32(zt)
    y = pl.w8a8_lora_linear(g["x"], codes, s_w, g["A"] if lora else None, g["B"] if lora else None, 2.0,
                            g["w_norm"] if norm else None, z if norm else None, synthetic.EPS, out_dtype=torch.float32)
    ref = _oracle(c, q_ref, s_ref, 2.0, norm, norm, lora) if z_ref is None else _oracle(c, q_ref, s_ref, 2.0, z=z_ref)
    _assert_close(y, ref, f"w8a8 large M {kw}")
    assert pl.last_device_status() == 0


def test_w8a8_repeatable_bitwise(cuda_ok):
    g, c = _case(3584, 3584, 64, 32, seed=2)
    codes, s_w = pl.w8a8_quantize_weight(g["W"])
    ys = [pl.w8a8_lora_linear(g["x"], codes, s_w, g["A"], g["B"], 2.0, g["w_norm"], g["z"]) for _ in range(3)]
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])
    g, c = _case(1000, 1024, 300, 32, seed=3)  # the persistent large-M kernel
    codes, s_w = pl.w8a8_quantize_weight(g["W"])
    ys = [pl.w8a8_lora_linear(g["x"], codes, s_w, g["A"], g["B"], 2.0, g["w_norm"], g["z"]) for _ in range(3)]
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])
