"""W8A8 rollout linear (FP8 E4M3, per-channel weight and per-token activation scales)
against the oracle (oracle/w8a8.py, "QuRL: Low-Precision Reinforcement Learning for
Efficient Reasoning", reading notes, method / overall framework).

The weight quantiser must be bit-exact (codes and FP32 scales).  The linear is compared
on FP32 output with max |y - y_ref| <= 1e-2 rms(y_ref); y_ref quantises the activations
from the FP64 RMSNorm-AQN rounded to FP32, so a few activation codes may sit one E4M3 step
apart where h lies within FP32 rounding of a rounding boundary."""

import numpy as np
import pytest
import torch

from oracle import w8a8
from precision_linear_gb300 import binding as pl
from precision_linear_gb300 import synthetic
from tests.gpu_cases import DEV, assert_bf16_is_rounded_f32, assert_linear_close, np32

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


def _oracle(c_cpu, q_ref, s_ref, lam, norm=True, noise=True, lora=True, rows=None, z=None):
    x = np32(c_cpu["x"]).astype(np.float64)
    if rows is not None:
        x = x[rows]
        if z is not None and z.ndim == 2:
            z = z[rows]
    zz = z if z is not None else (np32(c_cpu["z"]) if noise else None)
    return w8a8.w8a8_linear(x, q_ref, s_ref, "fp8", np32(c_cpu["A"]) if lora else None,
                            np32(c_cpu["B"]) if lora else None, lam, np32(c_cpu["w_norm"]) if norm else None,
                            zz if norm else None, synthetic.EPS)


@pytest.mark.parametrize("d_o,d_i,M", [(3584, 3584, 1), (3584, 3584, 8), (3584, 3584, 64), (512, 3584, 16),
                                       (18944, 3584, 8), (3584, 18944, 32), (300, 384, 5), (1000, 1024, 300)])
def test_w8a8_linear_matches_oracle(cuda_ok, d_o, d_i, M):
    g, c = _case(d_o, d_i, M, 32, seed=d_o + M, outliers=1e-3)
    codes, s_w, q_ref, s_ref = _quant_check(c["W"])
    args = (g["x"], codes, s_w, g["A"], g["B"], 2.0, g["w_norm"], g["z"], synthetic.EPS)
    y = pl.w8a8_lora_linear(*args, out_dtype=torch.float32)
    yb = pl.w8a8_lora_linear(*args)
    assert_bf16_is_rounded_f32(yb, y, f"w8a8 {d_o}x{d_i} M={M}")
    assert_linear_close(y, _oracle(c, q_ref, s_ref, 2.0), f"w8a8 {d_o}x{d_i} M={M}")


@pytest.mark.parametrize("kw", [dict(lora=False), dict(norm=False), dict(noise=False)])
def test_w8a8_variants(cuda_ok, kw):
    d_o, d_i, M = 1024, 3584, 24
    g, c = _case(d_o, d_i, M, 16, seed=9)
    codes, s_w, q_ref, s_ref = _quant_check(c["W"])
    lora, norm, noise = kw.get("lora", True), kw.get("norm", True), kw.get("noise", True)
    y = pl.w8a8_lora_linear(g["x"], codes, s_w, g["A"] if lora else None, g["B"] if lora else None, 2.0,
                            g["w_norm"] if norm else None, g["z"] if (norm and noise) else None, synthetic.EPS,
                            out_dtype=torch.float32)
    assert_linear_close(y, _oracle(c, q_ref, s_ref, 2.0, norm, noise, lora), f"w8a8 {kw}")


def test_w8a8_per_token_states_and_odd_rank(cuda_ok):
    d_o, d_i, M = 640, 1024, 12
    g, c = _case(d_o, d_i, M, 5, seed=4)
    codes, s_w, q_ref, s_ref = _quant_check(c["W"])
    z = (torch.randn(M, d_i, generator=torch.Generator().manual_seed(1)) * 1e-2)
    y = pl.w8a8_lora_linear(g["x"], codes, s_w, g["A"], g["B"], 2.0, g["w_norm"], z.to(DEV), synthetic.EPS,
                            out_dtype=torch.float32)
    assert_linear_close(y, _oracle(c, q_ref, s_ref, 2.0, z=np32(z)), "w8a8 per-token states")


def test_w8a8_m4096_sampled_rows(cuda_ok):
    """The 7B q projection at M = 4096: one full 128-token tile and a spread of rows."""
    d_o, d_i, M = 3584, 3584, 4096
    g, c = _case(d_o, d_i, M, 32, seed=44)
    codes, s_w, q_ref, s_ref = _quant_check(c["W"])
    y = pl.w8a8_lora_linear(g["x"], codes, s_w, g["A"], g["B"], 2.0, g["w_norm"], g["z"], synthetic.EPS,
                            out_dtype=torch.float32)
    rows = np.unique(np.concatenate([np.arange(256, 384), np.random.default_rng(3).choice(M, 32, replace=False)]))
    assert_linear_close(y[torch.from_numpy(rows).to(DEV)], _oracle(c, q_ref, s_ref, 2.0, rows=rows), "w8a8 M=4096")
    assert pl.last_device_status() == 0


def test_w8a8_repeatable_bitwise(cuda_ok):
    g, c = _case(3584, 3584, 64, 32, seed=2)
    codes, s_w = pl.w8a8_quantize_weight(g["W"])
    ys = [pl.w8a8_lora_linear(g["x"], codes, s_w, g["A"], g["B"], 2.0, g["w_norm"], g["z"]) for _ in range(3)]
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])
