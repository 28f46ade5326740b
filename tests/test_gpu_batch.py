"""Batches of independent calls (pl_nvfp4_lora_linear_batch) against the FP64 oracle.

Each call of a batch has its own input, batch size and weight; the decode-size batch runs
as one prologue and one main kernel over every call's weight tiles.  Every call must match
the oracle as a separate call would: max |y - y_ref| <= 1e-2 rms(y_ref)."""

import numpy as np
import pytest
import torch

from oracle import linear as olin
from precision_linear_gb300 import binding as pl
from precision_linear_gb300 import synthetic
from tests.gpu_cases import (DEV, assert_bf16_is_rounded_f32, assert_linear_close, make_case, np32,
                             oracle_quantize_cached, to_dev_nvfp4)

pytestmark = pytest.mark.gpu


def _batch_check(specs, lam=2.0):
    """specs: (d_o, d_i, M, r, seed, norm, z_rows); every call against the oracle."""
    calls, refs = [], []
    for d_o, d_i, M, r, seed, norm, z_rows in specs:
        case = make_case(d_o, d_i, M, r, 1e-2, seed)
        packed, sb, s_g = oracle_quantize_cached(("batch", d_o, d_i, seed), case["W"])
        codes, scales, sg = to_dev_nvfp4(packed, sb, s_g)
        z = case["z"]
        if z_rows:
            z = (torch.randn(M, d_i, generator=torch.Generator().manual_seed(seed)) * 1e-2).to(DEV)
        c = dict(x=case["x"], codes=codes, scales=scales, s_g=sg, A=case["A"] if r else None,
                 B=case["B"] if r else None, lam=lam, w_norm=case["w_norm"] if norm else None, z=z if norm else None)
        calls.append(c)
        f = lambda t: np32(t).astype(np.float64)
        refs.append(olin.nvfp4_lora_linear(f(case["x"]), packed, sb, s_g, f(case["A"]) if r else None,
                                           f(case["B"]) if r else None, lam, f(case["w_norm"]) if norm else None,
                                           f(z) if norm else None, synthetic.EPS))
    ys = pl.nvfp4_lora_linear_batch(calls, synthetic.EPS, out_dtype=torch.float32)
    yb = pl.nvfp4_lora_linear_batch(calls, synthetic.EPS)
    for i, (y, y16, ref) in enumerate(zip(ys, yb, refs)):
        what = f"batch call {i} {specs[i]}"
        assert_bf16_is_rounded_f32(y16, y, what)
        assert_linear_close(y, ref, what)
    assert pl.last_device_status() == 0
    return ys


def test_decode_sweep_as_one_batch(cuda_ok):
    """The 7B-shaped projection at M = 1, 8, 16, 32, 64, each call its own weight and input."""
    _batch_check([(3584, 3584, M, 32, 100 + M, True, False) for M in (1, 8, 16, 32, 64)])


def test_mixed_shapes_and_options(cuda_ok):
    _batch_check([(18944, 3584, 8, 32, 1, True, False), (512, 3584, 3, 5, 2, False, False),
                  (3584, 3584, 17, 0, 3, True, True), (200, 3584, 64, 64, 4, True, False)])


def test_batch_sharing_an_input_is_a_group(cuda_ok):
    """Two calls on the same x, norm and noise share one prologue pass; a third has its own."""
    case = make_case(3584, 3584, 12, 32, 1e-2, 9)
    other = make_case(512, 3584, 12, 32, 1e-2, 10)
    third = make_case(1024, 3584, 5, 16, 1e-2, 11)
    calls, refs = [], []
    for key, c_w, c_in in (("a", case, case), ("b", other, case), ("c", third, third)):
        packed, sb, s_g = oracle_quantize_cached(("share", key), c_w["W"])
        codes, scales, sg = to_dev_nvfp4(packed, sb, s_g)
        calls.append(dict(x=c_in["x"], codes=codes, scales=scales, s_g=sg, A=c_w["A"], B=c_w["B"], lam=2.0,
                          w_norm=c_in["w_norm"], z=c_in["z"]))
        f = lambda t: np32(t).astype(np.float64)
        refs.append(olin.nvfp4_lora_linear(f(c_in["x"]), packed, sb, s_g, f(c_w["A"]), f(c_w["B"]), 2.0,
                                           f(c_in["w_norm"]), f(c_in["z"]), synthetic.EPS))
    ys = pl.nvfp4_lora_linear_batch(calls, synthetic.EPS, out_dtype=torch.float32)
    for y, ref in zip(ys, refs):
        assert_linear_close(y, ref, "shared-input batch")


def test_full_batch_and_call_by_call_fallback(cuda_ok):
    """Eight calls with eight distinct inputs (the most one launch takes), and a batch with an
    M > 64 call, which runs one call after another."""
    _batch_check([(256, 512, 3 + i, 8, 20 + i, True, False) for i in range(8)])
    _batch_check([(256, 512, 100, 8, 40, True, False), (256, 512, 4, 8, 41, True, False)])


def test_batch_repeatable_bitwise(cuda_ok):
    a = _batch_check([(3584, 3584, M, 32, 200 + M, True, False) for M in (1, 64)])
    b = _batch_check([(3584, 3584, M, 32, 200 + M, True, False) for M in (1, 64)])
    assert all(torch.equal(u, v) for u, v in zip(a, b))
