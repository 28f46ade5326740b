"""GPU UAQ fold (pl_nvfp4_quantize_uaq, pl_uaq_fold_norm) vs the oracle (oracle/uaq.py):
the folded weight's codes, block scales and tensor scale bit for bit, the folded norm
scale bit for bit, and the folded layer through the linear within the linear's bound."""

import numpy as np
import pytest
import torch

from oracle import linear as olin
from oracle import uaq
from precision_linear_gb300 import binding as pl
from precision_linear_gb300 import synthetic
from tests.gpu_cases import DEV, assert_linear_close, np32

pytestmark = pytest.mark.gpu


def _check_fold(W, s):
    codes, scales, s_g = pl.nvfp4_quantize_uaq(W, s)
    torch.cuda.synchronize()
    packed, sb, sg_ref = uaq.quantize_folded(np32(W), s)
    got = np.float32(s_g.item())
    assert got.view(np.uint32) == np.float32(sg_ref).view(np.uint32), (got, sg_ref)
    bad_s = int((scales.cpu().numpy() != sb).sum())
    bad_c = int((codes.cpu().numpy() != packed).sum())
    assert bad_s == 0 and bad_c == 0, f"s={s}: {bad_s} scale and {bad_c} code-byte mismatches"
    return codes, scales, s_g, packed, sb, sg_ref


@pytest.mark.parametrize("d_o,d_i,outliers", [(3584, 3584, 1e-3), (512, 3584, 0.0), (129, 272, 1e-2), (1, 16, 0.0)])
@pytest.mark.parametrize("s", [1.5, 2.0, 0.75])
def test_folded_quantiser_bit_exact(cuda_ok, d_o, d_i, outliers, s):
    W = synthetic.weight(d_o, d_i, seed=d_o + 3 * d_i, outlier_frac=outliers).to(DEV)
    _check_fold(W, s)


def test_fold_by_one_is_the_plain_quantiser_and_by_two_only_halves_s_g(cuda_ok):
    W = synthetic.weight(1024, 512, seed=5).to(DEV)
    c0, s0, g0 = pl.nvfp4_quantize(W)
    c1, s1, g1 = pl.nvfp4_quantize_uaq(W, 1.0)
    c2, s2, g2 = pl.nvfp4_quantize_uaq(W, 2.0)
    assert torch.equal(c0, c1) and torch.equal(s0, s1) and torch.equal(g0, g1)
    assert torch.equal(c0, c2) and torch.equal(s0, s2) and float(g2.item()) == float(g0.item()) / 2


def test_folded_norm_scale_bit_exact(cuda_ok):
    w = synthetic.norm_scale(3584, seed=9).to(DEV)
    for s in (1.5, 2.0, 0.7):
        got = pl.uaq_fold_norm(w, s)
        _, want = uaq.fold(np.zeros((1, 3584), np.float32), np32(w), s)
        assert np.array_equal(np32(got).view(np.uint32), want.view(np.uint32))
    inplace = w.clone()
    pl.uaq_fold_norm(inplace, 1.5, out=inplace)
    assert torch.equal(inplace, pl.uaq_fold_norm(w, 1.5))


def test_folded_layer_through_the_linear(cuda_ok):
    d, M, r, s = 3584, 8, 32, uaq.UAQ_S
    c = synthetic.projection_case(d, d, M, r, 1e-2, 21, 0.0, device="cpu")
    g = {k: v.to(DEV) for k, v in c.items()}
    codes, scales, s_g, packed, sb, sg_ref = _check_fold(g["W"], s)
    w_f = pl.uaq_fold_norm(g["w_norm"], s)
    y = pl.nvfp4_lora_linear(g["x"], codes, scales, s_g, g["A"], g["B"], 2.0, w_f, g["z"], synthetic.EPS,
                             out_dtype=torch.float32)
    _, w_ref = uaq.fold(np32(c["W"]), np32(c["w_norm"]), s)
    ref = olin.nvfp4_lora_linear(np32(c["x"]).astype(np.float64), packed, sb, sg_ref, np32(c["A"]), np32(c["B"]), 2.0,
                                 w_ref, np32(c["z"]), synthetic.EPS)
    assert_linear_close(y, ref, "folded layer")
