"""GPU RMSNorm-AQN vs the FP64 oracle, elementwise relative error <= 2e-3."""

import numpy as np
import pytest
import torch

from oracle import linear as olin
from precision_linear_gb300 import binding as pl
from precision_linear_gb300 import synthetic
from tests.gpu_cases import DEV, NORM_REL_TOL, assert_bf16_is_rounded_f32, np32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,d", [(1, 256), (4, 256), (64, 3584), (7, 5120), (3, 18944), (4096, 3584), (2, 8),
                                 (5, 24)])
@pytest.mark.parametrize("noise", [True, False])
def test_rmsnorm_aqn_matches_oracle(cuda_ok, M, d, noise):
    x = synthetic.activations(M, d, seed=M + d)
    w = synthetic.norm_scale(d, seed=d)
    z = synthetic.noise(d, 1e-2, seed=d) if noise else None
    args = (x.to(DEV), w.to(DEV), z.to(DEV) if noise else None, synthetic.EPS)
    h = pl.rmsnorm_aqn(*args, out_dtype=torch.float32)
    hb = pl.rmsnorm_aqn(*args)
    assert_bf16_is_rounded_f32(hb, h, f"M={M} d={d}")
    ref = olin.rmsnorm_aqn(np32(x), np32(w), np32(z) if noise else None, synthetic.EPS)
    got = np32(h).astype(np.float64)
    rel = np.abs(got - ref) / np.maximum(np.abs(ref), 1e-30)
    assert float(rel.max()) <= NORM_REL_TOL, float(rel.max())


def test_rmsnorm_noise_changes_output_and_zero_noise_does_not(cuda_ok):
    x = synthetic.activations(8, 3584, seed=1).to(DEV)
    w = synthetic.norm_scale(3584, seed=1).to(DEV)
    z = synthetic.noise(3584, 1e-2, seed=1).to(DEV)
    h0 = pl.rmsnorm_aqn(x, w, None)
    hz0 = pl.rmsnorm_aqn(x, w, torch.zeros_like(z))
    hz = pl.rmsnorm_aqn(x, w, z)
    assert torch.equal(h0, hz0)
    assert not torch.equal(h0, hz)
