"""GPU AQN noise draws (pl_aqn_noise) vs the oracle (oracle/aqn.py), and the drawn
state fed through the RMSNorm-AQN and the linear.

Tolerance of the draws: both sides take the same Philox words and the same 23-bit
uniforms (exact in FP32), so they differ only by FP32 rounding on the GPU: logf and
sincospif (at most 1 ulp each per the CUDA math documentation), the IEEE square root
and three products (half an ulp each), about 4 ulp of the result in all, 2.4e-7
relative.  The test allows |z - z_ref| <= 2e-6 |z_ref| + 2e-6 sigma: eight times that,
and far below the O(sigma) difference of any wrong word, lane or counter."""

import numpy as np
import pytest
import torch

from oracle import aqn
from oracle import linear as olin
from precision_linear_gb300 import binding as pl
from precision_linear_gb300 import synthetic
from tests.gpu_cases import (DEV, NORM_REL_TOL, assert_linear_close, make_case, np32, oracle_linear,
                             oracle_quantize_cached, to_dev_nvfp4)

pytestmark = pytest.mark.gpu

RTOL, ATOL_SIGMA = 2e-6, 2e-6


def _assert_draws_close(got, want, sig, what):
    err = np.abs(np32(got).astype(np.float64) - want)
    lim = RTOL * np.abs(want) + ATOL_SIGMA * sig
    bad = int((err > lim).sum())
    assert bad == 0, f"{what}: {bad} of {err.size} draws off (max err {err.max():.3e})"


@pytest.mark.parametrize("seed,norm_id,scope0,n_scopes,d,sig", [
    (2024, 0, 0, 1, 3584, 0.01),              # one per-rollout state of a 7B norm
    (7, 3, 5, 4, 18944, 0.0005),              # several scopes, the schedule's last stage
    ((1 << 40) | 123, 63, (1 << 32) - 2, 4, 1001, 0.05),  # scope crosses the low word; ragged d
    (9, 1, 0, 3, 27651, 0.001),               # 32B intermediate width, ragged
    (1, 0, 0, 1, 1, 1.0),                     # one channel
    (11, 5, 0, 64, 5120, 0.00687656),         # one state per token of a 64-token batch
])
def test_noise_matches_oracle(cuda_ok, seed, norm_id, scope0, n_scopes, d, sig):
    sig32 = float(np.float32(sig))
    z = pl.aqn_noise(d, seed, norm_id, scope0, n_scopes, sig32, device=DEV)
    torch.cuda.synchronize()
    ref = aqn.noise(seed, norm_id, scope0, n_scopes, d, sig32)
    _assert_draws_close(z, ref, sig32, f"seed={seed} norm={norm_id} scope0={scope0} n={n_scopes} d={d}")


def test_noise_zero_sigma_and_repeatability(cuda_ok):
    z0 = pl.aqn_noise(4096, 5, 2, 0, 2, 0.0, device=DEV)
    assert float(z0.abs().max()) == 0.0
    a = pl.aqn_noise(4096, 5, 2, 0, 2, 0.01, device=DEV)
    b = pl.aqn_noise(4096, 5, 2, 0, 2, 0.01, device=DEV)
    assert torch.equal(a, b)
    row1 = pl.aqn_noise(4096, 5, 2, 1, 1, 0.01, device=DEV)
    assert torch.equal(row1[0], a[1])  # a scope's state does not depend on its neighbours


def test_drawn_state_through_norm_and_linear(cuda_ok):
    """Stage 3 of the 0.01 -> 0.0005 schedule, drawn on the device, as the z of the
    RMSNorm-AQN and of the decode linear; the oracle uses its own draw of the state."""
    d, d_o, M, r, seed = 3584, 3584, 8, 32, 77
    sig = pl.aqn_sigma(3, 0.01, 0.0005)
    z_dev = pl.aqn_noise(d, seed, 0, 0, 1, sig, device=DEV)[0]
    z_ref = aqn.noise(seed, 0, 0, 1, d, sig)[0].astype(np.float32)

    x = synthetic.activations(M, d, seed=3)
    w = synthetic.norm_scale(d, seed=4)
    h = pl.rmsnorm_aqn(x.to(DEV), w.to(DEV), z_dev, synthetic.EPS, out_dtype=torch.float32)
    ref = olin.rmsnorm_aqn(np32(x), np32(w), z_ref, synthetic.EPS)
    rel = np.abs(np32(h).astype(np.float64) - ref) / np.maximum(np.abs(ref), 1e-30)
    assert float(rel.max()) <= NORM_REL_TOL

    case = make_case(d_o, d, M, r, 1e-2, seed, 0.0)
    packed, sb, s_g = oracle_quantize_cached((d_o, d, seed, 0.0), case["W"])
    dev_w = to_dev_nvfp4(packed, sb, s_g)
    y = pl.nvfp4_lora_linear(case["x"], *dev_w, case["A"], case["B"], 2.0, case["w_norm"], z_dev, synthetic.EPS,
                             out_dtype=torch.float32)
    ref_case = dict(case)
    ref_case["z"] = torch.from_numpy(z_ref)
    assert_linear_close(y, oracle_linear(ref_case, packed, sb, s_g, 2.0), "linear with the drawn z")
