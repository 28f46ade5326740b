"""One AQN noise state per token row: the RMSNorm-AQN and the linear with z [M, d].

The pages let the caller declare the persistence scope of the noise state -- per
rollout, per response or per token ("QeRL: When Quantized Weights Help Reinforcement
Learning, and Where the Evidence Stops", section 6, "A training algorithm that exposes
the stochastic state").  In a batched decode call each row is a different response (or
token), so each row takes its own state.  Here the states are drawn on the device by
pl_aqn_noise (one scope per row) and fed through every kernel path of the linear; the
oracle draws the same states itself (oracle/aqn.py) and computes the FP64 result."""

import numpy as np
import pytest
import torch

from oracle import aqn
from oracle import linear as olin
from precision_linear_gb300 import binding as pl
from precision_linear_gb300 import synthetic
from tests.gpu_cases import (DEV, NORM_REL_TOL, assert_bf16_is_rounded_f32, assert_linear_close, make_case, np32,
                             oracle_linear, oracle_quantize_cached, to_dev_nvfp4)

pytestmark = pytest.mark.gpu


def _states(seed, norm_id, scope0, M, d, sig, rows=None):
    """Device states [M, d] from pl_aqn_noise and the oracle's own draw (FP32 values)."""
    z_dev = pl.aqn_noise(d, seed, norm_id, scope0, M, sig, device=DEV)
    if rows is None:
        z_ref = aqn.noise(seed, norm_id, scope0, M, d, sig)
    else:
        z_ref = np.stack([aqn.noise(seed, norm_id, scope0 + int(m), 1, d, sig)[0] for m in rows])
    return z_dev, z_ref.astype(np.float32)


@pytest.mark.parametrize("M,d", [(8, 3584), (64, 3584), (5, 18944), (3, 24)])
def test_rmsnorm_rows_match_oracle(cuda_ok, M, d):
    sig = float(np.float32(1e-2))
    z_dev, z_ref = _states(1234, 0, 100, M, d, sig)
    x = synthetic.activations(M, d, seed=M + d)
    w = synthetic.norm_scale(d, seed=d)
    h = pl.rmsnorm_aqn(x.to(DEV), w.to(DEV), z_dev, synthetic.EPS, out_dtype=torch.float32)
    hb = pl.rmsnorm_aqn(x.to(DEV), w.to(DEV), z_dev, synthetic.EPS)
    assert_bf16_is_rounded_f32(hb, h, f"rows M={M} d={d}")
    ref = olin.rmsnorm_aqn(np32(x), np32(w), z_ref, synthetic.EPS)
    rel = np.abs(np32(h).astype(np.float64) - ref) / np.maximum(np.abs(ref), 1e-30)
    assert float(rel.max()) <= NORM_REL_TOL, float(rel.max())


def test_rmsnorm_rows_with_a_padded_stride(cuda_ok):
    """z rows further apart than d (a view into a wider buffer)."""
    M, d, ld = 6, 256, 264
    buf = torch.randn(M, ld, generator=torch.Generator().manual_seed(3)).mul_(1e-2).to(DEV)
    z = buf[:, :d]
    x = synthetic.activations(M, d, seed=2).to(DEV)
    w = synthetic.norm_scale(d, seed=2).to(DEV)
    h = pl.rmsnorm_aqn(x, w, z, synthetic.EPS, out_dtype=torch.float32)
    ref = olin.rmsnorm_aqn(np32(x), np32(w), np32(z), synthetic.EPS)
    rel = np.abs(np32(h).astype(np.float64) - ref) / np.maximum(np.abs(ref), 1e-30)
    assert float(rel.max()) <= NORM_REL_TOL


# Every kernel path of the linear: the shapes of the one-kernel decode path (3584^2; with
# one state per row they take the two-kernel path, whose prologue reads the rows), two-kernel
# decode (the 7B gate and down shapes), large M (CTA pairs), generic CUDA cores
# (d_i % 256 != 0).
@pytest.mark.parametrize("d_o,d_i,M,path", [
    (3584, 3584, 8, 2), (3584, 3584, 64, 2),
    (18944, 3584, 8, 1), (3584, 18944, 64, 1),
    (1000, 1024, 300, 3),
    (300, 272, 9, 0),
])
def test_linear_with_per_token_states(cuda_ok, d_o, d_i, M, path):
    r, seed = 32, d_o + M
    assert pl.linear_path(M, d_i, d_o, r) == path  # the path with one state per call
    sig = pl.aqn_sigma(2, 0.01, 0.0005)
    z_dev, z_ref = _states(99, 1, 7 * M, M, d_i, sig)
    case = make_case(d_o, d_i, M, r, 1e-2, seed, 0.0)
    packed, sb, s_g = oracle_quantize_cached((d_o, d_i, seed, 0.0), case["W"])
    dev_w = to_dev_nvfp4(packed, sb, s_g)
    args = (case["x"], *dev_w, case["A"], case["B"], 2.0, case["w_norm"], z_dev, synthetic.EPS)
    y = pl.nvfp4_lora_linear(*args, out_dtype=torch.float32)
    yb = pl.nvfp4_lora_linear(*args)
    assert_bf16_is_rounded_f32(yb, y, f"per-token states d_o={d_o} d_i={d_i} M={M}")
    ref_case = dict(case)
    ref_case["z"] = torch.from_numpy(z_ref)
    assert_linear_close(y, oracle_linear(ref_case, packed, sb, s_g, 2.0), f"per-token states path {path}")
    # the states differ per row: every row given row 0's state (the same kernel path) agrees
    # with y in row 0 only
    z_row0 = z_dev[0:1].expand(M, d_i).contiguous()
    y_shared = pl.nvfp4_lora_linear(*args[:8], z_row0, synthetic.EPS, out_dtype=torch.float32)
    assert torch.equal(y[0], y_shared[0]) and not torch.equal(y[1:], y_shared[1:])


@pytest.mark.parametrize("d_o,d_i,M", [(3584, 18944, 16), (18944, 3584, 8), (1000, 1024, 300), (300, 272, 9)])
def test_equal_rows_reproduce_the_shared_state_bitwise(cuda_ok, d_o, d_i, M):
    """Every row given the same state: the per-row form is bit for bit the shared form
    (both add w_norm + z in FP32 before any other use).  Shapes whose kernel path does not
    change with the noise layout; the one-kernel decode shapes run per-row states on the
    two-kernel path, checked against the oracle above."""
    assert pl.linear_path(M, d_i, d_o, 16) != 2
    case = make_case(d_o, d_i, M, 16, 1e-2, 5, 0.0)
    dev_w = pl.nvfp4_quantize(case["W"])
    z_rows = case["z"].unsqueeze(0).expand(M, d_i).contiguous()
    common = (case["x"], *dev_w, case["A"], case["B"], 2.0, case["w_norm"])
    y1 = pl.nvfp4_lora_linear(*common, case["z"], synthetic.EPS, out_dtype=torch.float32)
    y2 = pl.nvfp4_lora_linear(*common, z_rows, synthetic.EPS, out_dtype=torch.float32)
    assert torch.equal(y1, y2)


def test_prefill_m4096_per_token_states_sampled_rows(cuda_ok):
    """The 7B q projection at M = 4096 with a state per token, one full 128-token tile and
    a spread of other rows checked against the oracle."""
    wl = synthetic.WORKLOADS["prefill_7b"]
    p = wl.projs[0]
    M = wl.Ms[0]
    rows = np.unique(np.concatenate([np.arange(128, 256), np.random.default_rng(1).choice(M, 32, replace=False)]))
    z_dev, z_ref = _states(2025, 0, 0, M, p.d_i, wl.sigma, rows=rows)
    case = make_case(p.d_o, p.d_i, M, wl.r, wl.sigma, synthetic.proj_seed(wl, 0, 0))
    packed, sb, s_g = oracle_quantize_cached((p.d_o, p.d_i, "prefill-q"), case["W"])
    y = pl.nvfp4_lora_linear(case["x"], *to_dev_nvfp4(packed, sb, s_g), case["A"], case["B"], wl.lam,
                             case["w_norm"], z_dev, synthetic.EPS, out_dtype=torch.float32)
    x = np32(case["x"]).astype(np.float64)[rows]
    ref = olin.nvfp4_lora_linear(x, packed, sb, s_g, np32(case["A"]), np32(case["B"]), wl.lam,
                                 np32(case["w_norm"]), z_ref, synthetic.EPS)
    assert_linear_close(y[torch.from_numpy(rows).to(DEV)], ref, "prefill per-token states")
