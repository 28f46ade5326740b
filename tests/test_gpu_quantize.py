"""GPU quantiser vs the oracle: codes, E4M3 scales and s_g bit for bit."""

import numpy as np
import pytest
import torch

from precision_linear_gb300 import binding as pl
from precision_linear_gb300 import synthetic
from tests.gpu_cases import DEV, np32, oracle_quantize

pytestmark = pytest.mark.gpu


def _check(W):
    codes, scales, s_g = pl.nvfp4_quantize(W)
    torch.cuda.synchronize()
    packed, sb, sg_ref = oracle_quantize(W)
    got_sg = np.float32(s_g.item())
    assert got_sg.view(np.uint32) == np.float32(sg_ref).view(np.uint32), (got_sg, sg_ref)
    sc = scales.cpu().numpy()
    bad_s = np.argwhere(sc != sb)
    assert bad_s.size == 0, f"{len(bad_s)} scale mismatches, first {bad_s[:3].tolist()}"
    cd = codes.cpu().numpy()
    bad_c = np.argwhere(cd != packed)
    assert bad_c.size == 0, f"{len(bad_c)} code-byte mismatches, first {bad_c[:3].tolist()}"
    return codes, scales, s_g


@pytest.mark.parametrize("d_o,d_i,outliers", [(256, 256, 0.0), (3584, 3584, 1e-3), (512, 3584, 0.0),
                                              (1, 16, 0.0), (3, 48, 0.0), (129, 272, 1e-2)])
def test_quantize_bit_exact(cuda_ok, d_o, d_i, outliers):
    W = synthetic.weight(d_o, d_i, seed=d_o + d_i, outlier_frac=outliers).to(DEV)
    _check(W)


def test_quantize_7b_layer_bit_exact(cuda_ok):
    for i, p in enumerate(synthetic.QWEN7B_LAYER):
        W = synthetic.weight(p.d_o, p.d_i, seed=synthetic.proj_seed(synthetic.WORKLOADS["layer_7b"], 0, i)).to(DEV)
        _check(W)


def test_quantize_32b_sampled_projections_bit_exact(cuda_ok):
    wl = synthetic.WORKLOADS["stack_32b"]
    for layer, i in [(0, 0), (31, 3), (63, 6)]:
        p = wl.projs[i]
        W = synthetic.weight(p.d_o, p.d_i, seed=synthetic.proj_seed(wl, layer, i), device=DEV)
        _check(W)


def test_quantize_edge_values(cuda_ok):
    g = torch.Generator().manual_seed(11)
    W = (torch.randn(64, 512, generator=g) * 0.02)
    W[0] = 0.0                                  # all-zero row
    W[1, 32:48] = 0.0                           # all-zero block
    W[2, :16] = 1e-30                           # block far below the tensor max: scale underflows
    W[3, :16] = torch.tensor([6, .25, .75, 1.25, 1.75, 2.5, 3.5, 5, -.25, -.75, -1.25, -1.75,
                              -2.5, -3.5, -5, 0]) * 0.0078125   # exact threshold ties
    W[4, :] = -W[4, :]
    W[5, 7] = 3.0                               # tensor max (outlier)
    W[6, :16] = -1e-9                           # negative values that round to zero
    _check(W.to(torch.bfloat16).to(DEV))
    # huge and tiny tensors
    _check((torch.randn(32, 256, generator=g) * 1e30).to(torch.bfloat16).to(DEV))
    _check((torch.randn(32, 256, generator=g) * 1e-30).to(torch.bfloat16).to(DEV))
    # all zero
    c, s, sg = _check(torch.zeros(16, 64, dtype=torch.bfloat16, device=DEV))
    assert sg.item() == 1.0


def test_quantize_repeatable(cuda_ok):
    W = synthetic.weight(3584, 3584, seed=2, outlier_frac=1e-3).to(DEV)
    a = [pl.nvfp4_quantize(W) for _ in range(3)]
    for c, s, g in a[1:]:
        assert torch.equal(c, a[0][0]) and torch.equal(s, a[0][1]) and torch.equal(g, a[0][2])
