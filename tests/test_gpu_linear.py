"""GPU NVFP4 + LoRA linear vs the FP64 oracle (max |y - y_ref| <= 1e-2 rms(y_ref)).

The GPU linear is fed the oracle's own NVFP4 encoding of each weight, so these
tests do not depend on the GPU quantiser; one end-to-end test chains the GPU
quantiser into the GPU linear."""

import numpy as np
import pytest
import torch

from precision_linear_gb300 import binding as pl
from precision_linear_gb300 import synthetic
from tests.gpu_cases import (DEV, assert_bf16_is_rounded_f32, assert_linear_close, make_case, np32,
                             oracle_linear, oracle_quantize, oracle_quantize_cached, to_dev_nvfp4)

pytestmark = pytest.mark.gpu


def _run(case, dev_w, lam, norm=True, noise=True, lora=True, out_dtype=torch.float32):
    return pl.nvfp4_lora_linear(case["x"], *dev_w, case["A"] if lora else None, case["B"] if lora else None,
                                lam, case["w_norm"] if norm else None, case["z"] if (norm and noise) else None,
                                synthetic.EPS, out_dtype=out_dtype)


def _check(d_o, d_i, M, r, lam=2.0, seed=0, outliers=0.0, sigma=1e-2, **kw):
    """FP32 output within the tolerance of the oracle; BF16 output == RN(FP32 output)."""
    case = make_case(d_o, d_i, M, r, sigma, seed, outliers)
    packed, sb, s_g = oracle_quantize_cached((d_o, d_i, seed, outliers), case["W"])
    dev_w = to_dev_nvfp4(packed, sb, s_g)
    y = _run(case, dev_w, lam, **kw)
    yb = _run(case, dev_w, lam, out_dtype=torch.bfloat16, **kw)
    what = f"d_o={d_o} d_i={d_i} M={M} r={r} {kw}"
    assert_bf16_is_rounded_f32(yb, y, what)
    ref = oracle_linear(case, packed, sb, s_g, lam, **kw)
    return assert_linear_close(y, ref, what)


def test_tiny(cuda_ok):
    wl = synthetic.WORKLOADS["tiny"]
    _check(256, 256, 4, wl.r, wl.lam, seed=wl.seed)


@pytest.mark.parametrize("M", [1, 8, 16, 32, 64])
def test_decode_projection_sweep(cuda_ok, M):
    wl = synthetic.WORKLOADS["decode_proj_7b"]
    _check(3584, 3584, M, wl.r, wl.lam, seed=wl.seed, outliers=wl.outlier_frac)


@pytest.mark.parametrize("kw", [dict(lora=False), dict(norm=False), dict(noise=False), dict(lam=0.0)])
def test_path_variants(cuda_ok, kw):
    lam = kw.pop("lam", 2.0)
    _check(3584, 3584, 16, 32, lam, seed=5, **kw)


@pytest.mark.parametrize("r", [1, 8, 64])
def test_ranks(cuda_ok, r):
    _check(1024, 512, 9, r, seed=r)


@pytest.mark.parametrize("d_o,d_i,M", [(1, 256, 1), (100, 256, 3), (129, 512, 17), (300, 768, 63),
                                       (257, 512, 64), (130, 512, 65), (77, 272, 5), (40, 48, 2),
                                       (384, 256, 200)])
def test_ragged_shapes(cuda_ok, d_o, d_i, M):
    _check(d_o, d_i, M, 8, seed=d_o * 7 + M)


# Large-M shapes of the CTA-pair contraction: an odd rank (B rows read element-wise), d_o
# not a multiple of the 256-row pair tile, M not a multiple of the token tile, several tiles
# per pair (persistent rounds), and the narrow-tile choice when tiles are fewer than pairs.
@pytest.mark.parametrize("d_o,d_i,M,r", [(1000, 1024, 700, 5), (4000, 2048, 1500, 32), (2304, 512, 4096, 16),
                                         (520, 768, 3000, 1)])
def test_large_m_shapes(cuda_ok, d_o, d_i, M, r):
    assert pl.linear_path(M, d_i, d_o, r) == 3
    _check(d_o, d_i, M, r, seed=d_o + M + r)


# Decode shapes of the two-kernel tcgen05 path (too many tiles, or too long a K slice, for
# the fused kernel): one chunk per CTA (fewer than the A ring's slots), no adapter, an odd
# rank, K split over a cluster with ragged slices, N = 64 with r = 64.
@pytest.mark.parametrize("d_o,d_i,M,r", [(20000, 256, 1, 0), (20000, 512, 7, 5), (2000, 8192, 3, 5),
                                         (3000, 9216, 64, 64), (130, 18944, 33, 32)])
def test_tc_path_shapes(cuda_ok, d_o, d_i, M, r):
    assert pl.linear_path(M, d_i, d_o, r) == 1
    _check(d_o, d_i, M, r, seed=d_o + M + r, lora=r > 0)


def _layer_on_device(cases):
    """synthetic.layer_case on the device, the shared norm inputs moved once (still shared)."""
    moved = {}

    def mv(t):
        if t is None:
            return None
        if id(t) not in moved:
            moved[id(t)] = t.to(DEV)
        return moved[id(t)]

    return {n: {k: mv(v) for k, v in c.items()} for n, c in cases.items()}


def _check_layer(wl, layer, M, rows=None, key=""):
    """Every projection of one decoder layer, wired as in the layer (q/k/v read the attention
    norm's x, w_norm and z; gate/up the FFN norm's), against the oracle; rows: the token rows
    compared (all when None)."""
    cases = _layer_on_device(synthetic.layer_case(wl, layer, M))
    assert cases["q"]["x"] is cases["k"]["x"] is cases["v"]["x"]
    assert cases["gate"]["z"] is cases["up"]["z"] and cases["gate"]["x"] is not cases["q"]["x"]
    for p in wl.projs:
        c = cases[p.name]
        norm = p.norm is not None
        packed, sb, s_g = oracle_quantize_cached((wl.name, layer, p.name), c["W"])
        y = _run(c, to_dev_nvfp4(packed, sb, s_g), wl.lam, norm=norm)
        ref = oracle_linear(c, packed, sb, s_g, wl.lam, norm=norm, rows=rows)
        if rows is not None:
            y = y[torch.from_numpy(rows).to(DEV)]
        assert_linear_close(y, ref, f"{wl.name} layer {layer} {p.name} M={M} {key}")


@pytest.mark.parametrize("M", [8, 32, 64])
def test_7b_layer_set(cuda_ok, M):
    _check_layer(synthetic.WORKLOADS["layer_7b"], 0, M)


def test_7b_layer_prefill_m4096_sampled_rows(cuda_ok):
    """M = 4096: two full 128-token tiles (the first and one in the middle) and a spread of
    other rows of every projection."""
    wl = synthetic.WORKLOADS["prefill_7b"]
    M = wl.Ms[0]
    rows = np.unique(np.concatenate([np.arange(0, 128), np.arange(2048, 2176),
                                     np.random.default_rng(0).choice(M, 48, replace=False)]))
    _check_layer(wl, 0, M, rows=rows)


@pytest.mark.parametrize("layer", [0, 31, 63])
def test_32b_stack_sampled_layer(cuda_ok, layer):
    wl = synthetic.WORKLOADS["stack_32b"]
    for M in wl.Ms:
        _check_layer(wl, layer, M)


def test_end_to_end_gpu_quantiser_into_linear(cuda_ok):
    case = make_case(3584, 3584, 32, 32, 1e-2, 2, 1e-3)
    dev_w = pl.nvfp4_quantize(case["W"])
    y = _run(case, dev_w, 2.0)
    packed, sb, s_g = oracle_quantize(case["W"])
    assert_linear_close(y, oracle_linear(case, packed, sb, s_g, 2.0), "gpu quantiser -> gpu linear")


def test_repeatable_bitwise(cuda_ok):
    for M in (1, 64, 300):
        case = make_case(1024, 3584, M, 32, seed=M)
        dev_w = pl.nvfp4_quantize(case["W"])
        ys = [_run(case, dev_w, 2.0) for _ in range(3)]
        assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])
