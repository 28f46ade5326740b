"""Grouped projections: pl_nvfp4_lora_linear_group against the FP64 oracle.

The projections behind one RMSNorm read the same x, w_norm and noise state ("QeRL: When
Quantized Weights Help Reinforcement Learning, and Where the Evidence Stops", section
5.1: Q, K and V share one noise vector, Gate and Up the other).  A group call computes
h once and runs every projection's weight tiles in one main kernel; each projection must
still match the oracle within max |y - y_ref| <= 1e-2 rms(y_ref)."""

import numpy as np
import pytest
import torch

from oracle import aqn
from precision_linear_gb300 import binding as pl
from precision_linear_gb300 import synthetic
from tests.gpu_cases import (DEV, assert_bf16_is_rounded_f32, assert_linear_close, oracle_linear,
                             oracle_quantize_cached, to_dev_nvfp4)

pytestmark = pytest.mark.gpu


def _layer(wl, M):
    cases = synthetic.layer_case(wl, 0, M)
    moved = {}

    def mv(t):
        if t is None:
            return None
        if id(t) not in moved:
            moved[id(t)] = t.to(DEV)
        return moved[id(t)]

    return {n: {k: mv(v) for k, v in c.items()} for n, c in cases.items()}


def _group_check(wl, names, M, z_rows=None, ranks=None, norm=True):
    cases = _layer(wl, M)
    c0 = cases[names[0]]
    projs, encs = [], []
    for i, n in enumerate(names):
        c = cases[n]
        packed, sb, s_g = oracle_quantize_cached((wl.name, n), c["W"])
        codes, scales, sg = to_dev_nvfp4(packed, sb, s_g)
        q = dict(codes=codes, scales=scales, s_g=sg, lam=wl.lam)
        r = wl.r if ranks is None else ranks[i]
        if r > 0:
            q.update(A=c["A"][:r].contiguous(), B=c["B"][:, :r].contiguous())
        projs.append(q)
        encs.append((packed, sb, s_g, q))
    z = (z_rows if z_rows is not None else c0["z"]) if norm else None
    w = c0["w_norm"] if norm else None
    ys = pl.nvfp4_lora_linear_group(c0["x"], projs, w, z, synthetic.EPS, out_dtype=torch.float32)
    yb = pl.nvfp4_lora_linear_group(c0["x"], projs, w, z, synthetic.EPS)
    for n, y, y16, (packed, sb, s_g, q) in zip(names, ys, yb, encs):
        assert_bf16_is_rounded_f32(y16, y, f"group {names} {n} M={M}")
        ref_case = dict(x=c0["x"], w_norm=c0["w_norm"], z=z if z is not None else c0["z"],
                        A=q.get("A", c0["A"]), B=q.get("B", c0["B"]))
        ref = oracle_linear(ref_case, packed, sb, s_g, wl.lam, norm=norm, noise=norm, lora="A" in q)
        assert_linear_close(y, ref, f"group {names} {n} M={M}")
    return ys


@pytest.mark.parametrize("M", [1, 8, 64])
def test_qkv_group(cuda_ok, M):
    _group_check(synthetic.WORKLOADS["layer_7b"], ["q", "k", "v"], M)


@pytest.mark.parametrize("M", [8, 64])
def test_gate_up_group(cuda_ok, M):
    _group_check(synthetic.WORKLOADS["layer_7b"], ["gate", "up"], M)


def test_32b_qkv_group(cuda_ok):
    _group_check(synthetic.WORKLOADS["stack_32b"], ["q", "k", "v"], 16)


def test_group_mixed_ranks_and_no_norm(cuda_ok):
    wl = synthetic.WORKLOADS["layer_7b"]
    _group_check(wl, ["q", "k", "v"], 9, ranks=[0, 5, 32])
    _group_check(wl, ["k", "v"], 3, norm=False)


def test_group_per_token_states(cuda_ok):
    wl = synthetic.WORKLOADS["layer_7b"]
    M, d = 16, 3584
    sig = float(np.float32(wl.sigma))
    z_dev = pl.aqn_noise(d, 4242, 0, 300, M, sig, device=DEV)
    z_ref = torch.from_numpy(aqn.noise(4242, 0, 300, M, d, sig).astype(np.float32)).to(DEV)
    # the oracle side takes its own draw of the states
    cases = _layer(wl, M)
    ys = _group_check(wl, ["gate", "up"], M, z_rows=z_ref)
    projs = []
    for n in ("gate", "up"):
        packed, sb, s_g = oracle_quantize_cached((wl.name, n), cases[n]["W"])
        codes, scales, sg = to_dev_nvfp4(packed, sb, s_g)
        projs.append(dict(codes=codes, scales=scales, s_g=sg, A=cases[n]["A"], B=cases[n]["B"], lam=wl.lam))
    ys_dev = pl.nvfp4_lora_linear_group(cases["gate"]["x"], projs, cases["gate"]["w_norm"], z_dev, synthetic.EPS,
                                        out_dtype=torch.float32)
    for a, b in zip(ys, ys_dev):
        rms = float(torch.sqrt(torch.mean(a.double() ** 2)))
        assert float(torch.max(torch.abs(a - b))) <= 1e-3 * rms


def test_large_group_runs_projection_by_projection(cuda_ok):
    """Five projections (more than one launch takes, at decode and at large M): one call per
    projection."""
    wl = synthetic.WORKLOADS["layer_7b"]
    _group_check(wl, ["q", "k", "v", "k", "v"], 4)
    _group_check(wl, ["k", "v", "k", "v", "k"], 100)


@pytest.mark.parametrize("names,M", [(["q", "k", "v"], 300), (["gate", "up"], 130), (["k", "v"], 100)])
def test_large_m_group(cuda_ok, names, M):
    """M > 64: one row pass, one adapter down-projection per member and one contraction over
    every member's weight tiles (ragged token tiles at M = 300 and 130)."""
    assert pl.linear_path(M, 3584, 512, 32) == 3
    _group_check(synthetic.WORKLOADS["layer_7b"], names, M)


def test_large_m_group_mixed_ranks_no_norm_and_row_states(cuda_ok):
    wl = synthetic.WORKLOADS["layer_7b"]
    _group_check(wl, ["q", "k", "v"], 100, ranks=[0, 8, 32])
    _group_check(wl, ["k", "v"], 77, norm=False)
    M = 96
    z_rows = (torch.randn(M, 3584, generator=torch.Generator().manual_seed(77)) * wl.sigma).to(DEV)
    _group_check(wl, ["k", "v"], M, z_rows=z_rows)


def test_prefill_qkv_group_m4096_sampled_rows(cuda_ok):
    """The 7B q/k/v group at M = 4096: one full 128-token tile and a spread of other rows of
    every member against the oracle."""
    from oracle import linear as olin
    from tests.gpu_cases import np32
    wl = synthetic.WORKLOADS["prefill_7b"]
    M = wl.Ms[0]
    cases = _layer(wl, M)
    names = ["q", "k", "v"]
    c0 = cases["q"]
    rows = np.unique(np.concatenate([np.arange(256, 384), np.random.default_rng(3).choice(M, 24, replace=False)]))
    projs, encs = [], []
    for n in names:
        packed, sb, s_g = oracle_quantize_cached((wl.name, n, "m4096"), cases[n]["W"])
        codes, scales, sg = to_dev_nvfp4(packed, sb, s_g)
        projs.append(dict(codes=codes, scales=scales, s_g=sg, A=cases[n]["A"], B=cases[n]["B"], lam=wl.lam))
        encs.append((packed, sb, s_g))
    ys = pl.nvfp4_lora_linear_group(c0["x"], projs, c0["w_norm"], c0["z"], synthetic.EPS, out_dtype=torch.float32)
    x = np32(c0["x"]).astype(np.float64)[rows]
    sel = torch.from_numpy(rows).to(DEV)
    for n, y, (packed, sb, s_g) in zip(names, ys, encs):
        ref = olin.nvfp4_lora_linear(x, packed, sb, s_g, np32(cases[n]["A"]), np32(cases[n]["B"]), wl.lam,
                                     np32(c0["w_norm"]), np32(c0["z"]), synthetic.EPS)
        assert_linear_close(y[sel], ref, f"prefill group {n}")


def test_group_repeatable_bitwise(cuda_ok):
    wl = synthetic.WORKLOADS["layer_7b"]
    a = _group_check(wl, ["gate", "up"], 32)
    b = _group_check(wl, ["gate", "up"], 32)
    assert all(torch.equal(u, v) for u, v in zip(a, b))
