"""Pins of the oracle's RMSNorm-AQN and LoRA forward (CPU only).

Against the pages: the LoRA parameter count (QeRL review, section 2.1), the
RMSNorm noise identity over 50 float64 cases (section 5.1, checked as in section
9.3); against closed forms of RMSNorm; against pure-Python brute force of the
whole path on the tiny workload.
"""

import math

import numpy as np

from oracle import linear, nvfp4
from precision_linear_gb300 import synthetic
from tests.conftest import read_golden


def test_lora_param_count_matches_pages():
    g = read_golden("lora_count.txt")
    d_i, d_o, r = int(g["d_i"]), int(g["d_o"]), int(g["r"])
    assert d_i * d_o == g["matrix_weights"]
    n = linear.lora_param_count(d_i, d_o, r)
    assert n == g["adapter_params"]
    assert 100.0 * n / (d_i * d_o) == g["percent_of_matrix"]


def test_aqn_identity_50_cases():
    """h_z W == h diag(1 + z/w) W (row-vector form, W in R^{d_i x d_o})."""
    g = read_golden("aqn_identity.txt")
    rng = np.random.default_rng(2024)
    worst = 0.0
    for case in range(int(g["cases"])):
        M, d, d_o = rng.integers(1, 9), rng.integers(4, 97), rng.integers(1, 65)
        x = rng.normal(size=(M, d))
        w = 1.0 + 0.1 * rng.normal(size=d)
        z = 1e-2 * rng.normal(size=d)
        W = rng.normal(size=(d, d_o))
        lhs = linear.rmsnorm_aqn(x, w, z, 1e-6) @ W
        rhs = linear.rmsnorm_aqn(x, w, None, 1e-6) @ (np.diag(1.0 + z / w) @ W)
        worst = max(worst, float(np.max(np.abs(lhs - rhs))))
    assert worst <= 1e-12
    # the same order of magnitude as the review's own float64 check
    assert worst < 100 * g["reported_max_abs_err"]


def test_rmsnorm_closed_forms():
    d, eps = 64, 1e-6
    w = np.ones(d)
    for c in (0.5, -3.0, 100.0):
        h = linear.rmsnorm_aqn(np.full((1, d), c), w, None, eps)
        assert np.allclose(h, c / math.sqrt(c * c + eps), rtol=0, atol=1e-15)
    a = 7.0
    x = np.zeros((1, d))
    x[0, 5] = a
    h = linear.rmsnorm_aqn(x, w, None, eps)
    assert math.isclose(h[0, 5], a / math.sqrt(a * a / d + eps), rel_tol=1e-15)
    assert np.count_nonzero(h) == 1
    # eps = 0: invariant to row scaling, and mean(u^2) == 1
    x = np.random.default_rng(0).normal(size=(3, d))
    h1 = linear.rmsnorm_aqn(x, w, None, 0.0)
    h2 = linear.rmsnorm_aqn(x * 37.5, w, None, 0.0)
    assert np.allclose(h1, h2, rtol=1e-14, atol=0)
    assert np.allclose(np.mean(h1 * h1, axis=1), 1.0, rtol=1e-14)
    # zero noise equals no noise; noise enters additively on the scale
    z = np.zeros(d)
    assert np.array_equal(linear.rmsnorm_aqn(x, w, z, eps), linear.rmsnorm_aqn(x, w, None, eps))


def _tiny_case():
    wl = synthetic.WORKLOADS["tiny"]
    p = wl.projs[0]
    c = synthetic.projection_case(p.d_o, p.d_i, wl.Ms[0], wl.r, wl.sigma, wl.seed)
    return wl, {k: v.float().numpy().astype(np.float64) if k != "W" else v.float().numpy() for k, v in c.items()}


def test_linear_bruteforce_tiny():
    """Whole path in pure-Python loops (own nibble decode, own norm, own matmul)."""
    wl, c = _tiny_case()
    packed, sb, s_g = nvfp4.quantize(c["W"])
    y = linear.nvfp4_lora_linear(c["x"], packed, sb, s_g, c["A"], c["B"], wl.lam,
                                 c["w_norm"], c["z"], synthetic.EPS)
    M, d_i = c["x"].shape
    d_o, r = c["B"].shape
    # weights
    Wq = [[0.0] * d_i for _ in range(d_o)]
    for o in range(d_o):
        for k in range(d_i):
            byte = int(packed[o, k >> 1])
            code = (byte >> 4) & 15 if k & 1 else byte & 15
            e, m = (code >> 1) & 3, code & 1
            q = (0.5 * m) if e == 0 else (2.0 ** (e - 1)) * (1.0 + 0.5 * m)
            if code & 8:
                q = -q
            Wq[o][k] = float(s_g) * nvfp4.e4m3_decode(int(sb[o, k >> 4])) * q
    for m_ in range(M):
        xs = c["x"][m_].tolist()
        ms = sum(v * v for v in xs) / d_i
        inv = 1.0 / math.sqrt(ms + synthetic.EPS)
        h = [xs[k] * inv * (c["w_norm"][k] + c["z"][k]) for k in range(d_i)]
        t = [sum(c["A"][j][k] * h[k] for k in range(d_i)) for j in range(r)]
        for o in range(d_o):
            acc = sum(Wq[o][k] * h[k] for k in range(d_i))
            acc += wl.lam * sum(c["B"][o][j] * t[j] for j in range(r))
            assert math.isclose(y[m_, o], acc, rel_tol=1e-11, abs_tol=1e-13), (m_, o)


def test_lora_branch_and_no_norm_path():
    wl, c = _tiny_case()
    packed, sb, s_g = nvfp4.quantize(c["W"])
    args = (c["x"], packed, sb, s_g, c["A"], c["B"])
    y2 = linear.nvfp4_lora_linear(*args, 2.0, c["w_norm"], c["z"])
    y0 = linear.nvfp4_lora_linear(*args, 0.0, c["w_norm"], c["z"])
    h = linear.rmsnorm_aqn(c["x"], c["w_norm"], c["z"], 1e-6)
    assert np.allclose(y2 - y0, 2.0 * (h @ c["A"].T) @ c["B"].T, rtol=1e-12, atol=1e-14)
    # no norm: the backbone acts on x itself
    yn = linear.nvfp4_lora_linear(c["x"], packed, sb, s_g, None, None, 0.0)
    assert np.allclose(yn, c["x"] @ nvfp4.dequantize(packed, sb, s_g).T, rtol=1e-12, atol=1e-14)


def test_rmsnorm_per_row_states_brute_force():
    """One noise state per token row (the per-response / per-token persistence scope of
    section 6): row m of the oracle equals a pure-Python evaluation of
    x_m / sqrt(mean(x_m^2) + eps) * (w + z_m), and a wrong row pairing is caught."""
    rng = np.random.default_rng(11)
    M, d, eps = 4, 7, 1e-6
    x = rng.normal(size=(M, d))
    w = 1.0 + 0.1 * rng.normal(size=d)
    z = 1e-2 * rng.normal(size=(M, d))
    got = linear.rmsnorm_aqn(x, w, z, eps)
    for m in range(M):
        ms = sum(float(v) * float(v) for v in x[m]) / d
        inv = 1.0 / math.sqrt(ms + eps)
        for j in range(d):
            assert math.isclose(got[m, j], float(x[m, j]) * inv * (float(w[j]) + float(z[m, j])), rel_tol=1e-14)
    swapped = linear.rmsnorm_aqn(x, w, z[::-1], eps)
    assert np.max(np.abs(swapped - got)) > 1e-4
