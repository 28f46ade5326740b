"""Pins of the AQN noise oracle (oracle/aqn.py) to things other than itself.

* Philox4x32-10: the generator's published known-answer vectors (tests/golden).
* Schedule ("QeRL: When Quantized Weights Help ...", section 5.2): sigma_0 = 0, stage 1
  exactly the start value, stage 9 exactly the end value, a constant ratio between
  neighbouring noisy stages (equal steps in log sigma), for both of the pages' ranges.
* Stage rule: ten equal parts of the planned horizon, warm-up first.
* Uniforms exact in FP32 and strictly inside (0, 1); normals with the moments,
  distribution and independence of N(0, sigma^2); the counter layout (norm, scope,
  seed) gives separate, reproducible streams.
"""

import math
import os

import numpy as np
import pytest

from oracle import aqn
from tests.conftest import ROOT

GOLDEN = os.path.join(ROOT, "tests", "golden", "philox4x32_10_kat.txt")


def _kat():
    rows = []
    for line in open(GOLDEN, encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(t, 16) for t in line.split()]
        rows.append((tuple(w[0:4]), tuple(w[4:6]), tuple(w[6:10])))
    return rows


def test_philox_known_answers():
    rows = _kat()
    assert len(rows) == 3
    for ctr, key, want in rows:
        assert aqn.philox4x32_10(ctr, key) == want


def test_counter_and_key_layout_through_a_known_answer():
    """The third known-answer vector has six distinct words: read as seed = key (low word
    first) and counter = (block, norm, scope low, scope high), the state's block must be
    the Box-Muller transform of the vector's published output words, computed here by
    hand from the definition (u = (2 (x >> 9) + 1) 2^-24)."""
    ctr, key, out = _kat()[2]
    seed = key[0] | (key[1] << 32)
    scope = ctr[2] | (ctr[3] << 32)
    got = aqn.noise_block(seed, ctr[1], scope, ctr[0])
    u = [(2 * (w >> 9) + 1) * 2.0 ** -24 for w in out]
    ra, rb = math.sqrt(-2 * math.log(u[0])), math.sqrt(-2 * math.log(u[2]))
    want = (ra * math.cos(2 * math.pi * u[1]), ra * math.sin(2 * math.pi * u[1]),
            rb * math.cos(2 * math.pi * u[3]), rb * math.sin(2 * math.pi * u[3]))
    assert all(math.isclose(g, w, rel_tol=1e-14, abs_tol=1e-15) for g, w in zip(got, want))
    # and the array draw agrees with the one-block form at small block indices
    z = aqn.noise(seed, ctr[1], scope, 1, 64, 1.0)[0]
    for b in (0, 5, 15):
        assert np.allclose(z[4 * b:4 * b + 4], aqn.noise_block(seed, ctr[1], scope, b), rtol=0, atol=1e-15)


def test_philox_array_form_matches_scalar_form():
    rng = np.random.default_rng(7)
    c = rng.integers(0, 2 ** 32, size=(4, 64), dtype=np.uint64)
    k0, k1 = 0x12345678, 0x9ABCDEF0
    got = aqn.philox4x32_10_array(c[0], c[1], c[2], c[3], k0, k1)
    for i in range(64):
        want = aqn.philox4x32_10((int(c[0, i]), int(c[1, i]), int(c[2, i]), int(c[3, i])), (k0, k1))
        assert tuple(int(g[i]) for g in got) == want


@pytest.mark.parametrize("start,end", [(0.01, 0.0005), (0.05, 0.0005)])
def test_schedule_endpoints_and_log_spacing(start, end):
    s = [aqn.sigma(k, start, end) for k in range(aqn.STAGES)]
    assert s[0] == 0.0
    assert s[1] == start
    assert math.isclose(s[9], end, rel_tol=1e-15)
    ratio = (end / start) ** (1 / 8)
    for k in range(1, 9):
        assert math.isclose(s[k + 1] / s[k], ratio, rel_tol=1e-14)
    assert all(s[k] > s[k + 1] for k in range(1, 9))  # decreasing noise after the warm-up
    with pytest.raises(ValueError):
        aqn.sigma(10, start, end)


def test_schedule_values_for_table4_range():
    # 0.01 -> 0.0005 over nine levels: ratio 0.05 ** (1/8) = 0.68766...
    s = [aqn.sigma(k, 0.01, 0.0005) for k in range(10)]
    assert math.isclose(s[5], 0.01 * 0.05 ** 0.5, rel_tol=1e-15)  # the geometric midpoint
    assert math.isclose(s[2], 0.01 * 0.05 ** 0.125, rel_tol=1e-15)


def test_schedule_matches_the_printed_endpoints():
    rows = [l.split() for l in open(os.path.join(ROOT, "tests", "golden", "aqn_schedule.txt"), encoding="utf-8")
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for start, end, k, want in rows:
        assert math.isclose(aqn.sigma(int(k), float(start), float(end)), float(want), rel_tol=1e-15, abs_tol=0)


def test_stage_rule():
    assert aqn.stage(0, 1000) == 0
    assert aqn.stage(99, 1000) == 0
    assert aqn.stage(100, 1000) == 1
    assert aqn.stage(899, 1000) == 8
    assert aqn.stage(900, 1000) == 9
    assert aqn.stage(1000, 1000) == 9
    assert aqn.stage(5000, 1000) == 9  # past the horizon: the last stage
    st = [aqn.stage(d, 37) for d in range(0, 38)]
    assert st == sorted(st) and st[0] == 0 and st[-1] == 9 and set(st) == set(range(10))
    with pytest.raises(ValueError):
        aqn.stage(1, 0)


def test_uniforms_exact_in_fp32_and_inside_open_interval():
    x = np.array([0, 1, 511, 512, 2 ** 31, 2 ** 32 - 1], dtype=np.uint64)
    u = aqn.uniform(x)
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    assert u[0] == 2.0 ** -24 and u[-1] == 1.0 - 2.0 ** -24
    assert u[1] == u[0] and u[3] == 3 * 2.0 ** -24  # the low 9 bits are dropped
    assert np.all((u > 0) & (u < 1))


def _ks_sqrt_n_d(x: np.ndarray) -> float:
    """sqrt(n) times the Kolmogorov-Smirnov distance between the sample and N(0, 1)."""
    xs = np.sort(np.asarray(x, dtype=np.float64))
    n = xs.size
    cdf = 0.5 * (1.0 + np.array([math.erf(v / math.sqrt(2.0)) for v in xs]))
    i = np.arange(1, n + 1)
    d = max(float(np.max(i / n - cdf)), float(np.max(cdf - (i - 1) / n)))
    return math.sqrt(n) * d


# Kolmogorov's limit: P(sqrt(n) D > lam) ~ 2 exp(-2 lam^2) for large lam; 1e-4 at lam = 2.226
KS_CRIT_1E4 = math.sqrt(math.log(2.0 / 1e-4) / 2.0)


def test_ks_statistic_separates_normal_from_shifted():
    rng = np.random.default_rng(3)
    assert _ks_sqrt_n_d(rng.standard_normal(1 << 14)) < KS_CRIT_1E4
    assert _ks_sqrt_n_d(rng.standard_normal(1 << 14) + 0.1) > KS_CRIT_1E4
    assert _ks_sqrt_n_d(rng.standard_normal(1 << 14) * 1.1) > KS_CRIT_1E4


def test_noise_moments_and_distribution():
    sig = 0.01
    z = aqn.noise(seed=2024, norm_id=3, scope0=0, n_scopes=1, d=1 << 16, sig=sig)[0]
    n = z.size
    assert abs(z.mean()) < 5 * sig / math.sqrt(n)
    assert abs(z.var() / sig ** 2 - 1) < 5 * math.sqrt(2 / n)
    assert _ks_sqrt_n_d(z / sig) < KS_CRIT_1E4
    # fourth moment of a normal is 3 sigma^4
    assert abs(np.mean((z / sig) ** 4) - 3) < 0.1
    # each of the four channels of a block is itself N(0, 1): no lane is mis-assigned
    for q in range(4):
        assert _ks_sqrt_n_d(z[q::4] / sig) < KS_CRIT_1E4


def test_noise_channels_are_uncorrelated():
    z = aqn.noise(seed=11, norm_id=0, scope0=0, n_scopes=1, d=1 << 16, sig=1.0)[0]
    n4 = z.size // 4
    blk = z.reshape(n4, 4)
    lim = 5 / math.sqrt(n4)
    for a in range(4):
        for b in range(a + 1, 4):
            assert abs(np.corrcoef(blk[:, a], blk[:, b])[0, 1]) < lim
    # neighbouring blocks (the counter's block word) are independent too
    assert abs(np.corrcoef(blk[:-1, 0], blk[1:, 0])[0, 1]) < lim


def test_streams_per_norm_scope_and_seed():
    d = 4096
    base = aqn.noise(5, 0, 0, 4, d, 1.0)
    assert np.array_equal(base, aqn.noise(5, 0, 0, 4, d, 1.0))  # reproducible from the seed
    # a scope row does not depend on how many rows are drawn with it
    assert np.array_equal(aqn.noise(5, 0, 2, 1, d, 1.0)[0], base[2])
    # the scope's high word and the norm index select other streams
    others = [aqn.noise(5, 1, 0, 1, d, 1.0)[0], aqn.noise(6, 0, 0, 1, d, 1.0)[0],
              aqn.noise(5, 0, 1 << 32, 1, d, 1.0)[0], base[1]]
    lim = 5 / math.sqrt(d)
    for o in others:
        assert abs(np.corrcoef(base[0], o)[0, 1]) < lim
    # sigma only scales
    assert np.allclose(aqn.noise(5, 0, 0, 1, d, 0.25)[0], 0.25 * base[0], rtol=0, atol=1e-15)
    # a ragged channel count takes the first d of the block-padded draw
    assert np.array_equal(aqn.noise(5, 0, 0, 1, 4095, 1.0)[0], base[0, :4095])
