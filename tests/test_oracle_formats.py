"""Pins of the oracle's number formats (CPU only).

E2M1 against the grid the QeRL review prints (section 3.1); E4M3 against the OCP
FP8 definition's closed forms and PyTorch's float8_e4m3fn (a library routine);
the round-to-nearest-even code selection against brute force.
"""

import math
import struct

import numpy as np
import pytest
import torch

from oracle import nvfp4
from tests.conftest import read_golden


def test_e2m1_grid_matches_pages():
    grid = read_golden("e2m1_grid.txt")["_values"]
    assert len(grid) == 8
    assert [nvfp4.e2m1_decode(c) for c in range(8)] == grid
    # codes 8..15 are the negatives, code 8 is a signed zero
    for c in range(8):
        assert nvfp4.e2m1_decode(c | 8) == -grid[c]
    assert math.copysign(1.0, nvfp4.e2m1_decode(8)) == -1.0
    # non-uniform spacing, as the page stresses
    gaps = np.diff(grid)
    assert sorted(set(gaps.tolist())) == [0.5, 1.0, 2.0]


def test_e4m3_decode_matches_torch_all_256():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mine = nvfp4.E4M3_TABLE
    nan_ref = np.isnan(ref)
    assert np.array_equal(nan_ref, np.isnan(mine))
    assert np.array_equal(ref[~nan_ref], mine[~nan_ref])


def test_e4m3_closed_forms():
    d = nvfp4.e4m3_decode
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))
    assert d(0x01) == 2.0 ** -9  # smallest subnormal
    assert d(0x07) == 7 / 8 * 2.0 ** -6  # largest subnormal
    assert d(0x08) == 2.0 ** -6  # smallest normal
    assert d(0x38) == 1.0  # exponent field = bias
    assert np.all(np.diff(nvfp4.E4M3_POS) > 0)


def _f32_neighbours(x):
    b = struct.unpack("<I", struct.pack("<f", x))[0]
    return [struct.unpack("<f", struct.pack("<I", b + k))[0] for k in (-1, 0, 1)]


def _e4m3_sweep():
    grid = nvfp4.E4M3_POS
    vals = list(grid)
    mids = (grid[:-1] + grid[1:]) / 2
    for m in mids:
        vals += _f32_neighbours(float(m))
    rng = np.random.default_rng(7)
    vals += list(np.exp2(rng.uniform(-12, math.log2(448), 20000)))
    vals += [0.0, 2.0 ** -11, 2.0 ** -10, 2.0 ** -10 * 1.0000001, 2.0 ** -9]
    return np.array(vals, dtype=np.float32)


def test_e4m3_encode_matches_torch_in_range():
    t = _e4m3_sweep()
    t = t[t <= 448.0]
    ref = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = nvfp4.e4m3_encode(t)
    bad = np.nonzero(ref != mine)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first t={t[bad[:5]]}"


def test_e4m3_encode_ties_and_saturation():
    enc = nvfp4.e4m3_encode
    # 2^-10 is the midpoint between 0 and the smallest subnormal: tie -> even (0)
    assert enc(2.0 ** -10) == 0
    # midpoint of 1.0 (0x38) and 1.125 (0x39) goes to the even code 0x38
    assert enc(1.0625) == 0x38
    # midpoint of 1.125 (0x39) and 1.25 (0x3A) goes to 0x3A
    assert enc(1.1875) == 0x3A
    for t in (448.0, 449.0, 464.0, 480.0, 1e6, 3.0e38):
        assert enc(t) == 0x7E


def _brute_nearest_even(v, grid):
    best = None
    for i, g in enumerate(grid):
        d = abs(v - g)
        if best is None or d < best[0] or (d == best[0] and i % 2 == 0):
            best = (d, i)
    return best[1]


def test_e2m1_nearest_even_thresholds():
    # exact midpoints between adjacent grid values go to the even code
    expect = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for v, c in expect.items():
        assert nvfp4.e2m1_magnitude_code(np.float32(v)) == c
    for v in (5.0000005, 6.0, 7.0, 1e30, float("inf")):
        assert nvfp4.e2m1_magnitude_code(np.float32(v)) == 7


def test_e2m1_nearest_even_bruteforce():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.uniform(0, 7, 3000), rng.choice([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], 200)])
    v = v.astype(np.float32)
    got = nvfp4.e2m1_magnitude_code(v)
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for vi, gi in zip(v.tolist(), got.tolist()):
        assert gi == _brute_nearest_even(vi, grid)
