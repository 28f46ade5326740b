"""Pins of the W8A8 oracle (oracle/w8a8.py): brute-force integer dot products, the
rounding bounds of both formats, exact reconstruction of inputs that sit on the grid,
the FP8 encoder against torch's float8_e4m3fn cast (a library routine), zero rows."""

import numpy as np
import pytest
import torch

from oracle import w8a8


def test_int8_linear_equals_brute_force_loops():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((2, 5))
    W = rng.standard_normal((3, 5)) * 0.02
    qw, sw = w8a8.quantize_int8_rows(W)
    y = w8a8.w8a8_linear(x, qw, sw, "int8")
    qx, sx = w8a8.quantize_int8_rows(x.astype(np.float32))
    for m in range(2):
        for o in range(3):
            acc = 0
            for k in range(5):
                acc += int(qx[m, k]) * int(qw[o, k])
            assert np.isclose(y[m, o], float(sx[m]) * float(sw[o]) * acc, rtol=1e-15, atol=0)


def test_int8_rounding_bound_and_range():
    rng = np.random.default_rng(1)
    X = (rng.standard_normal((64, 300)) * rng.uniform(0.01, 10, size=(64, 1))).astype(np.float32)
    q, s = w8a8.quantize_int8_rows(X)
    err = np.abs(X.astype(np.float64) - w8a8.dequant_rows(q, s, "int8"))
    assert np.all(err <= s[:, None] * (0.5 + 1e-6))
    assert np.all(np.max(np.abs(q.astype(np.int32)), axis=1) == 127)  # the row maximum maps onto 127
    assert q.dtype == np.int8 and int(q.min()) >= -127


def test_inputs_on_the_grid_are_exact():
    rng = np.random.default_rng(2)
    W = rng.integers(-127, 128, size=(8, 32)).astype(np.float64)
    W[:, 0] = 127  # every row reaches the grid's end, so s = 2^-7 exactly
    W *= 2.0 ** -7
    x = rng.integers(-127, 128, size=(4, 32)).astype(np.float64)
    x[:, 0] = -127
    x *= 2.0 ** -3
    qw, sw = w8a8.quantize_int8_rows(W)
    assert np.all(sw == np.float32(2.0 ** -7))
    assert np.array_equal(w8a8.dequant_rows(qw, sw, "int8"), W)
    y = w8a8.w8a8_linear(x, qw, sw, "int8")
    assert np.array_equal(y, x @ W.T)


def test_fp8_encoder_matches_torch_cast_in_range():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 1e-2,
                        np.array([0.0, -0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10])]).astype(np.float32)
    ours = w8a8.e4m3_encode_signed(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # torch keeps -0 as 0x80 and a negative value rounding to zero as -0; the oracle's
    # reading gives every zero the +0 code: compare the rest bit for bit
    zero = (ref & 0x7F) == 0
    assert np.array_equal(ours[~zero], ref[~zero])
    assert np.all(ours[zero] == 0)


def test_fp8_rounding_bound():
    rng = np.random.default_rng(4)
    X = (rng.standard_normal((32, 256)) * 3).astype(np.float32)
    q, s = w8a8.quantize_fp8_rows(X)
    rec = w8a8.dequant_rows(q, s, "fp8")
    v = np.abs(X.astype(np.float64)) / s[:, None]
    normal = v >= 2.0 ** -6  # E4M3 normal range: half an ulp is at most 2^-4 relative
    err = np.abs(X - rec) / s[:, None]
    assert np.all(err[normal] <= v[normal] * 2.0 ** -4 * (1 + 1e-9))
    assert np.all(err[~normal] <= 2.0 ** -10 + 1e-12)  # subnormal spacing 2^-9, half of it
    y = w8a8.w8a8_linear(X[:4], q, s, "fp8")
    assert y.shape == (4, 32) and np.all(np.isfinite(y))


def test_zero_rows_and_bad_format():
    q, s = w8a8.quantize_int8_rows(np.zeros((2, 16), np.float32))
    assert np.all(q == 0) and np.all(s == 1)
    c, s8 = w8a8.quantize_fp8_rows(np.zeros((2, 16), np.float32))
    assert np.all(c == 0) and np.all(s8 == 1)
    with pytest.raises(ValueError):
        w8a8.w8a8_linear(np.ones((1, 16)), q, s, "int4")
