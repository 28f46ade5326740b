"""Pins of the oracle's NVFP4 quantiser and packing (CPU only).

Against the pages: the argmin reconstruction rule and the 9P/16 storage equation
(QeRL review, section 3.1); against brute force: per-element argmin on small
blocks, pure-Python nibble decode; against closed forms: the error bound of
round-to-nearest on the E2M1 grid.
"""

import numpy as np
import pytest
import torch

from oracle import nvfp4
from precision_linear_gb300 import synthetic
from tests.conftest import read_golden


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def _weights(d_o, d_i, seed=0, outliers=0.0):
    return synthetic.weight(d_o, d_i, seed, outliers).float().numpy()


def test_tensor_scale_and_max_block():
    W = _weights(64, 256, seed=1, outliers=1e-2)
    packed, sb, s_g = nvfp4.quantize(W)
    amax = np.abs(W).max()
    assert s_g == np.float32(amax / np.float32(2688.0))
    # the block holding the tensor maximum uses the largest E4M3 scale 448
    o, k = np.unravel_index(np.argmax(np.abs(W)), W.shape)
    assert sb[o, k // 16] == 0x7E
    assert np.all(nvfp4.E4M3_TABLE[sb] <= 448.0)
    # and that element reconstructs exactly to +-amax (6 * s_g * 448 = amax up to rounding of s_g)
    codes = nvfp4.unpack_codes(packed)
    assert codes[o, k] & 7 == 7


def test_argmin_rule_matches_exact_argmin():
    """Codes equal the pages' argmin |w - s_g s_b q| except where |w|/S sits
    within an FP32 rounding of a decision threshold."""
    W = _weights(96, 512, seed=2, outliers=1e-2)
    packed, sb, s_g = nvfp4.quantize(W)
    codes = nvfp4.unpack_codes(packed)
    exact = nvfp4.argmin_codes_exact(W, s_g, sb)
    diff = np.nonzero(codes != exact)
    S = (np.float64(s_g) * nvfp4.E4M3_TABLE[sb]).repeat(16, axis=1)
    v = np.abs(W.astype(np.float64)) / S
    thresholds = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    What = nvfp4.dequantize(packed, sb, s_g)
    Wex = nvfp4.dequantize(nvfp4.pack_codes(exact), sb, s_g)
    for o, k in zip(*diff):
        # only quasi-ties: |w|/S within FP32 rounding of a decision threshold ...
        assert np.min(np.abs(v[o, k] - thresholds)) <= 4e-7 * v[o, k]
        # ... where both choices are equally near w up to that rounding
        e_contract = abs(W[o, k] - What[o, k])
        e_exact = abs(W[o, k] - Wex[o, k])
        assert e_contract - e_exact <= 1e-6 * S[o, k]
    # quasi-ties are rare: weights that are exact binary fractions of the block
    # maximum (e.g. amax/8 -> |w|/S = 0.75) are the ones that land there
    assert len(diff[0]) <= 1e-3 * W.size


def test_argmin_bruteforce_tiny_blocks():
    """Pure-Python brute force over all 16 codes for seeded blocks and constructed
    ties (values exactly at S * midpoint)."""
    rng = np.random.default_rng(5)
    rows = [rng.normal(0, 0.02, 16) for _ in range(24)]
    # a block whose max is exactly 6*S and whose other entries hit every midpoint
    s = 0.01
    rows.append(np.array([6, .25, .75, 1.25, 1.75, 2.5, 3.5, 5, -.25, -.75, -1.25, -1.75, -2.5, -3.5, -5, 0]) * s)
    W = _bf16(np.stack(rows))
    W = np.concatenate([W, np.zeros((W.shape[0], 0))], axis=1).astype(np.float32)
    W16 = np.zeros((W.shape[0], 16), np.float32)
    W16[:] = W
    packed, sb, s_g = nvfp4.quantize(W16)
    codes = nvfp4.unpack_codes(packed)
    for o in range(W16.shape[0]):
        S = float(np.float32(s_g * np.float32(nvfp4.e4m3_decode(int(sb[o, 0])))))
        for k in range(16):
            w = float(W16[o, k])
            v = float(np.float32(np.float32(abs(w)) / np.float32(S)))
            best = None
            for c in range(16):
                q = nvfp4.e2m1_decode(c)
                if c == 8:
                    continue  # -0 is never produced
                if (w < 0) != (q < 0) and q != 0:
                    continue
                d = abs(v - abs(q))
                mag = c & 7
                if best is None or d < best[0] or (d == best[0] and mag % 2 == 0 and best[1] & 7 != mag):
                    best = (d, c)
            assert codes[o, k] == best[1], (o, k, w, v, codes[o, k], best)


def test_round_to_nearest_error_bound():
    W = _weights(128, 1024, seed=3, outliers=1e-3)
    packed, sb, s_g = nvfp4.quantize(W)
    What = nvfp4.dequantize(packed, sb, s_g)
    S = (np.float64(s_g) * nvfp4.E4M3_TABLE[sb]).repeat(16, axis=1)
    a = np.abs(W.astype(np.float64))
    inside = a <= 6 * S
    # half the local grid gap: 0.25 below 2 (gap 0.5), 0.5 below 4, 1 below 6
    half_gap = np.where(a < 2 * S, 0.25, np.where(a < 4 * S, 0.5, 1.0)) * S
    err = np.abs(W - What)
    assert np.all(err[inside] <= half_gap[inside] * (1 + 1e-6) + 1e-30)
    # outside the grid the value saturates to +-6 S
    assert np.allclose(np.abs(What[~inside]), 6 * S[~inside])


def test_zero_tensor_block_and_negative_zero():
    W = np.zeros((4, 32), np.float32)
    packed, sb, s_g = nvfp4.quantize(W)
    assert s_g == 1.0 and not packed.any() and not sb.any()
    W = _weights(4, 64, seed=4)
    W[1, 16:32] = 0.0  # one all-zero block
    W[2, 0] = -1e-9  # rounds to magnitude 0: must get the +0 code
    packed, sb, s_g = nvfp4.quantize(W)
    codes = nvfp4.unpack_codes(packed)
    assert sb[1, 1] == 0 and not codes[1, 16:32].any()
    assert codes[2, 0] == 0
    assert not np.any(codes == 8)


def test_pack_nibble_order():
    codes = np.array([[1, 2, 3, 4, 15, 0, 7, 8] + [0] * 8], dtype=np.uint8)
    packed = nvfp4.pack_codes(codes)
    assert packed.tolist()[0][:4] == [0x21, 0x43, 0x0F, 0x87]
    assert np.array_equal(nvfp4.unpack_codes(packed), codes)


def test_dequantize_pure_python():
    W = _weights(8, 64, seed=6, outliers=0.05)
    packed, sb, s_g = nvfp4.quantize(W)
    What = nvfp4.dequantize(packed, sb, s_g)
    for o in range(8):
        for k in range(64):
            byte = int(packed[o, k // 2])
            code = (byte >> 4) if (k % 2) else (byte & 0xF)
            sign = -1.0 if code & 8 else 1.0
            e, m = (code >> 1) & 3, code & 1
            q = sign * (0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + m / 2))
            sc = int(sb[o, k // 16])
            se, sm = (sc >> 3) & 15, sc & 7
            s_b = (sm / 8) * 2.0 ** -6 if se == 0 else (1 + sm / 8) * 2.0 ** (se - 7)
            assert What[o, k] == float(s_g) * s_b * q


@pytest.mark.parametrize("d_o,d_i", [(256, 256), (3584, 3584), (512, 3584), (18944, 3584), (3584, 18944),
                                     (8192, 5120), (1024, 5120), (5120, 27648)])
def test_storage_is_9P_over_16(d_o, d_i):
    g = read_golden("nvfp4_storage.txt")
    P = d_o * d_i
    expect = P * int(g["bytes_numerator"]) // int(g["bytes_denominator"])
    assert nvfp4.storage_bytes(d_o, d_i) == expect
    # shapes of the arrays the quantiser returns (checked on a 16-row slice)
    W = np.zeros((16, d_i), np.float32)
    packed, sb, _ = nvfp4.quantize(W)
    assert (packed.nbytes + sb.nbytes) * (d_o // 16) == expect
    assert 8 * expect / P == g["bits_per_weight"]
    ratio = (2 * P) / expect
    assert ratio == g["ratio_vs_bf16_numerator"] / g["ratio_vs_bf16_denominator"]
    assert round(ratio, 2) == g["ratio_vs_bf16_printed"]
