"""NVFP4 format and fixed-scale quantiser -- CPU oracle (test infrastructure only).

Source: "QeRL: When Quantized Weights Help Reinforcement Learning, and Where the
Evidence Stops" (zhongzhuzhou.org), section 3.1 "What the four bits represent":

* E2M1 is one sign bit, two exponent bits and one mantissa bit; its non-negative
  values are 0, 0.5, 1, 1.5, 2, 3, 4, 6.
* One FP8 E4M3 block scale s_b per 16 consecutive weights, one FP32 tensor
  scale s_g for the whole tensor.
* Reconstruction:  w_hat[b, j] = s_g * s_b * q[b, j],  q in the E2M1 grid.
* Fixed-scale nearest-grid quantiser:  q = argmin_q |w - s_g s_b q|.
* Storage: P/2 bytes of 4-bit payload + P/16 bytes of block scales = 9P/16.

The pages leave open how s_g and s_b are chosen, the rounding of s_b, the tie
rule, the nibble order and the block axis.  Readings taken here:

* s_g = fp32(amax_t / 2688) with 2688 = 6 * 448 (largest E2M1 magnitude times
  largest finite E4M3), so the block holding the tensor maximum gets s_b = 448;
  s_g = 1 for an all-zero tensor.
* s_b = E4M3( fp32( amax_b / fp32(6 * s_g) ) ), rounded to nearest, ties to the
  even code, saturating at 448 (OCP FP8 E4M3 "FN" encoding, subnormals kept).
* Code selection runs in FP32: S = fp32(s_g * s_b); v = fp32(|w| / S); the
  magnitude is the nearest E2M1 grid point to v with ties to the even code
  (mantissa bit 0), saturating at 6; S == 0 gives code 0.  A value that rounds
  to magnitude 0 gets the +0 code, so every reconstructed value has exactly one
  code.  ``argmin_codes_exact`` gives the exact-real argmin of the pages for
  comparison.
* Blocks run along d_i (the input / reduction axis), 16 per block, no padding.
* Packing: byte [o][k/2] holds code(o, k) in its low nibble and code(o, k+1) in
  its high nibble (k even); scales are stored [o][k/16], one byte each.
"""

from __future__ import annotations

import numpy as np

BLOCK = 16  # weights per E4M3 block scale (section 3.1)
E2M1_MAX = 6.0
E4M3_MAX = 448.0
TENSOR_SCALE_DIVISOR = np.float32(E2M1_MAX * E4M3_MAX)  # 2688, exact in FP32


# ----------------------------------------------------------------------------
# E2M1 (FP4): 1 sign, 2 exponent bits (bias 1), 1 mantissa bit.
# ----------------------------------------------------------------------------
def e2m1_decode(code: int) -> float:
    """Value of a 4-bit E2M1 code, from its bit fields (sign | exp(2) | mant(1))."""
    code = int(code) & 0xF
    sign = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:  # subnormal: 0 or 0.5
        mag = 0.5 * m
    else:
        mag = 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return sign * mag


E2M1_TABLE = np.array([e2m1_decode(c) for c in range(16)], dtype=np.float64)
E2M1_POS = E2M1_TABLE[:8].copy()  # increasing magnitudes, index == magnitude code


# ----------------------------------------------------------------------------
# E4M3 (OCP FP8 "E4M3FN"): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
# no infinities, S.1111.111 is NaN, largest finite 448.
# ----------------------------------------------------------------------------
def e4m3_decode(code: int) -> float:
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        mag = (m / 8.0) * 2.0 ** -6
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return sign * mag


E4M3_TABLE = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
E4M3_POS = E4M3_TABLE[:0x7F].copy()  # codes 0x00..0x7E: increasing, finite, >= 0


def _nearest_even(values: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the nearest grid point to each value (grid increasing, starting at
    0): the number of midpoints between neighbours that lie strictly below the
    value, moved up by one when the value sits exactly on a midpoint whose upper
    neighbour has the even index (ties to even).  Values beyond the last grid point
    saturate to it.  Midpoints of FP32 grids are exact in FP64."""
    v = np.asarray(values, dtype=np.float64)
    mids = (grid[:-1] + grid[1:]) / 2.0
    k = np.searchsorted(mids, v, side="left")  # midpoints < v
    on_mid = mids[np.minimum(k, mids.shape[0] - 1)] == v
    k = k + (on_mid & (k % 2 == 1))
    return k.astype(np.int64)


def e4m3_encode(t) -> np.ndarray:
    """Round non-negative finite FP32 values to E4M3 codes: nearest, ties to the
    even code, saturating to 448 (0x7E).  Subnormal E4M3 values are produced."""
    t = np.asarray(t, dtype=np.float32)
    return _nearest_even(t, E4M3_POS).astype(np.uint8)


def e2m1_magnitude_code(v) -> np.ndarray:
    """Nearest E2M1 magnitude code (0..7) to non-negative v, ties to even code,
    saturating at 6 (code 7).  +inf maps to code 7."""
    return _nearest_even(v, E2M1_POS).astype(np.uint8)


# ----------------------------------------------------------------------------
# Quantiser (FP32 arithmetic contract) and packing.
# ----------------------------------------------------------------------------
def tensor_scale(W: np.ndarray) -> np.float32:
    """s_g = fp32(max|W| / 2688); 1 for an all-zero tensor."""
    amax = np.float32(np.max(np.abs(W.astype(np.float32)))) if W.size else np.float32(0)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(amax / TENSOR_SCALE_DIVISOR)


def block_scale_codes(W: np.ndarray, s_g: np.float32) -> np.ndarray:
    """E4M3 codes of the block scales, shape [d_o, d_i/16]."""
    d_o, d_i = W.shape
    blocks = np.abs(W.astype(np.float32)).reshape(d_o, d_i // BLOCK, BLOCK)
    amax_b = blocks.max(axis=2).astype(np.float32)
    denom = np.float32(np.float32(E2M1_MAX) * np.float32(s_g))
    t = (amax_b / denom).astype(np.float32)
    return e4m3_encode(t)


def element_codes(W: np.ndarray, s_g: np.float32, sb_codes: np.ndarray) -> np.ndarray:
    """4-bit codes (0..15) of every weight, shape [d_o, d_i] (elementwise, so it is
    evaluated in row chunks that stay cache-resident)."""
    d_o, d_i = W.shape
    rows = max(1, (1 << 20) // d_i)
    if d_o > rows:
        return np.concatenate([element_codes(W[o:o + rows], s_g, sb_codes[o:o + rows])
                               for o in range(0, d_o, rows)])
    W32 = W.astype(np.float32).reshape(d_o, d_i // BLOCK, BLOCK)
    s_b = E4M3_TABLE[sb_codes].astype(np.float32)
    S = (np.float32(s_g) * s_b).astype(np.float32)[..., None]
    absw = np.abs(W32)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = (absw / np.where(S == 0, np.float32(1), S)).astype(np.float32)
    mag = e2m1_magnitude_code(v)
    mag = np.where(np.broadcast_to(S == 0, mag.shape), 0, mag).astype(np.uint8)
    neg = (W32 < 0) & (mag != 0)
    return (mag | (neg.astype(np.uint8) << 3)).reshape(d_o, d_i).astype(np.uint8)


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """[d_o, d_i] 4-bit codes -> [d_o, d_i/2] bytes, even k in the low nibble."""
    lo = codes[:, 0::2].astype(np.uint8)
    hi = codes[:, 1::2].astype(np.uint8)
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    d_o, half = packed.shape
    out = np.empty((d_o, 2 * half), dtype=np.uint8)
    out[:, 0::2] = packed & 0x0F
    out[:, 1::2] = packed >> 4
    return out


def quantize(W: np.ndarray):
    """NVFP4-quantise W ([d_o, d_i], values already BF16-representable).

    Returns (packed codes uint8 [d_o, d_i/2], E4M3 scale codes uint8 [d_o, d_i/16],
    s_g float32)."""
    W = np.asarray(W)
    d_o, d_i = W.shape
    if d_i % BLOCK:
        raise ValueError("d_i must be a multiple of 16")
    s_g = tensor_scale(W)
    sb = block_scale_codes(W, s_g)
    codes = element_codes(W, s_g, sb)
    return pack_codes(codes), sb, s_g


def argmin_codes_exact(W: np.ndarray, s_g: float, sb_codes: np.ndarray) -> np.ndarray:
    """The pages' argmin |w - s_g s_b q| over the 15 distinct E2M1 values, in exact
    real arithmetic (FP64 here; every product and difference is exact), ties to
    the even code, +0 for zero.  Used to count where the FP32 contract departs
    from the exact argmin."""
    d_o, d_i = W.shape
    W64 = W.astype(np.float64).reshape(d_o, d_i // BLOCK, BLOCK)
    S = (float(s_g) * E4M3_TABLE[sb_codes])[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        # |w - S q| compared on |w| against S * grid (sign handled separately)
        d = np.abs(np.abs(W64)[..., None] - S[..., None] * E2M1_POS)
    best = np.argmin(d, axis=-1)  # first minimum = lower index
    # ties: argmin picked the lower index; move to the upper one when it is even
    nxt = np.clip(best + 1, 0, 7)
    dbest = np.take_along_axis(d, best[..., None], -1)[..., 0]
    dnext = np.take_along_axis(d, nxt[..., None], -1)[..., 0]
    move = (nxt != best) & (dnext == dbest) & (nxt % 2 == 0)
    mag = np.where(move, nxt, best).astype(np.uint8)
    mag = np.where(S == 0, 0, mag).astype(np.uint8)
    neg = (W64 < 0) & (mag != 0)
    return (mag | (neg.astype(np.uint8) << 3)).reshape(d_o, d_i)


def dequantize(packed: np.ndarray, sb_codes: np.ndarray, s_g) -> np.ndarray:
    """Reconstruction w_hat = s_g * s_b * q in FP64, shape [d_o, d_i]."""
    codes = unpack_codes(packed)
    d_o, d_i = codes.shape
    q = E2M1_TABLE[codes].reshape(d_o, d_i // BLOCK, BLOCK)
    s_b = E4M3_TABLE[sb_codes][..., None]
    return (float(s_g) * s_b * q).reshape(d_o, d_i)


def storage_bytes(d_o: int, d_i: int) -> int:
    """Bytes of payload plus block scales (the tensor scale's 4 bytes excluded)."""
    P = d_o * d_i
    return P // 2 + P // BLOCK
