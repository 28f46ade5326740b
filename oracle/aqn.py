"""AQN noise state: schedule, stage and counter-based draws -- CPU oracle.

Test infrastructure only: tests, the smoke check and the bench's CPU baseline may
import this module; the library never does.

Source: "QeRL: When Quantized Weights Help Reinforcement Learning, and Where the
Evidence Stops" (zhongzhuzhou.org):

* section 5.1: the noise enters the RMSNorm scale, h = u (.) (w + z), one channel
  vector z per normalisation, shared by the projections that read that norm;
* section 5.2 "A schedule needs consistent endpoints": ten stages, stage 0 without
  noise, then sigma_k = sigma_start * (sigma_end / sigma_start) ** ((k - 1) / 8) for
  k = 1 .. 9, so stage 1 is exactly the start and stage 9 exactly the end value;
* section 6 "A training algorithm that exposes the stochastic state": the stage
  follows from the number of completed updates and the planned horizon, and the noise
  is drawn from a recorded seed under a declared persistence scope (one state per
  rollout, per response or per token).

The pages leave open the stage boundaries, the distribution's details and the
generator.  Readings taken here:

* stage = min(9, floor(10 * done / total)): ten stages of equal length, stage 0
  (the warm-up, sigma 0) first;
* z ~ N(0, sigma_k^2), independent over the d channels;
* generator: Philox4x32-10, the counter-based generator of Salmon, Moraes, Dror and
  Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC 2011), restated from its
  published definition: ten rounds, each multiplying two of the four counter words
  by 0xD2511F53 and 0xCD9E8D57 and mixing the high halves with the other words and
  the key, the key bumped by the Weyl constants 0x9E3779B9 and 0xBB67AE85 after
  every round.  Key = the 64-bit seed (low word first); counter = (block index,
  norm index, scope index low word, scope index high word), where block b holds
  channels 4b .. 4b+3 and the scope index names the rollout, response or token the
  state belongs to;
* uniforms: u = (2 * (x >> 9) + 1) * 2^-24 for each 32-bit word x: 23 random bits,
  exactly representable in FP32, strictly inside (0, 1);
* normals (Box-Muller): from words (x0, x1) of a block, rho = sqrt(-2 ln u0) and
  channels 4b, 4b+1 get rho cos(2 pi u1), rho sin(2 pi u1); from (x2, x3) likewise
  channels 4b+2, 4b+3; z = sigma * normal.
"""

from __future__ import annotations

import math

import numpy as np

STAGES = 10  # stage 0 (no noise) and the nine noisy stages 1 .. 9 (section 5.2)

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK32 = 0xFFFFFFFF


# ----------------------------------------------------------------------------
# Schedule (section 5.2) and stage (section 6)
# ----------------------------------------------------------------------------
def sigma(stage: int, sigma_start: float, sigma_end: float) -> float:
    """sigma_0 = 0; sigma_k = start * (end / start) ** ((k - 1) / 8), k = 1 .. 9 (FP64)."""
    k = int(stage)
    if k < 0 or k >= STAGES:
        raise ValueError(f"stage {k} outside 0 .. {STAGES - 1}")
    if k == 0:
        return 0.0
    return float(sigma_start) * (float(sigma_end) / float(sigma_start)) ** ((k - 1) / 8.0)


def stage(done: int, total: int) -> int:
    """Stage of the schedule after `done` of `total` planned updates: ten equal parts."""
    if total < 1 or done < 0:
        raise ValueError("need total >= 1 and done >= 0")
    return min(STAGES - 1, (STAGES * int(done)) // int(total))


# ----------------------------------------------------------------------------
# Philox4x32-10 (Salmon et al., SC 2011)
# ----------------------------------------------------------------------------
def philox4x32_10(counter, key):
    """One block of four 32-bit words from a 4-word counter and a 2-word key (Python ints)."""
    c0, c1, c2, c3 = (int(v) & _MASK32 for v in counter)
    k0, k1 = (int(v) & _MASK32 for v in key)
    for _ in range(10):
        p0 = PHILOX_M0 * c0
        p1 = PHILOX_M1 * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0, p1 & _MASK32, (p0 >> 32) ^ c3 ^ k1, p0 & _MASK32)
        k0 = (k0 + PHILOX_W0) & _MASK32
        k1 = (k1 + PHILOX_W1) & _MASK32
    return c0, c1, c2, c3


def philox4x32_10_array(c0, c1, c2, c3, k0: int, k1: int):
    """The same rounds over arrays of counters (uint64 arrays holding 32-bit values)."""
    m = np.uint64(_MASK32)
    c0, c1, c2, c3 = (np.asarray(v, dtype=np.uint64) & m for v in (c0, c1, c2, c3))
    k0, k1 = np.uint64(k0 & _MASK32), np.uint64(k1 & _MASK32)
    for _ in range(10):
        p0 = np.uint64(PHILOX_M0) * c0  # < 2^64: no wrap
        p1 = np.uint64(PHILOX_M1) * c2
        c0, c1, c2, c3 = ((p1 >> np.uint64(32)) ^ c1 ^ k0, p1 & m, (p0 >> np.uint64(32)) ^ c3 ^ k1, p0 & m)
        k0 = (k0 + np.uint64(PHILOX_W0)) & m
        k1 = (k1 + np.uint64(PHILOX_W1)) & m
    return c0, c1, c2, c3


def uniform(words) -> np.ndarray:
    """u = (2 (x >> 9) + 1) 2^-24 in FP64 (the same value is exact in FP32)."""
    x = np.asarray(words, dtype=np.uint64)
    return (2.0 * (x >> np.uint64(9)).astype(np.float64) + 1.0) * 2.0 ** -24


# ----------------------------------------------------------------------------
# Noise state
# ----------------------------------------------------------------------------
def box_muller(x0, x1, x2, x3):
    """The four normals of one block from its four Philox words (arrays or scalars)."""
    u0, u1, u2, u3 = uniform(x0), uniform(x1), uniform(x2), uniform(x3)
    rho_a = np.sqrt(-2.0 * np.log(u0))
    rho_b = np.sqrt(-2.0 * np.log(u2))
    return (rho_a * np.cos(2.0 * math.pi * u1), rho_a * np.sin(2.0 * math.pi * u1),
            rho_b * np.cos(2.0 * math.pi * u3), rho_b * np.sin(2.0 * math.pi * u3))


def noise_block(seed: int, norm_id: int, scope: int, b: int):
    """Channels 4b .. 4b+3 of the unit-sigma state of (seed, norm_id, scope), FP64."""
    x = philox4x32_10((b, norm_id, scope & _MASK32, (scope >> 32) & _MASK32), (seed & _MASK32, (seed >> 32) & _MASK32))
    return tuple(float(v) for v in box_muller(*(np.uint64(w) for w in x)))


def noise(seed: int, norm_id: int, scope0: int, n_scopes: int, d: int, sig: float) -> np.ndarray:
    """z [n_scopes][d] (FP64): row s is the state of scope index scope0 + s of norm `norm_id`."""
    if d < 1 or n_scopes < 1:
        raise ValueError("need d >= 1 and n_scopes >= 1")
    nb = (d + 3) // 4
    out = np.empty((n_scopes, 4 * nb), dtype=np.float64)
    k0, k1 = seed & _MASK32, (seed >> 32) & _MASK32
    blocks = np.arange(nb, dtype=np.uint64)
    for s in range(n_scopes):
        sc = int(scope0) + s
        x0, x1, x2, x3 = philox4x32_10_array(blocks, np.full(nb, norm_id, np.uint64),
                                             np.full(nb, sc & _MASK32, np.uint64),
                                             np.full(nb, (sc >> 32) & _MASK32, np.uint64), k0, k1)
        out[s, 0::4], out[s, 1::4], out[s, 2::4], out[s, 3::4] = box_muller(x0, x1, x2, x3)
    return float(sig) * out[:, :d]
