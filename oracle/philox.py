"""Counter-based Gaussian noise for the oracle: Philox4xW-10 and Box-Muller.

TEST INFRASTRUCTURE ONLY (see the package header).

The pages fix only the distribution of the privacy noise, N(0, sigma^2 C^2 I)
("Scalable and Efficient Training of Large CNNs with DP", Preliminaries, the
Gaussian mechanism; "Scaling up DP Deep Learning with Fast Per-Example Gradient
Clipping", section 2, the Gaussian mechanism).  The generator is therefore our
reading: Philox4x32-10 as published by Salmon, Moraes, Dror and Shaw,
"Parallel random numbers: as easy as 1, 2, 3" (SC'11), section 3.2 and its
table of multipliers and round keys, followed by the Box-Muller transform.

The round function is written once for word widths 32 and 64.  The 64-bit
instance is pinned bit for bit against numpy.random.Philox (a Philox4x64-10
library implementation); the 32-bit instance, which the noise uses, shares the
same code and differs only in the published constants.

Noise stream (element index e >= 0, 64-bit seed, stream id s):
  block q = e // 4, lane r = e % 4
  counter = (q mod 2^32, q // 2^32, s, 0), key = (seed mod 2^32, seed // 2^32)
  (x0, x1, x2, x3) = Philox4x32-10(counter, key)
  u_k = (floor(x_k / 2^9) + 1/2) / 2^23          (exact in fp32, in (0, 1))
  z0, z1 = sqrt(-2 ln u0) * (cos 2 pi u1, sin 2 pi u1)
  z2, z3 = sqrt(-2 ln u2) * (cos 2 pi u3, sin 2 pi u3)
  element e takes z_r.
Stream 0 is the gradient noise; stream 1 is the adaptive bound's noise.
"""
from __future__ import annotations

import numpy as np

# Multipliers and round-key increments of Philox4xW (Salmon et al. 2011).
PHILOX_CONSTANTS = {
    32: dict(M0=0xD2511F53, M1=0xCD9E8D57, W0=0x9E3779B9, W1=0xBB67AE85),
    64: dict(M0=0xD2E7470EE14C6C93, M1=0xCA5A826395121157,
             W0=0x9E3779B97F4A7C15, W1=0xBB67AE8584CAA73B),
}
_M32 = np.uint64(0xFFFFFFFF)


def _mulhilo(a: int, b: np.ndarray, width: int):
    """(hi, lo) words of the 2W-bit product a*b, elementwise on uint64 arrays."""
    b = b.astype(np.uint64)
    if width == 32:
        prod = np.uint64(a) * b                 # < 2^64: exact
        return prod >> np.uint64(32), prod & _M32
    # 64-bit words: schoolbook product on 32-bit limbs.
    a0, a1 = np.uint64(a & 0xFFFFFFFF), np.uint64(a >> 32)
    b0, b1 = b & _M32, b >> np.uint64(32)
    p00, p01, p10, p11 = a0 * b0, a0 * b1, a1 * b0, a1 * b1
    mid = (p00 >> np.uint64(32)) + (p01 & _M32) + (p10 & _M32)
    lo = (p00 & _M32) | ((mid & _M32) << np.uint64(32))
    hi = p11 + (p01 >> np.uint64(32)) + (p10 >> np.uint64(32)) + (mid >> np.uint64(32))
    return hi, lo


def philox4(counter, key, width: int = 32, rounds: int = 10):
    """Philox4xW-R block function.

    counter: 4 arrays (or ints) of W-bit words, key: 2 words.  Returns the 4
    output words as uint64 arrays.  Each round multiplies words 0 and 2 by the
    two multipliers, XORs the high halves with the other two words and the round
    key, and permutes; the key advances by the Weyl increments between rounds.
    """
    k = PHILOX_CONSTANTS[width]
    mask = np.uint64((1 << width) - 1)
    c = [np.asarray(x, dtype=np.uint64) & mask for x in counter]
    k0 = np.asarray(key[0], dtype=np.uint64) & mask
    k1 = np.asarray(key[1], dtype=np.uint64) & mask
    with np.errstate(over="ignore"):          # key words wrap modulo 2^W
        for r in range(rounds):
            if r:
                k0 = (k0 + np.uint64(k["W0"])) & mask
                k1 = (k1 + np.uint64(k["W1"])) & mask
            hi0, lo0 = _mulhilo(k["M0"], c[0], width)
            hi1, lo1 = _mulhilo(k["M1"], c[2], width)
            c = [(hi1 ^ c[1] ^ k0) & mask, lo1 & mask, (hi0 ^ c[3] ^ k1) & mask, lo0 & mask]
    return c


def uniform_from_word(x: np.ndarray) -> np.ndarray:
    """u = (floor(x / 2^9) + 1/2) / 2^23 in (0, 1), as float64 (exact)."""
    return ((np.asarray(x, dtype=np.uint64) >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def noise_words(n: int, seed: int, offset: int = 0, stream: int = 0):
    """Raw Philox4x32-10 words for elements offset .. offset+n-1: array [n_blocks, 4] and first block."""
    if n <= 0:
        return np.zeros((0, 4), dtype=np.uint64), 0
    q0 = offset // 4
    q1 = (offset + n - 1) // 4
    q = np.arange(q0, q1 + 1, dtype=np.uint64)
    ctr = (q & _M32, q >> np.uint64(32), np.full_like(q, stream & 0xFFFFFFFF), np.zeros_like(q))
    key = (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    x = philox4(ctr, key, width=32)
    return np.stack(x, axis=1), q0


def normal_noise(n: int, seed: int, offset: int = 0, stream: int = 0) -> np.ndarray:
    """Standard normal draws z_e for e = offset .. offset+n-1 (float64)."""
    if n <= 0:
        return np.zeros(0)
    words, q0 = noise_words(n, seed, offset, stream)
    u = uniform_from_word(words)                              # [blocks, 4]
    r01 = np.sqrt(-2.0 * np.log(u[:, 0]))
    r23 = np.sqrt(-2.0 * np.log(u[:, 2]))
    th1 = 2.0 * np.pi * u[:, 1]
    th3 = 2.0 * np.pi * u[:, 3]
    z = np.stack([r01 * np.cos(th1), r01 * np.sin(th1), r23 * np.cos(th3), r23 * np.sin(th3)], axis=1)
    flat = z.reshape(-1)
    start = offset - 4 * q0
    return flat[start:start + n].copy()
