"""Coupled Gumbel noise generated from a counter-based generator (oracle;
test infrastructure).

Source: SPOT review (onedev.kr), section "How it is used": drafter and target
share one Gumbel noise table per absolute output position, which makes the
target's transition a deterministic function of the noise, and marginalising
over the noise recovers the target's sampling distribution (the review's
Proposition 2).  The table can be replaced by a generator both sides
evaluate identically -- the reading taken here (the pages do not say how the
table is produced):

  G(seed, pos, v) = -L(-L(U)),   U = (floor(x / 2^9) + 1/2) * 2^-23,
  x = word (v mod 4) of Philox4x32-10(counter = (floor(v / 4), pos, 0, 0),
                                      key = (seed mod 2^32, floor(seed / 2^32)))

with `pos` the 32-bit position the caller assigns to the slot (one per
absolute output position of a request; drafter and target use the same) and
L the natural logarithm evaluated by the fixed sequence of IEEE fp32
operations below (each rounded to nearest, none fused), so that the GPU and
this oracle produce the same bits.

Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
as 1, 2, 3" (SC11).  Ten rounds of: (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2
(32 x 32 -> 64-bit products), c = (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0),
then the key is bumped by the Weyl constants (k0 += W0, k1 += W1).

L(x), x > 0 normal (argument reduction of Cody and Waite, "Software Manual
for the Elementary Functions", 1980; the series of Gregory for
ln((1 + s) / (1 - s)) = 2 atanh s):
  x = 2^e * m with m in [1, 2) (from the bits); if m > sqrt 2 then m = m / 2,
  e = e + 1, so m lies in [sqrt(1/2), sqrt 2] and |s| <= 0.1716 below;
  f = m - 1                     (exact)
  s = f / (2 + f)
  z = s * s
  t = ((((2/9) z + 2/7) z + 2/5) z + 2/3) z      (Horner, each step rounded)
  L = e * ln2 + (2 s + s * t)
The series is truncated after s^9: the remainder is below 2 s^11 / 11, a
relative 4e-9 of the result, under fp32's own rounding.
"""
from __future__ import annotations

import numpy as np

# Philox4x32 multipliers and Weyl key increments (the published constants)
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85

F32 = np.float32
LN2 = F32(np.log(2.0))
SQRT2 = F32(np.sqrt(2.0))
C3, C5, C7, C9 = F32(2.0 / 3.0), F32(2.0 / 5.0), F32(2.0 / 7.0), F32(2.0 / 9.0)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds, element-wise over arrays of 32-bit words.
    Returns the four output words as uint32 arrays."""
    mask = np.uint64(0xFFFFFFFF)
    c = [np.asarray(x, dtype=np.uint64) & mask for x in (c0, c1, c2, c3)]
    k0 = np.asarray(k0, dtype=np.uint64) & mask
    k1 = np.asarray(k1, dtype=np.uint64) & mask
    for _ in range(10):
        p0 = np.uint64(PHILOX_M0) * c[0]
        p1 = np.uint64(PHILOX_M1) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & mask
        hi1, lo1 = p1 >> np.uint64(32), p1 & mask
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
        k0 = (k0 + np.uint64(PHILOX_W0)) & mask
        k1 = (k1 + np.uint64(PHILOX_W1)) & mask
    return [x.astype(np.uint32) for x in c]


def uniform_from_bits(x) -> np.ndarray:
    """U = (floor(x / 2^9) + 1/2) * 2^-23 in fp32 (exact), in the open interval (0, 1)."""
    k = (np.asarray(x, dtype=np.uint32) >> np.uint32(9)).astype(np.float32)
    return (k + F32(0.5)) * F32(2.0 ** -23)


def log_f32(x) -> np.ndarray:
    """Natural logarithm of positive normal fp32 values by the fixed operation
    sequence of the module docstring (numpy float32 arithmetic is IEEE
    round-to-nearest per operation)."""
    x = np.asarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    e = ((bits >> np.uint32(23)) & np.uint32(0xFF)).astype(np.int32) - 127
    m = ((bits & np.uint32(0x7FFFFF)) | np.uint32(0x3F800000)).view(np.float32)
    big = m > SQRT2
    m = np.where(big, m * F32(0.5), m).astype(np.float32)
    e = e + big.astype(np.int32)
    f = m - F32(1.0)
    s = f / (F32(2.0) + f)
    z = s * s
    t = C9 * z
    t = t + C7
    t = t * z
    t = t + C5
    t = t * z
    t = t + C3
    t = t * z
    ln1p = F32(2.0) * s + s * t
    return (e.astype(np.float32) * LN2 + ln1p).astype(np.float32)


def noise_bits(seed: int, pos, V: int) -> np.ndarray:
    """uint32 [len(pos), V]: word (v mod 4) of Philox4x32-10 at counter
    (floor(v / 4), pos, 0, 0) under key (seed low word, seed high word)."""
    pos = np.atleast_1d(np.asarray(pos, dtype=np.uint64))
    v = np.arange(V, dtype=np.uint64)
    c0 = np.broadcast_to(v >> np.uint64(2), (len(pos), V))
    c1 = np.broadcast_to(pos[:, None], (len(pos), V))
    words = philox4x32_10(c0, c1, 0, 0, int(seed) & 0xFFFFFFFF, (int(seed) >> 32) & 0xFFFFFFFF)
    sel = (v & np.uint64(3)).astype(np.int64)
    out = np.empty((len(pos), V), np.uint32)
    for j in range(4):
        m = sel == j
        out[:, m] = words[j][:, m]
    return out


def gumbel_rows(seed: int, pos, V: int) -> np.ndarray:
    """fp32 [len(pos), V]: G(seed, pos, v) = -L(-L(U))."""
    u = uniform_from_bits(noise_bits(seed, pos, V))
    return (-log_f32(-log_f32(u))).astype(np.float32)


def gumbel_generated(seed: int, pos: int, V: int) -> np.ndarray:
    """fp32 row G(seed, pos, v), v = 0..V-1."""
    return gumbel_rows(seed, [pos], V)[0]
