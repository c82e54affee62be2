"""Rotary position embedding with the RoPE-copy index (oracle; test infrastructure).

Source: SimSD summary, section 3 "Position Encoding Alignment": each mask
slot D~_k reuses the RoPE index of its paired data token D_k, so the pair
occupies one position.  The page fixes no RoPE convention; the reading used
here is the rotate-half form with theta_i = base^(-2i/d), base 10000, and
absolute position 0 at the first cache key.

Positions of one sequence's query rows (cache keys arrive already rotated):
  * fresh prompt row i        -> C + i
  * tail row r (0 <= r < 2B)  -> P + (r mod B), with P = C + N
so D_k (r = k-1) and D~_k (r = B + k-1) share position P + k - 1; or, with
explicit positions for the fresh rows and data rows, those, and D~_k again
takes D_k's.
"""
from __future__ import annotations

import numpy as np


def rope_positions(C: int, N: int, B: int, given=None) -> np.ndarray:
    """int64 [N + 2B] absolute position of each query row of one sequence.

    `given` (optional, N + B entries): explicit positions of the N fresh
    prompt rows and of the data rows D_1..D_B, for a pass whose positions are
    not contiguous (the remaining slots of a block after a commit, which
    keep their own slots' positions; a reading, the pages do not describe
    the loop).  Mask row D~_k still takes D_k's position (RoPE copy)."""
    if given is not None:
        given = [int(x) for x in given]
        assert len(given) == N + B
        return np.asarray(given[:N] + [given[N + (r % B)] for r in range(2 * B)], dtype=np.int64)
    P = C + N
    pos = [C + i for i in range(N)]
    pos += [P + (r % B) for r in range(2 * B)]
    return np.asarray(pos, dtype=np.int64)


def inv_freq(d: int, base: float = 10000.0) -> np.ndarray:
    """theta_i = base^(-2i/d), i = 0 .. d/2-1, float64."""
    return np.asarray([base ** (-2.0 * i / d) for i in range(d // 2)], dtype=np.float64)


def rotate(x: np.ndarray, pos: np.ndarray, base: float = 10000.0) -> np.ndarray:
    """Rotate-half RoPE in float64.

    x: [rows, heads, d]; pos: [rows].  For pair (x_i, x_{i+d/2}) at angle
    a = pos * theta_i: out_i = x_i cos a - x_{i+d/2} sin a,
    out_{i+d/2} = x_{i+d/2} cos a + x_i sin a.
    """
    x = np.asarray(x, dtype=np.float64)
    rows, heads, d = x.shape
    half = d // 2
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq(d, base)[None, :]   # [rows, half]
    cos = np.cos(ang)[:, None, :]
    sin = np.sin(ang)[:, None, :]
    x1 = x[:, :, :half]
    x2 = x[:, :, half:]
    out = np.empty_like(x)
    out[:, :, :half] = x1 * cos - x2 * sin
    out[:, :, half:] = x2 * cos + x1 * sin
    return out


def rope_copy_batch(seqs: np.ndarray, q: np.ndarray, k: np.ndarray, base: float = 10000.0, positions=None):
    """Rotate Q [rows, Hq, d] and K_new [rows, Hkv, d] of a packed batch
    (float64).  positions: optional [rows] table, read at each sequence's
    fresh rows and data rows (see rope_positions)."""
    qo = np.empty(q.shape, np.float64)
    ko = np.empty(k.shape, np.float64)
    for C, N, B, q_off, _kv_off, _t in np.asarray(seqs):
        rows = N + 2 * B
        given = None if positions is None else np.asarray(positions)[q_off:q_off + N + B]
        pos = rope_positions(int(C), int(N), int(B), given)
        qo[q_off:q_off + rows] = rotate(q[q_off:q_off + rows], pos, base)
        ko[q_off:q_off + rows] = rotate(k[q_off:q_off + rows], pos, base)
    return qo, ko
