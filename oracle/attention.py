"""Masked softmax attention of the verification pass (oracle; test infrastructure).

Source: SimSD summary, section 4 "Verification": the target runs one forward
pass over the paired input [prompt | D | D~] under the temporal causal mask,
producing logits for every drafted position at once.  This module computes
the attention layer of that pass, in float64, one (sequence, query head) at
a time, with the dense mask from ``oracle.mask``:

    O[row] = sum_key softmax_key( scale * <q_row, k_key> | allowed ) * v_key

with scale = 1/sqrt(d) (reading: the page fixes no scale) and grouped-query
heads: query head h reads kv head h // (Hq / Hkv) (reading: contiguous
groups).  Disallowed keys get weight exactly zero.
"""
from __future__ import annotations

from typing import Iterable, Optional

import numpy as np

from .mask import verify_mask


def masked_softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                             allowed: np.ndarray, scale: float) -> np.ndarray:
    """q [R, d], k/v [K, d], allowed [R, K] (0/1) -> [R, d], float64."""
    s = (q @ k.T) * scale
    s = np.where(allowed.astype(bool), s, -np.inf)
    m = np.max(s, axis=1, keepdims=True)
    w = np.where(allowed.astype(bool), np.exp(s - m), 0.0)
    return (w @ v) / np.sum(w, axis=1, keepdims=True)


def sequence_keys(seq, k_cache, v_cache, k_new, v_new, kv_head: int):
    """Keys/values of one sequence in mask order: [cache | fresh prompt | D | D~]."""
    C, N, B, q_off, kv_off, _ = (int(x) for x in seq)
    rows = N + 2 * B
    keys = np.concatenate([k_cache[kv_off:kv_off + C, kv_head], k_new[q_off:q_off + rows, kv_head]], axis=0)
    vals = np.concatenate([v_cache[kv_off:kv_off + C, kv_head], v_new[q_off:q_off + rows, kv_head]], axis=0)
    return keys, vals


def verify_attention(seqs: np.ndarray, tau: np.ndarray, q: np.ndarray, k_cache: np.ndarray,
                     v_cache: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
                     scale: Optional[float] = None,
                     rows_of: Optional[dict] = None) -> np.ndarray:
    """Attention output [rows, Hq, d] (float64) for a packed batch.

    All tensors are float64 values (post-RoPE Q and K_new).  ``rows_of`` may
    map sequence index -> iterable of local query rows to compute (others are
    left NaN); used to sample outputs at sizes too large for a full pass.
    """
    Hq = q.shape[1]
    Hkv = k_new.shape[1]
    d = q.shape[2]
    G = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    out = np.full(q.shape, np.nan, dtype=np.float64)
    for b, seq in enumerate(np.asarray(seqs)):
        C, N, B, q_off, _kv_off, t_off = (int(x) for x in seq)
        rows = N + 2 * B
        local = np.arange(rows) if rows_of is None or b not in rows_of else np.asarray(sorted(rows_of[b]), np.int64)
        if rows_of is not None and b not in rows_of:
            continue
        if local.size == 0:
            continue
        A = verify_mask(C, N, B, tau[t_off:t_off + B], rows=local)
        for h in range(Hq):
            kv = h // G
            keys, vals = sequence_keys(seq, k_cache, v_cache, k_new, v_new, kv)
            out[q_off + local, h] = masked_softmax_attention(q[q_off + local, h], keys, vals, A, scale)
    return out


def rows_sample(seqs: np.ndarray, per_seq_prompt: int, rng: np.random.Generator) -> dict:
    """Pick local rows per sequence: every tail row plus a few fresh prompt rows
    (first, last and random ones)."""
    pick = {}
    for b, (C, N, B, *_rest) in enumerate(np.asarray(seqs)):
        N, B = int(N), int(B)
        rows = set(range(N, N + 2 * B))
        if N > 0:
            rows |= {0, N - 1}
            rows |= set(int(x) for x in rng.integers(0, N, size=min(per_seq_prompt, N)))
        pick[b] = sorted(rows)
    return pick


def iter_heads(Hq: int, Hkv: int) -> Iterable[tuple]:
    G = Hq // Hkv
    for h in range(Hq):
        yield h, h // G
