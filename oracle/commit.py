"""Commit of a verification pass into the KV cache (oracle; test infrastructure).

Sources:
  * SimSD summary, section 4 "Speculative decoding pipeline", Acceptance: the
    longest accepted prefix (in the temporal order the draft induces) is
    committed and the loop repeats.
  * SimSD summary, "Main contributions" 3: the method composes with a KV cache
    and blockwise decoding.

Reading (the pages give no cache layout or commit rule): after the pass over
sequence b (C cached keys, N fresh prompt rows, block B, stage map tau, n_acc
accepted stages) the sequence's cache gains, appended after its C rows:
  * the keys and values of the N fresh prompt rows, in row order (they were
    attended causally and are final), then
  * those of the data rows of the accepted stages, in stage order: stage
    s = 1..n_acc is slot k = tau^{-1}(s), i.e. fresh row N + k.
Mask rows are never committed: they stand for undecided tokens.  Rows keep the
rotation they carry (each data row at its own slot's position), so the cache
holds the accepted tokens in decoding order; attention over cache keys does
not depend on their order.  The sequence's new cache length is C + N + n_acc.

Layouts: fresh rows k_new, v_new [total_rows, Hkv, d] packed per sequence at
q_off; destination caches k_dst, v_dst [dst_rows, Hkv, d] with sequence b's
cache starting at row dst_off[b].
"""
from __future__ import annotations

import numpy as np


def committed_rows(N: int, B: int, tau, n_acc: int) -> list:
    """Indices (within the sequence's N + 2B fresh rows) of the rows appended
    to its cache, in append order."""
    stage_to_slot = {}
    for k in range(B):
        stage_to_slot[int(tau[k])] = k
    rows = [i for i in range(N)]
    for s in range(1, n_acc + 1):
        rows.append(N + stage_to_slot[s])
    return rows


def commit_batch(seqs, tau_all, n_acc, k_new, v_new, k_dst, v_dst, dst_off):
    """Applies the commit of every sequence to copies of the destination
    caches.  seqs rows: (cache_len, new_len, block, q_off, kv_off, tau_off).
    Returns (k_out, v_out, new_len)."""
    k_out = np.array(k_dst, copy=True)
    v_out = np.array(v_dst, copy=True)
    new_len = np.zeros(len(seqs), dtype=np.int64)
    for b, s in enumerate(seqs):
        C, N, B, q_off, _, tau_off = (int(v) for v in s[:6])
        tau = [int(t) for t in tau_all[tau_off:tau_off + B]]
        n = int(n_acc[b])
        for j, r in enumerate(committed_rows(N, B, tau, n)):
            k_out[int(dst_off[b]) + C + j] = k_new[q_off + r]
            v_out[int(dst_off[b]) + C + j] = v_new[q_off + r]
        new_len[b] = C + N + n
    return k_out, v_out, new_len
