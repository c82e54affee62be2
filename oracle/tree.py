"""Tree (state-set) verification of one block per sequence (oracle; test
infrastructure).

Sources:
  * SPOT review (onedev.kr), section "How it works": the drafter grows a tree
    of candidate block states (DDTree), each edge committing one position
    with one token; section "How it is used": verification by state
    equality -- an edge (y, z) is accepted only if z equals the next state
    the target produces from y, so the accepted set is a single path -- with
    the target's transition made deterministic at T > 0 by the shared
    per-position Gumbel noise; the review notes that packing a tree exactly
    under bidirectional attention is open, and that widening the draft costs
    (1 + D) L positions whatever is accepted.
  * SimSD summary, section 2: in a block state, the mask slot of an
    undecided position sees the committed data tokens and the undecided mask
    slots, never an undecided data token.

Readings (the pages give no layout or rule for these):
  Tree of one sequence: E edges; edge e commits position pos[e] (0..B-1,
  undecided in its parent's state) with token token[e]; parent[e] is the
  edge leading to its parent node (-1: the root, the block state before the
  pass), parent[e] < e.  Node 0 is the root, node e + 1 the child of edge e;
  committed(n) are the positions of the edges on the path root -> n.
  Query rows: the N fresh prompt rows, then one mask-slot row M_p per
  position p (its query does not depend on the state).
  Keys: [cache (C) | fresh prompt (N) | edge data rows X_0..X_{E-1} | mask rows M_0..M_{B-1}].
  Output rows: the N fresh prompt rows (causal over cache and fresh prompt,
  as in the verification pass), then node-major (n, p) for n = 0..E,
  p = 0..B-1: row (n, p), for p undecided at n, is query M_p attending the
  whole prompt, the data rows of the edges on the path root -> n and the
  mask rows of the positions undecided at n (SimSD's rule for the state of
  n; a chain of edges in stage order gives back SimSD's mask rows exactly).
  Rows (n, p) with p committed at n are not defined.
  Acceptance: from the logits of row (n, p), the decision token dec(n, p)
  (argmax of l, or of fl(fl(l/T) + G) with the coupled noise of position p)
  and its confidence c(n, p) = l[dec] - logsumexp(l) (log-probability under
  softmax(l)); the target's transition from n commits p* = the undecided
  position of largest confidence (ties: lowest p) with token dec(n, p*).
  Walk from the root: while n has an undecided position, the child edge
  with (pos, token) = (p*, dec(n, p*)) (the lowest such edge) is accepted and
  becomes n; otherwise that transition is emitted and the walk stops.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

from .attention import masked_softmax_attention
from . import accept as oacc


def tree_nodes(B: int, parent, pos):
    """Per node n = 0..E: (committed position bitmask, list of path edges).
    Raises ValueError for an invalid tree."""
    E = len(parent)
    committed = [0]
    path: List[List[int]] = [[]]
    for e in range(E):
        par = int(parent[e])
        p = int(pos[e])
        if not (-1 <= par < e) or not (0 <= p < B):
            raise ValueError("invalid edge")
        base = committed[par + 1]
        if (base >> p) & 1:
            raise ValueError("edge commits a position already committed")
        committed.append(base | (1 << p))
        path.append(path[par + 1] + [e])
    return committed, path


def tree_mask(C: int, N: int, B: int, parent, pos) -> tuple:
    """uint8 [N + (E+1) B, C + N + E + B] allowed matrix and bool [rows]
    telling which output rows are defined."""
    E = len(parent)
    committed, path = tree_nodes(B, parent, pos)
    P = C + N
    rows = N + (E + 1) * B
    A = np.zeros((rows, P + E + B), np.uint8)
    defined = np.zeros(rows, bool)
    for i in range(N):                       # fresh prompt rows: causal
        A[i, :C + i + 1] = 1
        defined[i] = True
    for n in range(E + 1):
        for p in range(B):
            r = N + n * B + p
            if (committed[n] >> p) & 1:
                continue
            defined[r] = True
            A[r, :P] = 1
            for e in path[n]:
                A[r, P + e] = 1              # committed data token on the path
            for j in range(B):
                if not (committed[n] >> j) & 1:
                    A[r, P + E + j] = 1      # undecided mask slot
    return A, defined


# sequence record of a tree batch (fields of ssv_tree_seq in include/ssv.h)
TREE_FIELDS = ("cache_len", "new_len", "block", "n_edges", "q_off", "k_off", "kv_off", "edge_off", "o_off")


def tree_attention(seqs, parent_all, pos_all, q, k_cache, v_cache, k_new, v_new, scale=None) -> np.ndarray:
    """Output [total_out_rows, Hq, d] float64 (NaN on undefined rows).
    seqs: int [batch, 9] (TREE_FIELDS); q rows per sequence: N + B at q_off;
    k_new / v_new rows: N + E + B at k_off; outputs N + (E+1) B at o_off."""
    seqs = np.asarray(seqs)
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k_new.shape[1]
    G = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    total = int(max((s[8] + s[1] + (s[3] + 1) * s[2]) for s in seqs)) if len(seqs) else 0
    out = np.full((total, Hq, d), np.nan)
    for s in seqs:
        C, N, B, E, q_off, k_off, kv_off, e_off, o_off = (int(x) for x in s)
        parent = parent_all[e_off:e_off + E]
        pos = pos_all[e_off:e_off + E]
        A, defined = tree_mask(C, N, B, parent, pos)
        # query of each output row: fresh row i, or mask slot p for row (n, p)
        qsel = np.concatenate([np.arange(N), N + np.tile(np.arange(B), E + 1)]).astype(np.int64)
        rows = np.nonzero(defined)[0]
        for h in range(Hq):
            g = h // G
            keys = np.concatenate([k_cache[kv_off:kv_off + C, g], k_new[k_off:k_off + N + E + B, g]])
            vals = np.concatenate([v_cache[kv_off:kv_off + C, g], v_new[k_off:k_off + N + E + B, g]])
            out[o_off + rows, h] = masked_softmax_attention(q[q_off + qsel[rows], h], keys, vals, A[rows], scale)
    return out


@dataclasses.dataclass
class TreeResult:
    n_acc: int
    path: List[int]                  # accepted edges, root first
    emit_pos: int                    # -1 when nothing is emitted
    emit_tok: int
    gaps: List[float]                # per visited node with >= 2 undecided positions: best - second confidence


def row_decision(mode: int, l32: np.ndarray, g32: Optional[np.ndarray], T: float):
    """(decision token, confidence l[dec] - logsumexp(l) in fp64)."""
    dec = oacc.target_decision(mode, l32, g32, T)
    l64 = np.asarray(l32, np.float64)
    m = float(np.max(l64))
    lse = m + float(np.log(np.sum(np.exp(l64 - m))))
    return dec, float(l64[dec]) - lse


def tree_accept_sequence(mode, T, B, parent, pos, token, logits_rows, noise_rows=None) -> TreeResult:
    """logits_rows[n * B + p]: logits of row (n, p) (fp32 values); noise_rows[p]:
    the Gumbel row of position p (coupled noise), else None."""
    E = len(parent)
    committed, _ = tree_nodes(B, parent, pos)
    n, acc, path, gaps = 0, 0, [], []
    while True:
        und = [p for p in range(B) if not (committed[n] >> p) & 1]
        if not und:
            return TreeResult(acc, path, -1, -1, gaps)
        dc = [row_decision(mode, logits_rows[n * B + p], None if noise_rows is None else noise_rows[p], T) for p in und]
        conf = [c for _, c in dc]
        order = sorted(range(len(und)), key=lambda i: (-conf[i], und[i]))
        best = order[0]
        if len(order) > 1:
            gaps.append(conf[order[0]] - conf[order[1]])
        p_star, v_star = und[best], int(dc[best][0])
        child = [e for e in range(E) if int(parent[e]) + 1 == n and int(pos[e]) == p_star and int(token[e]) == v_star]
        if not child:
            return TreeResult(acc, path, p_star, v_star, gaps)
        e = child[0]
        path.append(e)
        acc += 1
        n = e + 1


def tree_accept_batch(mode, T, seqs, parent_all, pos_all, token_all, logits, noise=None, noise_row=None,
                      pos_off=None) -> List[TreeResult]:
    """seqs: TREE_FIELDS records; logits [rows, V] with row (n, p) of sequence b
    at o_off + N + n B + p (the output-row numbering of tree_attention);
    coupled noise: noise[noise_row[pos_off[b] + p]] for position p."""
    res = []
    for b, s in enumerate(np.asarray(seqs)):
        C, N, B, E, q_off, k_off, kv_off, e_off, o_off = (int(x) for x in s)
        rows = [np.asarray(logits[o_off + N + r], np.float32) for r in range((E + 1) * B)]
        nrows = None
        if noise is not None and T != 0.0:
            nrows = [noise[int(noise_row[int(pos_off[b]) + p])] for p in range(B)]
        res.append(tree_accept_sequence(mode, T, B, parent_all[e_off:e_off + E], pos_all[e_off:e_off + E],
                                        token_all[e_off:e_off + E], rows, nrows))
    return res
