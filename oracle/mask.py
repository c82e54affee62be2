"""Dense temporal attention mask of one sequence (oracle; test infrastructure).

Source: SimSD summary (Simple Speculative Decoding in Diffusion Language
Models), section 1 "Input Layout" and section 2 "Temporal Attention Mask".

Layout of one sequence, keys in this order::

    [ cache (C keys) | fresh prompt (N) | D_1 .. D_B | D~_1 .. D~_B ]

Query rows are the N fresh prompt rows followed by the 2B tail rows
(D_1..D_B, then D~_1..D~_B).  ``tau[k-1]`` is the stage of slot k, a
permutation of 1..B (the page names the map mu and labels its values tau;
this code calls the map tau).

Rules, as the page states them for mask slots:
  * D~_i may look at data token D_j when tau(j) < tau(i)  (earlier stage);
  * D~_i may look at mask slot D~_j when tau(j) >= tau(i) (current or later,
    still undecided);
  * D~_i never looks at a data token that its stage has not revealed yet.
The page is silent on the other rows; the readings used here are:
  * data token D_j looks at the whole prompt and at D_k with tau(k) <= tau(j),
    never at a mask slot;
  * fresh prompt row i (0-based) looks causally at keys 0 .. C+i, never at
    the tail;
  * every tail row looks at the whole prompt (cache and fresh rows).
"""
from __future__ import annotations

import numpy as np


def verify_mask(C: int, N: int, B: int, tau, rows=None) -> np.ndarray:
    """uint8 [N + 2B, C + N + 2B]; 1 where query row may attend key.

    ``rows`` optionally selects local query rows (the result then has one
    line per selected row, in the given order).
    """
    tau = [int(t) for t in tau]
    assert len(tau) == B and sorted(tau) == list(range(1, B + 1)), "tau must permute 1..B"
    P = C + N
    rows = list(range(N + 2 * B)) if rows is None else [int(r) for r in rows]
    A = np.zeros((len(rows), P + 2 * B), dtype=np.uint8)
    for out, row in enumerate(rows):
        if row < N:
            # fresh prompt row i = row: causal over cache + fresh prompt, never the tail
            A[out, :C + row + 1] = 1
        elif row < N + B:
            # data row D_j (slot j, 0-based): whole prompt, earlier-or-same-stage data
            j = row - N
            A[out, :P] = 1
            for k in range(B):
                if tau[k] <= tau[j]:
                    A[out, P + k] = 1
        else:
            # mask row D~_i
            i = row - N - B
            A[out, :P] = 1
            for j in range(B):
                if tau[j] < tau[i]:
                    A[out, P + j] = 1          # data token of an earlier stage
                if tau[j] >= tau[i]:
                    A[out, P + B + j] = 1      # undecided mask slot
    return A
