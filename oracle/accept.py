"""Acceptance step in temporal order (oracle; test infrastructure).

Sources:
  * SimSD summary, section 4 "Speculative decoding pipeline", Acceptance:
    standard rejection sampling is applied in the temporal order the draft
    induces, and the longest accepted prefix is committed.
  * SPOT review (onedev.kr), section "How it is used": verification by state
    equality (an edge is accepted only if the target's next state equals the
    drafted one, so the accepted set is one path; exact at T = 0) and, for
    T > 0, a coupled-noise match: one Gumbel noise table per absolute output
    position shared by drafter and target makes the target transition a
    deterministic function, and marginalising over the noise recovers the
    target's sampling distribution (the review's Proposition 2).

Per sequence: block width B, verified stages 1..gamma (0 <= gamma <= B),
stage map tau (slot k -> stage tau[k], a permutation of 1..B), draft token
d_k per slot, target logits row l_k of mask slot D~_k.  Stage s is slot
k = tau^{-1}(s).

Decisions (readings where the pages are silent are marked):
  ARGMAX   target decision t_k = argmax_v l_k[v]; ties -> lowest index
           (reading).  Accept stage iff d_k == t_k.
  GUMBEL   t_k = argmax_v fl32(fl32(l_k[v] / T) + G[row_k][v]), evaluated in
           IEEE fp32 round-to-nearest without contraction (reading: this fixes
           one exact value per candidate); T = 0 ignores G.  Accept iff
           d_k == t_k.  row_k is the table row the caller assigns to the
           slot's absolute output position.
  GUMBEL_GEN  as GUMBEL with G generated, not read (oracle.noise: Philox4x32-10
           at the slot's 32-bit position noise_row[k] and the call's seed,
           then -L(-L(U)) in fixed fp32 operations; a reading).
  REJECT   p = softmax(l_k / T), q = softmax(ql_k / T) (draft logits), in fp64.
           Accept iff u_k < p(d_k) / q(d_k)  (probability min(1, p/q)).
n_acc = number of leading accepted stages.  Then one target token is emitted
at stage c = n_acc + 1 if c <= B (reading): for ARGMAX/GUMBEL the decision
t at that stage; for REJECT at a rejected stage (c <= gamma) a sample of the
residual (p - q)_+ / Z, and after a fully accepted draft (c = gamma + 1 <= B)
a sample of p.  A sample from weights w (sum Z) with uniform u' is the
smallest index v with cumsum(w)[v] > u' * Z (inverse CDF, reading).  When
gamma = B and all stages are accepted nothing is emitted.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

MODE_ARGMAX = 0
MODE_GUMBEL = 1
MODE_REJECT = 2
MODE_GUMBEL_GEN = 3   # GUMBEL with the noise generated (oracle.noise) instead of read from a table


def stage_slots(tau) -> np.ndarray:
    """slot index (0-based) of each stage 1..B: inverse of the stage map."""
    tau = np.asarray(tau, dtype=np.int64)
    B = len(tau)
    assert sorted(tau.tolist()) == list(range(1, B + 1)), "tau must permute 1..B"
    inv = np.empty(B, dtype=np.int64)
    for k in range(B):
        inv[tau[k] - 1] = k
    return inv


def gumbel_scores(l32: np.ndarray, g32: np.ndarray, T: float) -> np.ndarray:
    """fl32(fl32(l / T) + G) element by element (numpy float32 ops are IEEE RN)."""
    l32 = np.asarray(l32, dtype=np.float32)
    g32 = np.asarray(g32, dtype=np.float32)
    t = np.float32(T)
    scaled = np.divide(l32, t, dtype=np.float32)
    return np.add(scaled, g32, dtype=np.float32)


def target_decision(mode: int, l32: np.ndarray, g32: Optional[np.ndarray], T: float) -> int:
    if mode == MODE_ARGMAX or T == 0.0:
        return int(np.argmax(np.asarray(l32, dtype=np.float32)))
    return int(np.argmax(gumbel_scores(l32, g32, T)))


def softmax64(logits: np.ndarray, T: float) -> np.ndarray:
    z = np.asarray(logits, dtype=np.float64) / float(np.float32(T))
    z = z - np.max(z)
    e = np.exp(z)
    return e / np.sum(e)


def inverse_cdf(w: np.ndarray, u: float):
    """Smallest v with cumsum(w)[v] > u * sum(w); returns (v, threshold, cdf)."""
    cdf = np.cumsum(np.asarray(w, dtype=np.float64))
    Z = float(cdf[-1])
    t = float(u) * Z
    v = int(np.searchsorted(cdf, t, side="right"))
    v = min(v, len(w) - 1)
    return v, t, cdf


@dataclasses.dataclass
class SeqResult:
    n_acc: int
    tokens: List[int]               # accepted drafts in stage order, then the emitted token
    emit_kind: Optional[str]        # None | "decision" | "residual" | "bonus"
    emit_slot: int                  # slot of the emitted token (-1 if none)
    accept_margins: List[float]     # |log u - log(p/q)| per tested stage (REJECT)
    sample_threshold: float = float("nan")
    sample_cdf: Optional[np.ndarray] = None

    @property
    def n_out(self) -> int:
        return len(self.tokens)


def accept_sequence(mode: int, T: float, tau, gamma: int, draft_tokens, logits_rows,
                    draft_rows=None, noise_rows=None, u_accept=None, u_sample: float = 0.0) -> SeqResult:
    """One sequence.  ``*_rows[k]`` are the rows of slot k (0-based)."""
    B = len(tau)
    assert 0 <= gamma <= B
    slots = stage_slots(tau)
    margins: List[float] = []
    n_acc = 0
    for s in range(1, gamma + 1):
        k = int(slots[s - 1])
        d = int(draft_tokens[k])
        if mode == MODE_REJECT:
            p = softmax64(logits_rows[k], T)
            q = softmax64(draft_rows[k], T)
            ratio = p[d] / q[d]
            u = float(u_accept[k])
            margins.append(abs(np.log(u) - np.log(ratio)) if u > 0 else float("inf"))
            ok = u < ratio
        else:
            g = None if noise_rows is None else noise_rows[k]
            ok = d == target_decision(mode, logits_rows[k], g, T)
        if not ok:
            break
        n_acc += 1
    tokens = [int(draft_tokens[int(slots[s - 1])]) for s in range(1, n_acc + 1)]
    c = n_acc + 1
    if c > B:
        return SeqResult(n_acc, tokens, None, -1, margins)
    k = int(slots[c - 1])
    if mode != MODE_REJECT:
        g = None if noise_rows is None else noise_rows[k]
        tokens.append(target_decision(mode, logits_rows[k], g, T))
        return SeqResult(n_acc, tokens, "decision", k, margins)
    p = softmax64(logits_rows[k], T)
    if c <= gamma:
        q = softmax64(draft_rows[k], T)
        w = np.maximum(p - q, 0.0)
        kind = "residual"
        if not np.any(w > 0):          # (p - q)_+ vanished: fall back to p
            w, kind = p, "bonus"
    else:
        w, kind = p, "bonus"
    v, t, cdf = inverse_cdf(w, u_sample)
    tokens.append(v)
    return SeqResult(n_acc, tokens, kind, k, margins, t, cdf)


def accept_batch(inp) -> dict:
    """Run ``accept_sequence`` over a packed batch (an ``AcceptInputs``-like object).

    Returns dict with int32 arrays n_acc [batch], n_out [batch],
    tokens [sum B] (stage order, -1 padded) and the per-sequence results.
    """
    from_values = _logit_values(inp, inp.logits)
    draft_values = None if inp.draft_logits is None else _logit_values(inp, inp.draft_logits)
    batch = len(inp.blocks)
    S = int(np.sum(inp.blocks))
    n_acc = np.zeros(batch, np.int32)
    n_out = np.zeros(batch, np.int32)
    tokens = np.full(S, -1, np.int32)
    results = []
    for b in range(batch):
        B, g, off = int(inp.blocks[b]), int(inp.gammas[b]), int(inp.slot_off[b])
        sl = slice(off, off + B)
        noise_rows = None
        mode = inp.mode
        if mode == MODE_GUMBEL and inp.T != 0.0:
            noise_rows = [inp.noise[int(inp.noise_row[off + k])] for k in range(B)]
        elif mode == MODE_GUMBEL_GEN:
            # each slot's noise generated at its position (the 32-bit pattern of noise_row)
            from oracle.noise import gumbel_rows
            pos = np.asarray(inp.noise_row[sl], np.int32).view(np.uint32)
            noise_rows = list(gumbel_rows(int(inp.noise_seed), pos, inp.V)) if inp.T != 0.0 else None
            mode = MODE_GUMBEL
        draft_rows = None if draft_values is None else draft_values[sl]
        r = accept_sequence(mode, inp.T, inp.tau[sl], g, inp.draft_tokens[sl], from_values[sl],
                            draft_rows, noise_rows, inp.u_accept[sl], float(inp.u_sample[b]))
        n_acc[b] = r.n_acc
        n_out[b] = r.n_out
        tokens[off:off + r.n_out] = r.tokens
        results.append(r)
    return dict(n_acc=n_acc, n_out=n_out, tokens=tokens, results=results)


def _logit_values(inp, arr) -> np.ndarray:
    """Logits as fp32 values (bf16 storage is widened exactly)."""
    if getattr(inp, "logits_dtype", "f32") == "bf16":
        return (np.asarray(arr, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    return np.asarray(arr, dtype=np.float32)


def sample_margin(res: SeqResult) -> float:
    """Distance of the sampling threshold u' Z to the nearer end of the chosen
    token's CDF interval, relative to Z: [cdf[v-1], cdf[v]) holds u' Z, so the
    inverse-CDF choice is unchanged by any perturbation of the CDF smaller
    than this."""
    cdf = res.sample_cdf
    Z = float(cdf[-1])
    v = res.tokens[-1]
    lo = 0.0 if v == 0 else float(cdf[v - 1])
    hi = float(cdf[v])
    return min(res.sample_threshold - lo, hi - res.sample_threshold) / Z
