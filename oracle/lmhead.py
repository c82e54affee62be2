"""LM head over the mask slots fused with acceptance (oracle; test infrastructure).

Sources:
  * SimSD summary, section 4 "Speculative decoding pipeline": the target model
    scores every drafted position in one forward pass; acceptance then runs in
    the temporal order the draft induces.
  * SPOT review, section "How it is used": state equality (T = 0) and the
    coupled-noise match argmax(l / T + G[position]).

Reading (the pages give the decisions, not how the logits are formed): the
target logits of mask slot k are l_k = W h_k, with W [V, hidden] the LM head
and h_k the final hidden state of D~_k.  Here l_k is formed exactly from the
stored bf16 values (fp64 products of bf16 values are exact; the fp64 sum of
`hidden` of them is exact to about hidden * 2^-53 relative) and rounded once
to fp32; the acceptance oracle's decision rules then apply to that fp32 row
unchanged.  Only rows of verified stages (stage <= min(gamma + 1, B)) are
formed.

A device that accumulates the same products in fp32 in some order lands
within error_bound() of the exact value; decisions whose top two scores are
closer than that are ambiguous, and several answers are then correct.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import accept as oacc


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """Exact fp64 values of bf16 bit patterns."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def lm_head_logits(h: np.ndarray, w: np.ndarray) -> np.ndarray:
    """l[r, v] = sum_k h[r, k] w[v, k] in fp64 (h [rows, hidden], w [V, hidden])."""
    return np.asarray(h, np.float64) @ np.asarray(w, np.float64).T


def error_bound(h: np.ndarray, w: np.ndarray, l_exact: np.ndarray) -> np.ndarray:
    """Bound on |l_dev - fl32(l_exact)| for an fp32 accumulation of the exact
    products in any order: (hidden) u sum_k |h_k w_vk| (the standard bound for
    a sum of n terms, with u = 2^-23 so that truncating adders are covered),
    plus one fp32 rounding of each side (2^-23 |l|)."""
    K = h.shape[1]
    u = 2.0 ** -23
    absdot = np.abs(np.asarray(h, np.float64)) @ np.abs(np.asarray(w, np.float64)).T
    return K * u * absdot + u * np.abs(l_exact)


def logits_from_bits(h_bits: np.ndarray, w_bits: np.ndarray, with_bound: bool = False, block: int = 8192):
    """lm_head_logits (and error_bound) from bf16 bit patterns, one block of
    vocabulary rows at a time (bounds the fp64 temporaries for a full LM head).
    Returns (logits [rows, V], bound [rows, V] or None)."""
    hv = bf16_values(h_bits)
    rows, V = hv.shape[0], w_bits.shape[0]
    logits = np.empty((rows, V), np.float64)
    bound = np.empty((rows, V), np.float64) if with_bound else None
    for v0 in range(0, V, block):
        wv = bf16_values(w_bits[v0:v0 + block])
        logits[:, v0:v0 + block] = lm_head_logits(hv, wv)
        if with_bound:
            bound[:, v0:v0 + block] = error_bound(hv, wv, logits[:, v0:v0 + block])
    return logits, bound


def verified_slots(inp) -> np.ndarray:
    """Slots whose rows the acceptance reads: stage <= min(gamma + 1, B)."""
    out = []
    for b in range(len(inp.blocks)):
        B, g, off = int(inp.blocks[b]), int(inp.gammas[b]), int(inp.slot_off[b])
        need = min(g + 1, B)
        for k in range(B):
            if int(inp.tau[off + k]) <= need:
                out.append(off + k)
    return np.asarray(out, np.int64)


def slot_logits(x, slots=None) -> np.ndarray:
    """fp64 logits of the given slots (default: every verified slot) as a
    [len(slots), V] array, for an LmheadInputs-like x (fields acc, h, w)."""
    slots = verified_slots(x.acc) if slots is None else np.asarray(slots, np.int64)
    return logits_from_bits(x.h[slots], x.w)[0]


def accept_lmhead(x) -> dict:
    """Acceptance of an LmheadInputs-like x over logits fl32(W h_k).

    Returns the acceptance oracle's dict (n_acc, n_out, tokens, results) plus
    'slots' (the verified slots) and 'logits' (their fp64 logits)."""
    inp = x.acc
    slots = verified_slots(inp)
    l64 = slot_logits(x, slots)
    S = int(np.sum(inp.blocks))
    l32 = np.zeros((S, inp.V), np.float32)
    l32[slots] = l64.astype(np.float32)
    full = dataclasses.replace(inp, logits=l32, logits_dtype="f32", draft_logits=None)
    r = oacc.accept_batch(full)
    r["slots"] = slots
    r["logits"] = l64
    return r
