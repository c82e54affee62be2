"""Pins of the fused LM head + acceptance oracle (SimSD summary, section 4;
SPOT review, "How it is used"; reading: the logits of mask slot k are
l_k = W h_k, formed exactly and rounded once to fp32)."""
import dataclasses
import math

import numpy as np
import pytest

import oracle.accept as A
import oracle.lmhead as L
from diffusion_speculative_verification_gb300 import workloads as W
from golden_io import read_fixture

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


class _X:
    """An LmheadInputs-like record built from plain values."""

    def __init__(self, acc, h_vals, w_vals):
        self.acc = acc
        self.h = W.f32_to_bf16_bits(np.asarray(h_vals, np.float32))
        self.w = W.f32_to_bf16_bits(np.asarray(w_vals, np.float32))
        self.hidden = self.h.shape[1]


def _acc(mode, T, V, blocks, gammas, tau, draft, noise=None, noise_row=None):
    blocks = np.asarray(blocks, np.int32)
    S = int(blocks.sum())
    slot_off = np.concatenate([[0], np.cumsum(blocks)[:-1]]).astype(np.int32)
    return W.AcceptInputs("pin", mode, float(T), V, "f32", blocks, np.asarray(gammas, np.int32), slot_off,
                          np.asarray(tau, np.int32), None, None, np.asarray(draft, np.int32), noise,
                          np.zeros(S, np.int32) if noise_row is None else np.asarray(noise_row, np.int32),
                          np.zeros(S, np.float32), np.zeros(len(blocks), np.float32))


def test_hand_worked_example():
    meta, rows = read_fixture("lmhead_V3_H2_B2_tau21.txt")
    V, B = meta["V"], meta["B"]
    acc = _acc(A.MODE_ARGMAX, 0.0, V, [B], [meta["gamma"]], meta["tau"], meta["draft"])
    x = _X(acc, rows[V:V + B], rows[:V])
    r = L.accept_lmhead(x)
    assert int(r["n_acc"][0]) == meta["nacc"]
    assert r["tokens"][:int(r["n_out"][0])].tolist() == list(meta["tokens"])


def test_logits_brute_force():
    """Each logit equals the dot product of its hidden row with the token's
    LM-head row, summed exactly (math.fsum) from the bf16 values."""
    rng = np.random.default_rng(0)
    h = W.f32_to_bf16_bits(rng.standard_normal((3, 7)).astype(np.float32))
    w = W.f32_to_bf16_bits(rng.standard_normal((5, 7)).astype(np.float32))
    hv, wv = L.bf16_values(h), L.bf16_values(w)
    got = L.lm_head_logits(hv, wv)
    for r in range(3):
        for v in range(5):
            want = math.fsum(float(hv[r, k]) * float(wv[v, k]) for k in range(7))
            assert got[r, v] == pytest.approx(want, rel=1e-15, abs=1e-300)


def test_planted_token_wins_every_position():
    """h aligned with LM-head row t makes t the decision, for every t; a
    transposed or mis-indexed product would not."""
    rng = np.random.default_rng(1)
    V, H = 9, 16
    w = rng.standard_normal((V, H)).astype(np.float32)
    wv = L.bf16_values(W.f32_to_bf16_bits(w))
    for t in range(V):
        h = 0.05 * rng.standard_normal(H) + 4.0 * wv[t] / H
        acc = _acc(A.MODE_ARGMAX, 0.0, V, [1], [0], [1], [0])
        x = _X(acc, h[None, :], w)
        r = L.accept_lmhead(x)
        assert r["tokens"][0] == t


def test_identity_head_reduces_to_plain_acceptance():
    """With W = I (V = hidden) the logits are the hidden rows themselves: the
    outcome equals the acceptance oracle on those rows as logits."""
    rng = np.random.default_rng(2)
    V = 24
    blocks, gammas = [5, 3, 4], [5, 2, 1]
    S = sum(blocks)
    tau = np.concatenate([W.random_tau(rng, b) for b in blocks])
    h = W.f32_to_bf16_bits(rng.standard_normal((S, V)).astype(np.float32))
    hv = L.bf16_values(h).astype(np.float32)
    draft = np.argmax(hv, axis=1).astype(np.int32)
    draft[rng.random(S) < 0.3] = 0
    for mode, T in ((A.MODE_ARGMAX, 0.0), (A.MODE_GUMBEL, 1.5)):
        noise = W.gumbel_table(rng, S, V)
        acc = _acc(mode, T, V, blocks, gammas, tau, draft, noise=noise, noise_row=np.arange(S)[::-1])
        x = _X(acc, L.bf16_values(h), np.eye(V))
        got = L.accept_lmhead(x)
        plain = A.accept_batch(dataclasses.replace(acc, logits=hv, logits_dtype="f32"))
        assert got["n_acc"].tolist() == plain["n_acc"].tolist()
        assert got["tokens"].tolist() == plain["tokens"].tolist()


def test_vocabulary_permutation_equivariance():
    """Permuting the LM-head rows permutes every decision the same way."""
    rng = np.random.default_rng(3)
    V, H, S = 40, 12, 6
    w = rng.standard_normal((V, H)).astype(np.float32)
    h = rng.standard_normal((S, H)).astype(np.float32)
    perm = rng.permutation(V)
    acc = _acc(A.MODE_ARGMAX, 0.0, V, [1] * S, [0] * S, [1] * S, [0] * S)
    a = L.accept_lmhead(_X(acc, h, w))["tokens"]
    b = L.accept_lmhead(_X(acc, h, w[perm]))["tokens"]
    assert [int(perm[t]) for t in b] == a.tolist()


def test_zero_noise_gumbel_equals_argmax():
    """Coupled noise with an all-zero table at T = 1 is the greedy rule."""
    rng = np.random.default_rng(4)
    V, H = 50, 8
    blocks = [4, 4]
    tau = np.concatenate([W.random_tau(rng, 4), W.random_tau(rng, 4)])
    w = rng.standard_normal((V, H)).astype(np.float32)
    h = rng.standard_normal((8, H)).astype(np.float32)
    draft = rng.integers(0, V, 8).astype(np.int32)
    g = L.accept_lmhead(_X(_acc(A.MODE_GUMBEL, 1.0, V, blocks, [3, 4], tau, draft,
                                noise=np.zeros((8, V), np.float32)), h, w))
    a = L.accept_lmhead(_X(_acc(A.MODE_ARGMAX, 0.0, V, blocks, [3, 4], tau, draft), h, w))
    assert g["tokens"].tolist() == a["tokens"].tolist()


def test_verified_slots():
    """Rows of stages 1..min(gamma + 1, B) are formed, nothing else."""
    acc = _acc(A.MODE_ARGMAX, 0.0, 4, [3, 2, 4], [1, 2, 0], [3, 1, 2, 2, 1, 4, 1, 2, 3], [0] * 9)
    assert L.verified_slots(acc).tolist() == [1, 2, 3, 4, 6]


def test_error_bound_covers_fp32_accumulation():
    """An fp32 accumulation (sequential, and numpy's blocked fp32 product) of
    the exact products stays inside error_bound; so does one with a
    truncating adder simulated by rounding toward zero at every step."""
    rng = np.random.default_rng(5)
    H, V = 512, 64
    h = L.bf16_values(W.f32_to_bf16_bits(rng.standard_normal((2, H)).astype(np.float32) / np.sqrt(H)))
    w = L.bf16_values(W.f32_to_bf16_bits(rng.standard_normal((V, H)).astype(np.float32)))
    exact = L.lm_head_logits(h, w)
    bound = L.error_bound(h, w, exact)
    blas = (h.astype(np.float32) @ w.astype(np.float32).T).astype(np.float64)
    assert np.all(np.abs(blas - exact.astype(np.float32)) <= bound)
    for r in range(2):
        for v in range(0, V, 7):
            acc_rn = np.float32(0.0)
            acc_tz = 0.0
            for k in range(H):
                p = np.float32(h[r, k] * w[v, k])  # bf16 x bf16 is exact in fp32
                acc_rn = np.float32(acc_rn + p)
                s = acc_tz + float(p)
                t = float(np.float32(s))
                if abs(t) > abs(s):
                    t = float(np.nextafter(np.float32(t), np.float32(0.0)))
                acc_tz = t
            e32 = float(np.float32(exact[r, v]))
            assert abs(float(acc_rn) - e32) <= bound[r, v]
            assert abs(acc_tz - e32) <= bound[r, v]


def test_generator_plants_the_cut():
    """With the generator's planting, accepted stages are exactly those before
    each sequence's cut: the oracle accepts every planted draft, rejects the
    cut stage and emits the token planted there."""
    x = W.make_lmhead_inputs("p", A.MODE_ARGMAX, 0.0, 300, 64, [4, 6, 1, 8], [4, 3, 0, 8], 6)
    r = L.accept_lmhead(x)
    S = int(np.sum(x.acc.blocks))
    l32 = np.zeros((S, 300), np.float32)
    l32[r["slots"]] = r["logits"].astype(np.float32)
    for b, res in enumerate(r["results"]):
        B, g, off = int(x.acc.blocks[b]), int(x.acc.gammas[b]), int(x.acc.slot_off[b])
        slots = A.stage_slots(x.acc.tau[off:off + B]) + off
        for s in range(res.n_acc):
            k = slots[s]
            assert np.argmax(l32[k]) == x.acc.draft_tokens[k]
            assert l32[k].max() > 30.0
        if res.n_acc < B:
            k = slots[res.n_acc]
            assert res.tokens[-1] == int(np.argmax(l32[k]))
