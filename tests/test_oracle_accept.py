"""Pins for oracle.accept (CPU only).

* Coupled noise, SPOT review "How it is used" (Proposition 2): over many
  Gumbel tables the law of argmax(l/T + G) is softmax(l/T); checked by a
  chi-square test at V = 4.
* Coupling: a drafter that shares the noise table and the model is always
  accepted; one with independent noise is accepted about sum_v p_v^2 of the
  time (the collapse the review reports for uncoupled sampling).
* Rejection sampling, SimSD summary section 4: the law of the emitted token
  is p, computed by integrating the oracle's own decisions over a fine grid
  of uniforms (brute force at V <= 5), at T = 0.7, 1 and 1.3 against the
  library softmax; the oracle's softmax(l / T) against the logistic closed
  form at V = 2 and the library routine.
* Longest accepted prefix in temporal (tau) order, emission rules.
"""
import numpy as np
import pytest

from oracle import accept as A
from diffusion_speculative_verification_gb300 import workloads as W


def softmax_ref(l, T):
    """softmax(l / T) by scipy (a library routine the oracle does not use),
    with T taken as the fp32 value the acceptance call receives."""
    from scipy.special import softmax
    return softmax(np.asarray(l, np.float64) / float(np.float32(T)))


@pytest.mark.parametrize("T", [0.7, 1.0, 1.3, 2.5])
def test_softmax64_two_tokens_closed_form(T):
    """V = 2: p_0 = 1 / (1 + e^((l_1 - l_0) / T)) exactly (the logistic
    function), so a mistake in how the oracle applies T fails here."""
    import math
    rng = np.random.default_rng(int(T * 100))
    T32 = float(np.float32(T))
    for _ in range(50):
        l = rng.standard_normal(2) * 3.0
        p = A.softmax64(l, T)
        p0 = 1.0 / (1.0 + math.exp((l[1] - l[0]) / T32))
        assert abs(p[0] - p0) < 4e-16 and abs(p[1] - (1.0 - p0)) < 4e-16
    # a temperature that is not applied (T taken as 1) is far off at T != 1
    if T != 1.0:
        l = np.array([0.0, 1.0])
        assert abs(A.softmax64(l, T)[0] - 1.0 / (1.0 + math.e)) > 1e-2


@pytest.mark.parametrize("T", [0.7, 1.3])
def test_softmax64_matches_library(T):
    rng = np.random.default_rng(int(T * 10))
    l = rng.standard_normal(7) * 2.0
    np.testing.assert_allclose(A.softmax64(l, T), softmax_ref(l, T), rtol=1e-14, atol=0)


@pytest.mark.parametrize("T", [0.5, 1.0, 1.5])
def test_gumbel_max_law(T):
    rng = np.random.default_rng(int(T * 10))
    l = np.array([0.3, -1.2, 1.1, 0.0], np.float32)
    n = 1_000_000
    G = (-np.log(-np.log(W.open_uniform(rng, (n, 4))))).astype(np.float32)
    scores = A.gumbel_scores(l[None, :], G, T)
    counts = np.bincount(np.argmax(scores, axis=1), minlength=4)
    p = softmax_ref(l, T)
    chi2 = float(np.sum((counts - n * p) ** 2 / (n * p)))
    assert chi2 < 16.27                               # chi2(3) 0.999 quantile
    sigma = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(counts / n - p) < 4.5 * sigma)
    # the per-row decision agrees with the vectorised scores
    for r in range(200):
        assert A.target_decision(A.MODE_GUMBEL, l, G[r], T) == int(np.argmax(scores[r]))


def test_gumbel_T0_is_argmax_and_ties_lowest_index():
    l = np.array([1.0, 3.0, 3.0, -2.0], np.float32)
    g = np.array([50.0, 0.0, 0.0, 0.0], np.float32)
    assert A.target_decision(A.MODE_GUMBEL, l, g, 0.0) == 1
    assert A.target_decision(A.MODE_ARGMAX, l, None, 0.0) == 1
    assert A.target_decision(A.MODE_GUMBEL, np.zeros(5, np.float32), np.zeros(5, np.float32), 1.0) == 0


def test_gumbel_score_is_fp32_rounded():
    # l/T is rounded to fp32 before G is added: choose values where that matters
    l = np.array([1.0, 1.0000001], np.float32)
    s = A.gumbel_scores(l, np.zeros(2, np.float32), 3.0)
    assert s.dtype == np.float32
    assert s[0] == np.float32(np.float32(1.0) / np.float32(3.0))


def _seq(mode, T, tau, gamma, drafts, rows, **kw):
    return A.accept_sequence(mode, T, tau, gamma, drafts, rows, **kw)


@pytest.mark.parametrize("T", [1.0, 1.5])
def test_coupling_shared_noise_always_accepted(T):
    rng = np.random.default_rng(7)
    B, V = 6, 50
    tau = rng.permutation(B) + 1
    accepted_uncoupled = []
    for trial in range(300):
        l = rng.standard_normal((B, V)).astype(np.float32) * 2
        G = (-np.log(-np.log(W.open_uniform(rng, (B, V))))).astype(np.float32)
        G2 = (-np.log(-np.log(W.open_uniform(rng, (B, V))))).astype(np.float32)
        # drafter with the same model and the same noise table
        drafts = np.array([int(np.argmax(np.float32(l[k] / np.float32(T)) + G[k])) for k in range(B)])
        r = _seq(A.MODE_GUMBEL, T, tau, B, drafts, l, noise_rows=G)
        assert r.n_acc == B and r.n_out == B and r.emit_kind is None
        # drafter with independent noise
        drafts2 = np.array([int(np.argmax(np.float32(l[k] / np.float32(T)) + G2[k])) for k in range(B)])
        r2 = _seq(A.MODE_GUMBEL, T, tau, 1, drafts2, l, noise_rows=G)
        accepted_uncoupled.append(r2.n_acc)
    # one stage accepted with probability sum_v p_v^2 (averaged over the logits draws): far below 1
    assert np.mean(accepted_uncoupled) < 0.5


@pytest.mark.parametrize("V,seed,T", [(2, 0, 1.0), (3, 1, 1.0), (4, 2, 1.0), (5, 3, 1.0), (2, 4, 0.7), (4, 5, 0.7),
                                       (3, 6, 1.3), (5, 7, 1.3)])
def test_rejection_law_is_p(V, seed, T):
    """Drafts drawn from q, accepted with probability min(1, p/q), residual
    samples of (p - q)_+ at a rejection: the emitted token's law is p =
    softmax(l / T), by integrating the oracle's own decisions over a grid of
    uniforms.  p and q here come from the library softmax."""
    rng = np.random.default_rng(seed)
    l = rng.standard_normal(V) * 1.5
    ql = l + rng.standard_normal(V) * 0.8
    p = softmax_ref(l, T)
    q = softmax_ref(ql, T)
    M = 2000
    grid = (np.arange(M) + 0.5) / M
    law = np.zeros(V)
    for dtok in range(V):
        acc = 0
        for u in grid:
            r = _seq(A.MODE_REJECT, T, [1], 1, [dtok], l[None, :], draft_rows=ql[None, :],
                     u_accept=[u], u_sample=0.5)
            acc += r.n_acc
        a = acc / M
        law[dtok] += q[dtok] * a
        if a < 1.0:
            samp = np.zeros(V)
            # force a rejection (u just below 1 exceeds any ratio < 1) and sweep u'
            for u2 in grid:
                r = _seq(A.MODE_REJECT, T, [1], 1, [dtok], l[None, :], draft_rows=ql[None, :],
                         u_accept=[1 - 1e-12], u_sample=u2)
                assert r.n_acc == 0 and r.emit_kind == "residual"
                samp[r.tokens[-1]] += 1.0 / M
            law += q[dtok] * (1 - a) * samp
    np.testing.assert_allclose(law, p, atol=3.0 / M, rtol=0)


@pytest.mark.parametrize("T", [1.0, 0.7, 1.3])
def test_bonus_law_is_p(T):
    rng = np.random.default_rng(5)
    l = rng.standard_normal(4)
    M = 4000
    grid = (np.arange(M) + 0.5) / M
    counts = np.zeros(4)
    for u2 in grid:
        # gamma = 0 < B = 1: nothing to verify, sample the bonus from p
        r = _seq(A.MODE_REJECT, T, [1], 0, [0], l[None, :], draft_rows=l[None, :], u_accept=[0.0], u_sample=u2)
        assert r.emit_kind == "bonus" and r.n_acc == 0
        counts[r.tokens[0]] += 1
    np.testing.assert_allclose(counts / M, softmax_ref(l, T), atol=2.0 / M)


def test_identical_draft_always_accepted():
    rng = np.random.default_rng(6)
    B, V = 5, 30
    l = rng.standard_normal((B, V))
    tau = rng.permutation(B) + 1
    drafts = rng.integers(0, V, B)
    r = _seq(A.MODE_REJECT, 1.0, tau, 3, drafts, l, draft_rows=l.copy(), u_accept=np.full(B, 0.999), u_sample=0.3)
    assert r.n_acc == 3 and r.emit_kind == "bonus"
    assert r.tokens[:3] == [int(drafts[np.where(tau == s)[0][0]]) for s in (1, 2, 3)]


@pytest.mark.parametrize("mode", [A.MODE_ARGMAX, A.MODE_GUMBEL])
def test_planted_mismatch_in_tau_order(mode):
    rng = np.random.default_rng(8)
    B, V, T = 8, 40, 1.0
    tau = np.array([5, 2, 8, 1, 7, 3, 6, 4])
    slots = A.stage_slots(tau)
    l = rng.standard_normal((B, V)).astype(np.float32)
    G = (-np.log(-np.log(W.open_uniform(rng, (B, V))))).astype(np.float32)
    Tm = 0.0 if mode == A.MODE_ARGMAX else T
    target = np.array([A.target_decision(mode, l[k], G[k], Tm) for k in range(B)])
    for cut in range(1, B + 2):
        drafts = target.copy()
        if cut <= B:
            k = slots[cut - 1]
            drafts[k] = (target[k] + 1) % V
        r = _seq(mode, Tm, tau, B, drafts, l, noise_rows=G)
        assert r.n_acc == min(cut - 1, B)
        assert r.tokens[:r.n_acc] == [int(target[slots[s]]) for s in range(r.n_acc)]
        if cut <= B:
            assert r.emit_kind == "decision" and r.tokens[-1] == int(target[slots[cut - 1]])
            assert r.emit_slot == slots[cut - 1]
        else:
            assert r.emit_kind is None and r.n_out == B
    # slot order is irrelevant: a mismatch at the slot of stage 1 rejects everything
    drafts = target.copy()
    drafts[slots[0]] = (target[slots[0]] + 1) % V
    assert _seq(mode, Tm, tau, B, drafts, l, noise_rows=G).n_acc == 0


def test_gamma_zero_and_bonus_stage():
    rng = np.random.default_rng(9)
    B, V = 4, 20
    l = rng.standard_normal((B, V)).astype(np.float32)
    tau = np.array([2, 4, 1, 3])
    r = _seq(A.MODE_ARGMAX, 0.0, tau, 0, np.zeros(B, int), l)
    assert r.n_acc == 0 and r.n_out == 1 and r.emit_slot == 2 and r.tokens[0] == int(np.argmax(l[2]))
    drafts = np.array([int(np.argmax(l[k])) for k in range(B)])
    r = _seq(A.MODE_ARGMAX, 0.0, tau, 2, drafts, l)
    assert r.n_acc == 2 and r.emit_slot == 3 and r.emit_kind == "decision"


def test_batch_matches_per_sequence():
    inp = W.make_accept_inputs("t", W.MODE_GUMBEL, 1.0, 64, [4, 8, 1, 3], [4, 5, 1, 0], seed=3)
    out = A.accept_batch(inp)
    for b in range(4):
        off, B = inp.slot_off[b], inp.blocks[b]
        rows = [inp.noise[inp.noise_row[off + k]] for k in range(B)]
        r = A.accept_sequence(inp.mode, inp.T, inp.tau[off:off + B], int(inp.gammas[b]),
                              inp.draft_tokens[off:off + B], inp.logits[off:off + B], noise_rows=rows)
        assert out["n_acc"][b] == r.n_acc and out["tokens"][off:off + r.n_out].tolist() == r.tokens
    # planted agreement: accepted lengths are not all zero
    inp = W.make_accept_inputs("t", W.MODE_ARGMAX, 0.0, 64, [8] * 16, [8] * 16, seed=4)
    assert A.accept_batch(inp)["n_acc"].max() > 0


def test_sample_margin_rule():
    w = np.array([0.0, 0.25, 0.25, 0.5])
    v, t, cdf = A.inverse_cdf(w, 0.55)
    assert v == 3                      # cdf = [0, .25, .5, 1]: first entry strictly above 0.55
    res = A.SeqResult(0, [v], "residual", 0, [], t, cdf)
    assert abs(A.sample_margin(res) - 0.05) < 1e-15      # 0.55 is 0.05 above the boundary at 0.5
    v, t, cdf = A.inverse_cdf(w, 0.3)
    res = A.SeqResult(0, [v], "bonus", 0, [], t, cdf)
    assert v == 2 and abs(A.sample_margin(res) - 0.05) < 1e-15
    v, t, cdf = A.inverse_cdf(w, 0.0)  # the first token of positive mass; t sits on its lower end
    assert v == 1 and A.sample_margin(A.SeqResult(0, [v], "bonus", 0, [], t, cdf)) == 0.0


@pytest.mark.parametrize("T", [1.0, 1.5])
def test_generated_noise_coupling(T):
    """Generated coupled noise (SPOT review, "How it is used"): a drafter that
    evaluates the same generator at the same positions, with the same model,
    is always accepted; the batch oracle reads each slot's noise at its
    position."""
    from oracle.noise import gumbel_rows
    inp = W.make_accept_inputs("gen", W.MODE_GUMBEL_GEN, T, 300, [6, 3], [6, 3], seed=21)
    pos = inp.noise_row.view(np.uint32)
    G = gumbel_rows(inp.noise_seed, pos, inp.V)
    l = inp.logits.astype(np.float32)
    inp.draft_tokens = np.array([int(np.argmax(A.gumbel_scores(l[k], G[k], T))) for k in range(len(pos))], np.int32)
    out = A.accept_batch(inp)
    assert out["n_acc"].tolist() == [6, 3] and out["n_out"].tolist() == [6, 3]
    # one changed draft at the slot of stage 1 rejects everything from there
    k0 = int(np.argmin(inp.tau[:6]))
    inp.draft_tokens[k0] = (inp.draft_tokens[k0] + 1) % inp.V
    out = A.accept_batch(inp)
    assert out["n_acc"][0] == 0 and out["tokens"][0] == int(np.argmax(A.gumbel_scores(l[k0], G[k0], T)))
