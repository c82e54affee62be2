"""Pins for oracle.tree, tree (state-set) verification (CPU only).

SPOT review, "How it works" / "How it is used": a draft tree of block
states, verified by state equality (the accepted set is one path); SimSD
summary section 2 for the mask of a block state.

* Mask: hand-worked fixture (tests/golden/tree_mask_C1_N1_B3_E3.txt);
  counting invariant (each defined tree row sees exactly C + N + B keys).
* A chain of edges in stage order is SimSD's layout: its rows equal SimSD's
  mask rows computed by the independently pinned verification oracle.
* Each defined row equals unmasked scaled-dot-product attention (torch,
  fp64, a library routine) over the prompt, its path's data rows and its
  undecided mask rows.
* Acceptance: a hand-worked walk; ties in confidence go to the lowest
  position and duplicate edges to the lowest edge; a fully committed node
  emits nothing; the planted inputs' path is what the walk accepts.
"""
import numpy as np
import pytest

from oracle import tree as TR
from oracle import accept as oacc
from oracle.attention import verify_attention
from golden_io import read_fixture
from diffusion_speculative_verification_gb300 import workloads as W


def test_mask_fixture():
    meta, rows = read_fixture("tree_mask_C1_N1_B3_E3.txt")
    A, defined = TR.tree_mask(meta["C"], meta["N"], meta["B"], meta["parent"], meta["pos"])
    np.testing.assert_array_equal(A, rows[:, 1:])
    np.testing.assert_array_equal(defined, rows[:, 0].astype(bool))


def test_invalid_trees_rejected():
    with pytest.raises(ValueError):
        TR.tree_nodes(3, [-1, 0], [1, 1])          # commits a committed position
    with pytest.raises(ValueError):
        TR.tree_nodes(3, [0], [1])                 # parent not earlier
    with pytest.raises(ValueError):
        TR.tree_nodes(3, [-1], [3])                # position outside the block


@pytest.mark.parametrize("seed", range(4))
def test_counting_invariant(seed):
    rng = np.random.default_rng(seed)
    B, E, C, N = int(rng.integers(1, 12)), int(rng.integers(0, 20)), int(rng.integers(0, 9)), int(rng.integers(0, 5))
    parent, pos = W.random_tree(rng, B, E)
    A, defined = TR.tree_mask(C, N, B, parent, pos)
    committed, path = TR.tree_nodes(B, parent, pos)
    for n in range(E + 1):
        for p in range(B):
            r = N + n * B + p
            assert defined[r] == (not (committed[n] >> p) & 1)
            if defined[r]:
                assert A[r].sum() == C + N + B
                assert A[r, C + N:C + N + E].sum() == len(path[n])


@pytest.mark.parametrize("B,gamma", [(4, 4), (6, 3), (1, 1)])
def test_chain_is_simsd(B, gamma):
    """Edges e = 0..gamma-1 commit the slots of stages 1..gamma in order; the
    edge data rows carry D of those slots, the mask rows D~: the row of the
    node at depth d for the slot of stage d + 1 equals SimSD's D~ row."""
    rng = np.random.default_rng(B * 10 + gamma)
    C, N, H, d = 7, 2, 2, 16
    a = W.make_attn_inputs("c", [C], [N], [B], H, H, d, W.F32, seed=B + gamma)
    tau = a.tau
    slots = np.empty(B, np.int64)
    slots[tau - 1] = np.arange(B)
    q = rng.standard_normal((N + 2 * B, H, d))
    kn = rng.standard_normal((N + 2 * B, H, d))
    vn = rng.standard_normal((N + 2 * B, H, d))
    kc = rng.standard_normal((C, H, d))
    vc = rng.standard_normal((C, H, d))
    simsd = verify_attention(a.seqs, tau, q, kc, vc, kn, vn)
    parent = np.arange(-1, gamma - 1, dtype=np.int32)
    pos = slots[:gamma].astype(np.int32)
    # tree layout: queries [fresh | mask slots], keys [fresh | edge data rows | mask rows]
    tq = np.concatenate([q[:N], q[N + B:]])
    tk = np.concatenate([kn[:N], kn[N + pos], kn[N + B:]])
    tv = np.concatenate([vn[:N], vn[N + pos], vn[N + B:]])
    seqs = np.array([[C, N, B, gamma, 0, 0, 0, 0, 0]])
    out = TR.tree_attention(seqs, parent, pos, tq, kc, vc, tk, tv)
    for depth in range(gamma):
        p = int(slots[depth])
        np.testing.assert_allclose(out[N + depth * B + p], simsd[N + B + p], rtol=0, atol=1e-12)
    np.testing.assert_allclose(out[:N], simsd[:N], rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_rows_equal_unmasked_sdpa(seed):
    import torch
    t = W.make_tree_inputs("s", [9, 0], [2, 3], [5, 7], [6, 11], 4, 2, 32, W.F32, seed=300 + seed)
    q, kn, vn = (W.values_f64(x, t.dtype) for x in (t.q, t.k_new, t.v_new))
    kc, vc = W.values_f64(t.k_cache, t.dtype), W.values_f64(t.v_cache, t.dtype)
    out = TR.tree_attention(t.seqs, t.parent, t.pos, q, kc, vc, kn, vn)
    for s in t.seqs:
        C, N, B, E, q_off, k_off, kv_off, e_off, o_off = (int(x) for x in s)
        committed, path = TR.tree_nodes(B, t.parent[e_off:e_off + E], t.pos[e_off:e_off + E])
        for n in range(E + 1):
            for p in range(B):
                if (committed[n] >> p) & 1:
                    assert np.all(np.isnan(out[o_off + N + n * B + p]))
                    continue
                sel = list(range(C + N)) + [C + N + e for e in path[n]] + \
                    [C + N + E + j for j in range(B) if not (committed[n] >> j) & 1]
                for h in range(4):
                    g = h // 2
                    keys = np.concatenate([kc[kv_off:kv_off + C, g], kn[k_off:k_off + N + E + B, g]])[sel]
                    vals = np.concatenate([vc[kv_off:kv_off + C, g], vn[k_off:k_off + N + E + B, g]])[sel]
                    want = torch.nn.functional.scaled_dot_product_attention(
                        torch.from_numpy(q[q_off + N + p, h][None, None]), torch.from_numpy(keys[None]),
                        torch.from_numpy(vals[None]))[0, 0].numpy()
                    np.testing.assert_allclose(out[o_off + N + n * B + p, h], want, rtol=0, atol=1e-12)


def test_walk_by_hand():
    # B = 2, V = 3; e0: root commits position 0 with token 1; e1: root commits position 1 with token 2
    parent, pos, token = [-1, -1], [0, 1], [1, 2]
    rows = {(0, 0): [0, 5, 0], (0, 1): [0, 0, 3], (1, 1): [4, 0, 0], (2, 0): [0, 0, 9]}
    logits = [np.array(rows.get((n, p), [0, 0, 0]), np.float32) for n in range(3) for p in range(2)]
    r = TR.tree_accept_sequence(oacc.MODE_ARGMAX, 0.0, 2, parent, pos, token, logits)
    # root: confidences 5 - lse(0,5,0) > 3 - lse(0,0,3): commit (0, 1) = e0; node 1: (1, 0) has no edge
    assert r.n_acc == 1 and r.path == [0] and (r.emit_pos, r.emit_tok) == (1, 0)
    assert len(r.gaps) == 1 and r.gaps[0] > 0


def test_ties_and_duplicates():
    # equal confidences at the root: the lowest position wins
    logits = [np.array([0, 2, 0], np.float32), np.array([2, 0, 0], np.float32)] + [np.zeros(3, np.float32)] * 6
    r = TR.tree_accept_sequence(oacc.MODE_ARGMAX, 0.0, 2, [-1, -1, -1], [0, 0, 1], [1, 1, 0], logits)
    assert r.path[0] == 0                      # edges 0 and 1 are equal: the lower one
    assert r.gaps[0] == 0.0
    # a fully committed node emits nothing
    r = TR.tree_accept_sequence(oacc.MODE_ARGMAX, 0.0, 1, [-1], [0], [1],
                                [np.array([0, 3, 0], np.float32), np.zeros(3, np.float32)])
    assert r.n_acc == 1 and r.emit_pos == -1 and r.emit_tok == -1


def test_gumbel_decision_uses_the_positions_noise():
    logits = [np.array([1.0, 0.0], np.float32), np.array([0.0, 0.0], np.float32)]
    noise = [np.array([0.0, 5.0], np.float32)]
    r = TR.tree_accept_sequence(oacc.MODE_GUMBEL, 1.0, 1, [], [], [], logits, noise)
    assert (r.emit_pos, r.emit_tok) == (0, 1)     # the noise, not the logit, decides the token


@pytest.mark.parametrize("seed", range(4))
def test_planted_path_is_accepted(seed):
    t = W.make_tree_inputs("p", [3] * 6, [0] * 6, [8, 5, 16, 3, 8, 12], [12, 6, 30, 2, 0, 20], 2, 1, 16, W.F32,
                           seed=400 + seed, V=50)
    res = TR.tree_accept_batch(t.mode, t.T, t.seqs, t.parent, t.pos, t.token, t.logits)
    for b, r in enumerate(res):
        s = t.seqs[b]
        E, e0 = int(s[3]), int(s[7])
        committed, path = TR.tree_nodes(int(s[2]), t.parent[e0:e0 + E], t.pos[e0:e0 + E])
        want_path, want_emit = t.planted[b]
        assert r.path == want_path and r.n_acc == len(want_path)
        assert r.path == (path[r.path[-1] + 1] if r.path else [])     # a path from the root
        assert (r.emit_pos, r.emit_tok) == (want_emit if want_emit is not None else (-1, -1))
