"""Pins of the commit oracle (SimSD summary, section 4, Acceptance: the
longest accepted prefix is committed; reading: fresh prompt rows first, then
the accepted data rows in stage order, mask rows never)."""
import numpy as np
import pytest

import oracle.commit as OC
import oracle.accept as A
from diffusion_speculative_verification_gb300 import workloads as W
from golden_io import read_fixture


def _one_sequence(C, N, B, tau, n_acc, Hkv=2, d=4, seed=0, dst_extra=3):
    """Fresh rows whose values encode their own row index, mask rows set to a
    sentinel, and a destination cache whose first C rows are old contents."""
    rng = np.random.default_rng(seed)
    rows = N + 2 * B
    k_new = rng.standard_normal((rows, Hkv, d))
    v_new = rng.standard_normal((rows, Hkv, d))
    k_new[N + B:] = -1e30  # mask rows: never committed
    v_new[N + B:] = -1e30
    cap = C + N + B + dst_extra
    k_dst = rng.standard_normal((cap, Hkv, d))
    v_dst = rng.standard_normal((cap, Hkv, d))
    seqs = np.array([[C, N, B, 0, 0, 0]], dtype=np.int64)
    out = OC.commit_batch(seqs, np.asarray(tau), [n_acc], k_new, v_new, k_dst, v_dst, [0])
    return k_new, v_new, k_dst, v_dst, out


def test_hand_worked_example():
    meta, _ = read_fixture("commit_C2_N1_B3_tau231_nacc2.txt")
    rows = OC.committed_rows(meta["N"], meta["B"], meta["tau"], meta["nacc"])
    assert rows == list(meta["rows"])
    k_new, v_new, k_dst, v_dst, (k_out, v_out, new_len) = _one_sequence(
        meta["C"], meta["N"], meta["B"], meta["tau"], meta["nacc"])
    assert new_len[0] == meta["newlen"]
    for j, r in enumerate(meta["rows"]):
        assert np.array_equal(k_out[meta["C"] + j], k_new[r])
        assert np.array_equal(v_out[meta["C"] + j], v_new[r])


@pytest.mark.parametrize("B", [1, 4, 13, 64])
def test_identity_stage_map_commits_a_contiguous_prefix(B):
    for n in (0, B // 2, B):
        assert OC.committed_rows(3, B, list(range(1, B + 1)), n) == list(range(3)) + [3 + k for k in range(n)]


def test_nothing_accepted_commits_only_prompt_rows():
    assert OC.committed_rows(5, 8, [3, 1, 2, 8, 7, 6, 5, 4], 0) == [0, 1, 2, 3, 4]


@pytest.mark.parametrize("seed", range(5))
def test_all_accepted_commits_every_data_row_once_and_no_mask_row(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 65))
    tau = [int(t) for t in rng.permutation(B) + 1]
    C, N = 4, int(rng.integers(0, 6))
    k_new, _, k_dst, _, (k_out, _, new_len) = _one_sequence(C, N, B, tau, B, seed=seed)
    appended = k_out[C:C + N + B]
    assert new_len[0] == C + N + B
    assert not np.any(appended <= -1e29)  # no mask row
    # as a set of rows: the prompt rows and every data row, each once
    got = sorted(map(tuple, appended.reshape(N + B, -1)))
    want = sorted(map(tuple, k_new[:N + B].reshape(N + B, -1)))
    assert got == want
    # stage order: the j-th appended data row is the slot whose stage is j + 1
    for s in range(1, B + 1):
        assert np.array_equal(appended[N + s - 1], k_new[N + tau.index(s)])


def test_rows_outside_the_appended_range_are_untouched():
    _, _, k_dst, v_dst, (k_out, v_out, new_len) = _one_sequence(6, 2, 5, [5, 4, 3, 2, 1], 3)
    n = int(new_len[0])
    assert np.array_equal(k_out[:6], k_dst[:6]) and np.array_equal(k_out[n:], k_dst[n:])
    assert np.array_equal(v_out[:6], v_dst[:6]) and np.array_equal(v_out[n:], v_dst[n:])


def test_committed_data_rows_carry_the_accepted_tokens():
    """The draft tokens of the committed slots, in append order, are the
    acceptance oracle's accepted prefix."""
    x = W.make_accept_inputs("commit", W.MODE_ARGMAX, 0.0, 300, [8, 5, 16, 3], [8, 4, 12, 3], seed=17)
    res = A.accept_batch(x)
    assert res["n_acc"].max() > 0
    for b in range(len(x.blocks)):
        off, B = int(x.slot_off[b]), int(x.blocks[b])
        tau = [int(t) for t in x.tau[off:off + B]]
        n = int(res["n_acc"][b])
        rows = OC.committed_rows(0, B, tau, n)
        committed_tokens = [int(x.draft_tokens[off + r]) for r in rows]
        assert committed_tokens == [int(t) for t in res["tokens"][off:off + n]]
