"""Pins for oracle.mask (CPU only).

The temporal attention mask of the SimSD summary, section 2: a hand-worked
example written from the rule text, plus counting invariants that any
off-by-one in the stage comparisons (< vs <=) would break.
"""
import numpy as np
import pytest

from oracle.mask import verify_mask
from golden_io import read_fixture


def test_hand_worked_example():
    meta, expected = read_fixture("mask_C1_N1_B3_tau231.txt")
    A = verify_mask(meta["C"], meta["N"], meta["B"], meta["tau"])
    np.testing.assert_array_equal(A, expected.astype(np.uint8))


@pytest.mark.parametrize("B", [1, 2, 3, 5, 8, 16, 32, 64])
def test_counting_invariants(B):
    rng = np.random.default_rng(B)
    for trial in range(5):
        tau = rng.permutation(B) + 1
        C, N = int(rng.integers(0, 5)), int(rng.integers(0, 4))
        A = verify_mask(C, N, B, tau)
        P = C + N
        tail = A[N:, P:]
        # each mask slot sees exactly B tail keys: the tau(j) < tau(i) data
        # tokens and the tau(j) >= tau(i) slots partition the B positions
        for i in range(B):
            assert tail[B + i].sum() == B
        # data token D_j sees exactly tau(j) data tokens and no mask slot
        for j in range(B):
            assert tail[j, :B].sum() == tau[j]
            assert tail[j, B:].sum() == 0
        # total allowed tail pairs
        assert tail.sum() == B * (B + 1) // 2 + B * B
        # every tail row sees the whole prompt
        assert np.all(A[N:, :P] == 1)
        # every row sees itself
        for i in range(N):
            assert A[i, C + i] == 1
        for r in range(2 * B):
            assert A[N + r, P + r] == 1


def test_prompt_rows_causal_and_blind_to_tail():
    A = verify_mask(4, 6, 3, [3, 1, 2])
    for i in range(6):
        assert A[i, :4 + i + 1].all() and not A[i, 4 + i + 1:].any()


def test_mask_slot_never_sees_unrevealed_data():
    rng = np.random.default_rng(0)
    B = 12
    tau = rng.permutation(B) + 1
    A = verify_mask(0, 0, B, tau)
    for i in range(B):
        for j in range(B):
            if tau[j] >= tau[i]:
                assert A[B + i, j] == 0    # future or own data token is hidden


def test_identity_stage_map_data_rows_are_causal():
    B = 7
    A = verify_mask(2, 3, B, list(range(1, B + 1)))
    sub = A[3:3 + B, 5:5 + B]
    np.testing.assert_array_equal(sub, np.tril(np.ones((B, B), np.uint8)))


def test_rejects_non_permutation():
    with pytest.raises(AssertionError):
        verify_mask(0, 0, 3, [1, 1, 2])
