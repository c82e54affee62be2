"""Pins for oracle.rope (CPU only).

RoPE with the RoPE-copy index (SimSD summary, section 3): positions from a
hand-worked fixture, the complex-exponential form of the rotation, the
relative-position property, and norm preservation.
"""
import numpy as np
import pytest

from oracle.rope import rope_positions, rotate, inv_freq, rope_copy_batch
from golden_io import read_fixture
from diffusion_speculative_verification_gb300 import workloads as W


def test_positions_fixture():
    meta, _ = read_fixture("rope_positions_C3_N2_B2.txt")
    pos = rope_positions(meta["C"], meta["N"], meta["B"])
    assert pos.tolist() == meta["pos"]


def test_given_positions_fixture():
    meta, _ = read_fixture("rope_positions_given_C5_N1_B2.txt")
    pos = rope_positions(meta["C"], meta["N"], meta["B"], meta["given"])
    assert pos.tolist() == meta["pos"]
    # the default positions are what a table holding them gives
    C, N, B = 9, 2, 4
    dflt = rope_positions(C, N, B)
    assert rope_positions(C, N, B, list(dflt[:N + B])).tolist() == dflt.tolist()


def test_given_positions_batch_reads_fresh_and_data_rows_only():
    a = W.make_attn_inputs("t", [3, 0], [2, 1], [3, 2], 2, 1, 64, W.F32, seed=21)
    q = W.values_f64(a.q_raw, a.dtype)
    k = W.values_f64(a.k_new_raw, a.dtype)
    rows = a.total_rows
    table = np.full(rows, -99, np.int64)   # mask-row entries must never be read
    per = [[11, 12, 40, 41, 42], [7, 30, 31]]
    for (C, N, B, q_off, _kv, _t), given in zip(a.seqs, per):
        table[q_off:q_off + N + B] = given
    qo, ko = rope_copy_batch(a.seqs, q, k, positions=table)
    for (C, N, B, q_off, _kv, _t), given in zip(a.seqs, per):
        pos = given[:N] + given[N:] + given[N:]
        np.testing.assert_array_equal(qo[q_off:q_off + N + 2 * B], rotate(q[q_off:q_off + N + 2 * B], np.array(pos)))
        np.testing.assert_array_equal(ko[q_off:q_off + N + 2 * B], rotate(k[q_off:q_off + N + 2 * B], np.array(pos)))


def test_pair_shares_position():
    for C, N, B in [(0, 0, 1), (16, 0, 4), (5, 9, 32)]:
        pos = rope_positions(C, N, B)
        np.testing.assert_array_equal(pos[N:N + B], pos[N + B:])
        assert pos[N] == C + N


@pytest.mark.parametrize("d", [64, 128])
def test_complex_exponential_form(d):
    rng = np.random.default_rng(d)
    x = rng.standard_normal((7, 3, d))
    pos = rng.integers(0, 9000, size=7)
    out = rotate(x, pos)
    half = d // 2
    theta = 10000.0 ** (-np.arange(half) * 2.0 / d)
    z = (x[:, :, :half] + 1j * x[:, :, half:]) * np.exp(1j * pos[:, None, None] * theta[None, None, :])
    # angles reach 9000 rad, so fp64 angle rounding alone is ~1e-12
    np.testing.assert_allclose(out[:, :, :half], z.real, rtol=0, atol=1e-10)
    np.testing.assert_allclose(out[:, :, half:], z.imag, rtol=0, atol=1e-10)


def test_position_zero_identity_and_norm():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 2, 128))
    np.testing.assert_array_equal(rotate(x, np.zeros(5, np.int64)), x)
    y = rotate(x, np.arange(5) * 1234)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_relative_position():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 1, 128))
    k = rng.standard_normal((1, 1, 128))
    base = (rotate(q, [40]) * rotate(k, [13])).sum()
    for shift in [1, 100, 4096]:
        shifted = (rotate(q, [40 + shift]) * rotate(k, [13 + shift])).sum()
        assert abs(shifted - base) < 1e-12 * 128


def test_inv_freq_endpoints():
    th = inv_freq(128)
    assert th[0] == 1.0
    assert abs(th[-1] - 10000.0 ** (-126 / 128)) < 1e-18


def test_batch_rope_copy_equal_inputs_equal_outputs():
    # the same raw vector placed in D_k and D~_k must come out identical
    a = W.make_attn_inputs("t", [3, 5], [2, 0], [4, 2], 2, 1, 64, W.F32, seed=5)
    q = W.values_f64(a.q_raw, a.dtype)
    k = W.values_f64(a.k_new_raw, a.dtype)
    for C, N, B, off, *_ in a.seqs:
        q[off + N + B:off + N + 2 * B] = q[off + N:off + N + B]
        k[off + N + B:off + N + 2 * B] = k[off + N:off + N + B]
    qo, ko = rope_copy_batch(a.seqs, q, k)
    for C, N, B, off, *_ in a.seqs:
        np.testing.assert_array_equal(qo[off + N:off + N + B], qo[off + N + B:off + N + 2 * B])
        np.testing.assert_array_equal(ko[off + N:off + N + B], ko[off + N + B:off + N + 2 * B])
