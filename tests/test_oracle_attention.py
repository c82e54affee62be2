"""Pins for oracle.attention (CPU only).

Reductions to textbook routines (torch's scaled_dot_product_attention in
float64 on the CPU, a library routine the oracle does not use):
  * B = 1 and the identity stage map: data rows are ordinary causal
    attention over [prompt, D];
  * every mask slot D~_i equals *unmasked* attention over the block state
    after stage tau(i)-1: prompt keys plus, per position j, D_j if
    tau(j) < tau(i) else D~_j (the prefix-conditioned context of the SimSD
    summary, section 2);
  * grouped-query heads equal multi-head attention with repeated kv heads.
Properties: no-leak (perturbing keys a row may not see leaves it
bit-identical) and permutation equivariance.
"""
import numpy as np
import pytest
import torch

from oracle.attention import verify_attention
from diffusion_speculative_verification_gb300 import workloads as W


def sdpa(q, k, v, causal):
    """q [R, d], k/v [K, d] float64 -> [R, d] via torch SDPA (R == K when causal)."""
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x))[None, None]
    out = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=causal)
    return out[0, 0].numpy()


def f64_inputs(a):
    return tuple(W.values_f64(x, a.dtype) for x in (a.q_raw, a.k_cache, a.v_cache, a.k_new_raw, a.v_new))


def run_oracle(a, q, kc, vc, kn, vn):
    return verify_attention(a.seqs, a.tau, q, kc, vc, kn, vn)


@pytest.mark.parametrize("C,N", [(0, 5), (7, 0), (6, 4)])
def test_B1_reduces_to_causal(C, N):
    a = W.make_attn_inputs("t", [C], [N], [1], 1, 1, 32, W.F32, seed=11)
    q, kc, vc, kn, vn = f64_inputs(a)
    o = run_oracle(a, q, kc, vc, kn, vn)
    rng = np.random.default_rng(0)
    qc = rng.standard_normal((C, 32))          # queries for cache rows (discarded)
    # prompt rows and D_1: causal over [cache, prompt, D_1]
    seq_q = np.concatenate([qc, q[:N + 1, 0]])
    seq_k = np.concatenate([kc[:, 0], kn[:N + 1, 0]])
    seq_v = np.concatenate([vc[:, 0], vn[:N + 1, 0]])
    ref = sdpa(seq_q, seq_k, seq_v, True)[C:]
    np.testing.assert_allclose(o[:N + 1, 0], ref, atol=1e-12, rtol=0)
    # mask slot D~_1: causal over [cache, prompt, D~_1] (last row)
    seq_q = np.concatenate([qc, q[:N, 0], q[N + 1:N + 2, 0]])
    seq_k = np.concatenate([kc[:, 0], kn[:N, 0], kn[N + 1:N + 2, 0]])
    seq_v = np.concatenate([vc[:, 0], vn[:N, 0], vn[N + 1:N + 2, 0]])
    ref = sdpa(seq_q, seq_k, seq_v, True)[-1]
    np.testing.assert_allclose(o[N + 1, 0], ref, atol=1e-12, rtol=0)


def test_identity_tau_data_rows_causal():
    C, N, B = 5, 3, 6
    a = W.make_attn_inputs("t", [C], [N], [B], 1, 1, 32, W.F32, seed=12)
    a.tau[:] = np.arange(1, B + 1)
    q, kc, vc, kn, vn = f64_inputs(a)
    o = run_oracle(a, q, kc, vc, kn, vn)
    qc = np.random.default_rng(1).standard_normal((C, 32))
    seq_q = np.concatenate([qc, q[:N + B, 0]])
    seq_k = np.concatenate([kc[:, 0], kn[:N + B, 0]])
    seq_v = np.concatenate([vc[:, 0], vn[:N + B, 0]])
    ref = sdpa(seq_q, seq_k, seq_v, True)[C:]
    np.testing.assert_allclose(o[:N + B, 0], ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("B", [1, 2, 5, 16])
def test_mask_rows_equal_block_state_attention(B):
    C, N = 9, 2
    a = W.make_attn_inputs("t", [C], [N], [B], 1, 1, 64, W.F32, seed=100 + B)
    q, kc, vc, kn, vn = f64_inputs(a)
    o = run_oracle(a, q, kc, vc, kn, vn)
    tau = a.tau
    for i in range(B):
        state = [N + j if tau[j] < tau[i] else N + B + j for j in range(B)]
        keys = np.concatenate([kc[:, 0], kn[:N, 0], kn[state, 0]])
        vals = np.concatenate([vc[:, 0], vn[:N, 0], vn[state, 0]])
        ref = sdpa(q[N + B + i:N + B + i + 1, 0], keys, vals, False)
        np.testing.assert_allclose(o[N + B + i, 0], ref[0], atol=1e-12, rtol=0)


def test_gqa_matches_repeated_heads():
    Hq, Hkv = 6, 2
    a = W.make_attn_inputs("t", [4, 2], [1, 3], [3, 2], Hq, Hkv, 32, W.F32, seed=13)
    q, kc, vc, kn, vn = f64_inputs(a)
    o = run_oracle(a, q, kc, vc, kn, vn)
    G = Hq // Hkv
    rep = lambda x: np.repeat(x, G, axis=1)
    o2 = verify_attention(a.seqs, a.tau, q, rep(kc), rep(vc), rep(kn), rep(vn))
    np.testing.assert_array_equal(o, o2)
    # and head h reads kv head h // G: swapping kv heads swaps head groups
    sw = lambda x: x[:, ::-1].copy()
    o3 = verify_attention(a.seqs, a.tau, q[:, list(range(G, Hq)) + list(range(G))], sw(kc), sw(vc), sw(kn), sw(vn))
    np.testing.assert_array_equal(o3[:, :Hq - G], o[:, G:])


def test_no_leak_bit_identical():
    C, N, B = 6, 2, 8
    a = W.make_attn_inputs("t", [C], [N], [B], 2, 1, 32, W.F32, seed=14)
    q, kc, vc, kn, vn = f64_inputs(a)
    o = run_oracle(a, q, kc, vc, kn, vn)
    tau = a.tau
    rng = np.random.default_rng(3)
    for i in range(B):
        kn2, vn2 = kn.copy(), vn.copy()
        hidden = [N + j for j in range(B) if tau[j] >= tau[i]]          # data not yet revealed (incl. D_i)
        hidden += [N + B + j for j in range(B) if tau[j] < tau[i]]      # slots already decided
        kn2[hidden] += rng.standard_normal(kn2[hidden].shape) * 10
        vn2[hidden] += rng.standard_normal(vn2[hidden].shape) * 10
        o2 = run_oracle(a, q, kc, vc, kn2, vn2)
        np.testing.assert_array_equal(o2[N + B + i], o[N + B + i])
    # prompt rows never see the tail
    kn2, vn2 = kn.copy(), vn.copy()
    kn2[N:] += 5.0
    vn2[N:] -= 3.0
    o2 = run_oracle(a, q, kc, vc, kn2, vn2)
    np.testing.assert_array_equal(o2[:N], o[:N])


def test_permutation_equivariance():
    C, N, B = 5, 0, 6
    a = W.make_attn_inputs("t", [C], [N], [B], 1, 1, 32, W.F32, seed=15)
    q, kc, vc, kn, vn = f64_inputs(a)
    o = run_oracle(a, q, kc, vc, kn, vn)
    perm = np.random.default_rng(4).permutation(B)
    rows = np.concatenate([perm, B + perm])
    a2 = W.make_attn_inputs("t", [C], [N], [B], 1, 1, 32, W.F32, seed=15)
    a2.tau[:] = a.tau[perm]
    o2 = verify_attention(a2.seqs, a2.tau, q[rows], kc, vc, kn[rows], vn[rows])
    np.testing.assert_allclose(o2, o[rows], atol=1e-13, rtol=0)


def test_row_sampling_matches_full():
    a = W.make_attn_inputs("t", [3, 0], [4, 6], [2, 3], 2, 1, 32, W.F32, seed=16)
    q, kc, vc, kn, vn = f64_inputs(a)
    full = run_oracle(a, q, kc, vc, kn, vn)
    part = verify_attention(a.seqs, a.tau, q, kc, vc, kn, vn, rows_of={1: [0, 5, 7]})
    off = a.seqs[1, 3]
    for r in [0, 5, 7]:
        np.testing.assert_array_equal(part[off + r], full[off + r])
    assert np.isnan(part[0]).all()
