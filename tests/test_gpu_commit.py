"""GPU parity of ssv_commit against the oracle (SimSD summary, section 4
"Speculative decoding pipeline": the accepted prefix, in the draft's temporal
order, is committed; "Main contributions" 3: the method runs over a KV cache).

The commit moves bytes, so the bar is bit-exact on the whole destination
(appended rows and every row it must leave alone) and on new_len."""
import numpy as np
import pytest

from diffusion_speculative_verification_gb300 import ssv, workloads as W, io as sio
import oracle.commit as ocommit
from gpu_common import ensure_built, random_attn_shape

pytestmark = pytest.mark.gpu


def setup_module():
    ensure_built()


CASES = {
    "small_bf16": lambda: W.make_attn_inputs("c", [2, 0, 5], [1, 4, 0], [3, 1, 6], 4, 2, 64, W.BF16, 31),
    "ragged_bf16": lambda: W.make_attn_inputs("c", [0, 300, 129, 7], [0, 200, 5, 0], [1, 32, 64, 7], 8, 2, 128,
                                              W.BF16, 32),
    "f32_d128": lambda: W.make_attn_inputs("c", [90, 3], [3, 0], [64, 2], 4, 2, 128, W.F32, 33),
    "f32_d64_hkv1": lambda: W.make_attn_inputs("c", [5, 6, 7], [8, 0, 1], [16, 5, 2], 2, 1, 64, W.F32, 34),
    "gqa1p7b": lambda: W.workload_attn("gqa1p7b"),
    "gqa8b": lambda: W.workload_attn("gqa8b"),
    "sweep": lambda: W.workload_attn("sweep"),
    "random_a": lambda: random_attn_shape(300),
    "random_b": lambda: random_attn_shape(301, W.F32, 64),
}


def _run(c: W.CommitInputs, seqs=None, tau=None, n_acc=None, total_rows=None):
    """Runs ssv_commit on device copies; returns (k_dst, v_dst, new_len, status) as numpy."""
    import torch
    a = c.attn
    seqs = a.seqs if seqs is None else seqs
    tau = a.tau if tau is None else tau
    n_acc = c.n_acc if n_acc is None else n_acc
    k_new, v_new = a.k_new_raw, a.v_new
    if total_rows is not None and total_rows > k_new.shape[0]:
        pad = np.zeros((total_rows - k_new.shape[0],) + k_new.shape[1:], k_new.dtype)
        k_new, v_new = np.concatenate([k_new, pad]), np.concatenate([v_new, pad])
    batch = ssv.Batch(seqs)
    kd, vd = sio.tensor(c.k_dst, a.dtype, "cuda"), sio.tensor(c.v_dst, a.dtype, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nl = ssv.commit(sio.tensor(k_new, a.dtype, "cuda"), sio.tensor(v_new, a.dtype, "cuda"), kd, vd, batch,
                    sio.int_tensor(tau, "cuda"), sio.int_tensor(n_acc, "cuda"), sio.int_tensor(c.dst_off, "cuda"),
                    sio.int_tensor(c.dst_cap, "cuda"), dev_status=status)
    st = ssv.get_status(status)
    return sio.to_numpy_storage(kd), sio.to_numpy_storage(vd), nl.cpu().numpy(), st


def _oracle(c: W.CommitInputs, keep=None, seqs=None, tau=None, n_acc=None, k_new=None, v_new=None):
    """Oracle commit of the sequences in `keep` (all by default)."""
    a = c.attn
    seqs = a.seqs if seqs is None else seqs
    tau = a.tau if tau is None else tau
    n_acc = c.n_acc if n_acc is None else n_acc
    k_new = a.k_new_raw if k_new is None else k_new
    v_new = a.v_new if v_new is None else v_new
    keep = list(range(len(seqs))) if keep is None else keep
    return ocommit.commit_batch(seqs[keep], tau, n_acc[keep], k_new, v_new, c.k_dst, c.v_dst, c.dst_off[keep])


@pytest.mark.parametrize("name", list(CASES))
def test_commit_parity(name):
    c = W.make_commit_inputs(CASES[name](), seed=sum(map(ord, name)) + 7)  # fixed per case, replayable
    k, v, nl, st = _run(c)
    assert st == ssv.SSV_OK
    k_ref, v_ref, nl_ref = _oracle(c)
    assert np.array_equal(nl, nl_ref)
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


@pytest.mark.parametrize("which", ["none", "all"])
def test_commit_extremes(which):
    a = W.make_attn_inputs("c", [4, 0, 11], [2, 3, 0], [5, 64, 1], 4, 2, 128, W.BF16, 35)
    c = W.make_commit_inputs(a, 36)
    c.n_acc = np.zeros_like(c.n_acc) if which == "none" else a.seqs[:, 2].astype(np.int32).copy()
    k, v, nl, st = _run(c)
    assert st == ssv.SSV_OK
    k_ref, v_ref, nl_ref = _oracle(c)
    assert np.array_equal(nl, nl_ref)
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


def test_commit_rows_between_sequences():
    """Sequences packed with gaps in q_off: rows in the gaps are never copied."""
    a = W.make_attn_inputs("c", [3, 8], [2, 1], [4, 6], 4, 2, 64, W.F32, 37)
    seqs = a.seqs.copy()
    rows0 = int(seqs[0, 1] + 2 * seqs[0, 2])
    seqs[1, 3] = rows0 + 5
    total = int(seqs[1, 3] + seqs[1, 1] + 2 * seqs[1, 2])
    rng = np.random.default_rng(38)
    k_new = W._store(W._normal(rng, (total, a.Hkv, a.d)), a.dtype)
    v_new = W._store(W._normal(rng, (total, a.Hkv, a.d)), a.dtype)
    a.k_new_raw, a.v_new = k_new, v_new
    c = W.make_commit_inputs(a, 39)
    k, v, nl, st = _run(c, seqs=seqs)
    assert st == ssv.SSV_OK
    k_ref, v_ref, nl_ref = _oracle(c, seqs=seqs)
    assert np.array_equal(nl, nl_ref)
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


@pytest.mark.parametrize("fault", ["bad_tau", "n_acc_over_b", "n_acc_negative", "no_room", "tau_off_out"])
def test_commit_rejects_one_sequence(fault):
    """A sequence that fails the device checks is reported, gets new_len -1 and
    has none of its rows written; the other sequences commit normally."""
    a = W.make_attn_inputs("c", [6, 2, 9], [3, 0, 2], [8, 5, 12], 4, 2, 128, W.BF16, 40)
    c = W.make_commit_inputs(a, 41)
    c.n_acc = np.array([3, 5, 7], np.int32)
    seqs, tau, n_acc = a.seqs.copy(), a.tau.copy(), c.n_acc.copy()
    bad, want = 1, ssv.SSV_ERR_INVALID
    if fault == "bad_tau":
        o = int(seqs[bad, 5])
        tau[o + 1] = tau[o]
        want = ssv.SSV_ERR_BAD_TAU
    elif fault == "n_acc_over_b":
        n_acc[bad] = int(seqs[bad, 2]) + 1
    elif fault == "n_acc_negative":
        n_acc[bad] = -1
    elif fault == "no_room":
        c.dst_cap = c.dst_cap.copy()
        c.dst_cap[bad] = int(seqs[bad, 0] + seqs[bad, 1] + n_acc[bad]) - 1
    elif fault == "tau_off_out":
        seqs[bad, 5] = len(tau) - 2
    k, v, nl, st = _run(c, seqs=seqs, tau=tau, n_acc=n_acc)
    assert st == want
    assert nl[bad] == -1
    keep = [b for b in range(len(seqs)) if b != bad]
    k_ref, v_ref, nl_ref = _oracle(c, keep=keep, seqs=seqs, tau=tau, n_acc=n_acc)
    assert np.array_equal(nl[keep], nl_ref)
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


def test_commit_host_errors():
    import torch
    a = W.make_attn_inputs("c", [2], [1], [3], 4, 2, 64, W.BF16, 42)
    c = W.make_commit_inputs(a, 43)
    batch = ssv.Batch(a.seqs)
    kn, vn = sio.tensor(a.k_new_raw, a.dtype, "cuda"), sio.tensor(a.v_new, a.dtype, "cuda")
    kd, vd = sio.tensor(c.k_dst, a.dtype, "cuda"), sio.tensor(c.v_dst, a.dtype, "cuda")
    ints = [sio.int_tensor(x, "cuda") for x in (a.tau, c.n_acc, c.dst_off, c.dst_cap)]
    nl = torch.full((1,), 77, dtype=torch.int32, device="cuda")

    def call(args):
        return int(ssv.lib().ssv_commit(ssv.C.byref(args), ssv._stream_ptr(None)))

    good = ssv.commit_args(kn, vn, kd, vd, batch, *ints, nl)
    bad = ssv.commit_args(kn, vn, kd, vd, batch, *ints, nl)
    bad.d = 96
    assert call(bad) == ssv.SSV_ERR_UNSUPPORTED
    bad = ssv.commit_args(kn, vn, kd, vd, batch, *ints, nl)
    bad.k_new = good.k_new + 2
    assert call(bad) == ssv.SSV_ERR_INVALID
    bad = ssv.commit_args(kn, vn, kd, vd, batch, *ints, nl)
    bad.k_dst = good.k_new           # destination overlaps the fresh rows
    assert call(bad) == ssv.SSV_ERR_INVALID
    bad = ssv.commit_args(kn, vn, kd, vd, batch, *ints, nl)
    bad.n_acc = None
    assert call(bad) == ssv.SSV_ERR_INVALID
    bad = ssv.commit_args(kn, vn, kd, vd, batch, *ints, nl)
    bad.dtype = 7
    assert call(bad) == ssv.SSV_ERR_INVALID
    torch.cuda.synchronize()
    assert int(nl.item()) == 77      # nothing was launched
    empty = ssv.commit_args(kn, vn, kd, vd, batch, *ints, nl)
    empty.batch = 0
    assert call(empty) == ssv.SSV_OK
    assert call(good) == ssv.SSV_OK
    torch.cuda.synchronize()
    assert int(nl.item()) == 2 + 1 + int(c.n_acc[0])


def test_commit_then_attention_sees_the_accepted_tokens():
    """Two passes over one cache: commit pass 1 into a cache laid out with room
    (dst_off = kv_off), then run pass 2's attention over the grown cache; it
    matches the oracle attention over the oracle-committed cache."""
    import torch
    from gpu_common import compare_attn
    import oracle.attention as oattn
    a = W.make_attn_inputs("c", [40, 0, 17], [5, 9, 0], [8, 4, 16], 8, 2, 128, W.BF16, 44)
    c = W.make_commit_inputs(a, 45)
    k, v, nl, st = _run(c)
    assert st == ssv.SSV_OK
    # pass 2: every sequence continues from its grown cache with a fresh block
    seqs2 = W.seq_table(nl.tolist(), [0] * a.batch, [6, 3, 10])
    seqs2[:, 4] = c.dst_off
    a2 = W.make_attn_inputs("c2", nl.tolist(), [0] * a.batch, [6, 3, 10], a.Hq, a.Hkv, a.d, a.dtype, 46)
    t = dict(q=sio.tensor(a2.q_raw, a.dtype, "cuda"), k_new=sio.tensor(a2.k_new_raw, a.dtype, "cuda"),
             v_new=sio.tensor(a2.v_new, a.dtype, "cuda"))
    batch2 = ssv.Batch(seqs2)
    kc, vc = sio.tensor(k, a.dtype, "cuda"), sio.tensor(v, a.dtype, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = ssv.verify_attn(t["q"], kc, vc, t["k_new"], t["v_new"], batch2, sio.int_tensor(a2.tau, "cuda"),
                        out_dtype=torch.float32, dev_status=status)
    assert ssv.get_status(status) == ssv.SSV_OK
    got = W.values_f64(sio.to_numpy_storage(o), W.F32)
    k_ref, v_ref, nl_ref = _oracle(c)
    assert np.array_equal(nl, nl_ref)
    ref = oattn.verify_attention(seqs2, a2.tau, W.values_f64(a2.q_raw, a.dtype), W.values_f64(k_ref, a.dtype),
                                 W.values_f64(v_ref, a.dtype), W.values_f64(a2.k_new_raw, a.dtype),
                                 W.values_f64(a2.v_new, a.dtype))
    compare_attn(got, ref, out_is_bf16=False, in_is_f32=False)
