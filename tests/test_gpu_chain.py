"""Two verification passes chained through the commit (GPU), against the
oracle.

SimSD summary, section 4 "Speculative decoding pipeline": the longest
accepted prefix is committed and the loop repeats; section 3: each mask slot
reuses its data token's RoPE index.  The pages do not describe the next
pass; the reading (stated in include/ssv.h): committed data rows keep their
slots' positions, and the next pass over the same block enters the emitted
target token as a fresh prompt row at its slot's position and redrafts the
block's remaining slots at theirs, through ssv_rope_copy's position table.
(A block with no slot left is followed by a new block of 4 slots after it.)

Pass 1: ssv_rope_copy -> ssv_verify_attn -> ssv_accept (greedy, planted
drafts) -> ssv_commit.  Pass 2: ssv_rope_copy (position table) ->
ssv_verify_attn over the committed caches.

* fp32 (SIMT kernel): pass 2's output against an oracle that rebuilds the
  whole chain from the raw inputs (fp64 rotation at the stated positions,
  oracle commit, fp64 attention), max abs 2e-5 (two fp32 rotations and an
  fp32 attention in between; the attention bar alone is 1e-5).
* bf16 (tensor-core kernel): each link against the oracle on the device's
  bytes (commit bit-exact, rotation within its bar, attention within 1e-2).
* Both: accepted lengths bit-exact; no two keys of a sequence in pass 2 share
  a position with a committed key of another slot (a check of the layout).
"""
import numpy as np
import pytest
import torch

from diffusion_speculative_verification_gb300 import workloads as W, ssv, io as sio
import oracle.rope as orope
import oracle.attention as oattn
import oracle.accept as oacc
import oracle.commit as ocommit
from gpu_common import ensure_built, compare_attn, bf16_ulp

pytestmark = pytest.mark.gpu


def setup_module():
    ensure_built()


def _stage_slots(tau):
    inv = np.empty(len(tau), np.int64)
    inv[np.asarray(tau) - 1] = np.arange(len(tau))
    return inv


def _run_chain(dtype, d, Hq, Hkv, cache, new, blocks, seed):
    rng = np.random.default_rng(seed)
    dev = "cuda"
    a1 = W.make_attn_inputs("chain1", cache, new, blocks, Hq, Hkv, d, dtype, seed)
    x1 = W.make_accept_inputs("chain1", W.MODE_ARGMAX, 0.0, 700, blocks, blocks, seed + 1, tau=a1.tau)
    # ---- pass 1 on the GPU ----
    t1 = sio.attn_to_device(a1, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    q1, k1 = torch.empty_like(t1["q"]), torch.empty_like(t1["k_new"])
    ssv.rope_copy(t1["q"], t1["k_new"], t1["batch"], a1.rope_base, q_out=q1, k_out=k1, dev_status=st)
    ssv.verify_attn(q1, t1["k_cache"], t1["v_cache"], k1, t1["v_new"], t1["batch"], t1["tau"], dev_status=st)
    d1 = sio.accept_to_device(x1, dev)
    n_acc, n_out, tokens = ssv.accept(d1["mode"], d1["T"], d1["logits"], d1["draft_tokens"], d1["tau"], d1["block"],
                                      d1["gamma"], d1["slot_off"], max_block=d1["max_block"], dev_status=st)
    n_acc_h = n_acc.cpu().numpy()
    ref1 = oacc.accept_batch(x1)
    assert np.array_equal(n_acc_h, ref1["n_acc"]) and np.array_equal(tokens.cpu().numpy(), ref1["tokens"])
    # destination caches: each sequence's pass-1 cache copied in, room after it
    batch = len(blocks)
    C1 = a1.seqs[:, 0].astype(np.int64)
    N1 = a1.seqs[:, 1].astype(np.int64)
    B1 = a1.seqs[:, 2].astype(np.int64)
    cap = C1 + N1 + B1 + 2
    dst_off = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int32)
    dst_rows = int(cap.sum())
    k_dst = np.zeros((dst_rows, Hkv, d), a1.k_cache.dtype)
    v_dst = np.zeros_like(k_dst)
    for b in range(batch):
        kv = int(a1.seqs[b][4])
        k_dst[dst_off[b]:dst_off[b] + C1[b]] = a1.k_cache[kv:kv + C1[b]]
        v_dst[dst_off[b]:dst_off[b] + C1[b]] = a1.v_cache[kv:kv + C1[b]]
    kd, vd = sio.tensor(k_dst, dtype, dev), sio.tensor(v_dst, dtype, dev)
    new_len = ssv.commit(k1, t1["v_new"], kd, vd, t1["batch"], t1["tau"], n_acc, sio.int_tensor(dst_off, dev),
                         sio.int_tensor(cap.astype(np.int32), dev), dev_status=st)
    assert np.array_equal(new_len.cpu().numpy(), C1 + N1 + n_acc_h)
    # ---- pass 2 layout: emitted token as a fresh row, remaining slots redrafted ----
    C2, N2, B2, given, taus = [], [], [], [], []
    for b in range(batch):
        P = int(C1[b] + N1[b])
        B = int(B1[b])
        slots = _stage_slots(a1.tau[int(a1.seqs[b][5]):int(a1.seqs[b][5]) + B])
        na = int(n_acc_h[b])
        fresh = [P + int(slots[na])] if na < B else []
        rem = sorted(int(s) for s in slots[na + 1:])
        data = [P + s for s in rem] if rem else [P + B + j for j in range(4)]
        C2.append(int(C1[b] + N1[b] + na))
        N2.append(len(fresh))
        B2.append(len(data))
        given.append(fresh + data)
        taus.append((rng.permutation(len(data)) + 1).astype(np.int32))
        # layout check: pass-2 positions are new to this sequence's cache
        committed = set(range(P)) | {P + int(s) for s in slots[:na]}
        assert not committed & set(fresh + data)
    seqs2 = W.seq_table(C2, N2, B2)
    seqs2[:, 4] = dst_off
    rows2 = int(np.sum(np.asarray(N2) + 2 * np.asarray(B2)))
    table = np.full(rows2, -1, np.int32)   # mask-row entries are never read
    for b in range(batch):
        q_off = int(seqs2[b][3])
        table[q_off:q_off + N2[b] + B2[b]] = given[b]
    a2 = W.make_attn_inputs("chain2", C2, N2, B2, Hq, Hkv, d, dtype, seed + 2)
    a2.seqs = seqs2
    a2.tau = np.concatenate(taus)
    # ---- pass 2 on the GPU ----
    batch2 = ssv.Batch(seqs2, dev)
    qr, kr = sio.tensor(a2.q_raw, dtype, dev), sio.tensor(a2.k_new_raw, dtype, dev)
    v2 = sio.tensor(a2.v_new, dtype, dev)
    q2, k2 = torch.empty_like(qr), torch.empty_like(kr)
    ssv.rope_copy(qr, kr, batch2, a2.rope_base, q_out=q2, k_out=k2, positions=sio.int_tensor(table, dev),
                  dev_status=st)
    tau2 = sio.int_tensor(a2.tau, dev)
    o2 = torch.empty(q2.shape, dtype=torch.float32, device=dev)
    ssv.verify_attn(q2, kd, vd, k2, v2, batch2, tau2, out=o2, dev_status=st)
    assert ssv.get_status(st) == ssv.SSV_OK
    return dict(a1=a1, n_acc=n_acc_h, k1=k1, kd=kd, vd=vd, k_dst=k_dst, v_dst=v_dst, dst_off=dst_off, a2=a2,
                table=table, q2=q2, k2=k2, o2=o2.cpu().numpy().astype(np.float64), dtype=dtype)


@pytest.mark.parametrize("d", [64, 128])
def test_chain_fp32_against_oracle_from_raw(d):
    r = _run_chain(W.F32, d, 4, 2, [40, 0, 130, 7], [3, 5, 0, 2], [8, 4, 16, 1], 61 + d)
    a1, a2 = r["a1"], r["a2"]
    # oracle: the whole chain from the raw inputs
    q1o, k1o = orope.rope_copy_batch(a1.seqs, W.values_f64(a1.q_raw, a1.dtype), W.values_f64(a1.k_new_raw, a1.dtype),
                                     a1.rope_base)
    kc, vc, nl = ocommit.commit_batch(a1.seqs, a1.tau, r["n_acc"], k1o, W.values_f64(a1.v_new, a1.dtype),
                                      W.values_f64(r["k_dst"], a1.dtype), W.values_f64(r["v_dst"], a1.dtype),
                                      r["dst_off"])
    q2o, k2o = orope.rope_copy_batch(a2.seqs, W.values_f64(a2.q_raw, a2.dtype), W.values_f64(a2.k_new_raw, a2.dtype),
                                     a2.rope_base, positions=r["table"])
    ref = oattn.verify_attention(a2.seqs, a2.tau, q2o, kc, vc, k2o, W.values_f64(a2.v_new, a2.dtype))
    err = np.abs(r["o2"] - ref)
    assert err.max() <= 2e-5, err.max()


def test_chain_bf16_each_link():
    r = _run_chain(W.BF16, 128, 16, 4, [300, 0, 1030], [0, 70, 3], [8, 32, 16], 71)
    a1, a2 = r["a1"], r["a2"]
    # commit: bit-exact on the device's pass-1 rotated rows
    k1 = sio.to_numpy_storage(r["k1"])
    kc_ref, vc_ref, _ = ocommit.commit_batch(a1.seqs, a1.tau, r["n_acc"], k1, a1.v_new, r["k_dst"], r["v_dst"],
                                             r["dst_off"])
    kc = sio.to_numpy_storage(r["kd"])
    vc = sio.to_numpy_storage(r["vd"])
    assert np.array_equal(kc, kc_ref) and np.array_equal(vc, vc_ref)
    # pass-2 rotation at the table's positions: the rotation bar
    q2o, k2o = orope.rope_copy_batch(a2.seqs, W.values_f64(a2.q_raw, a2.dtype), W.values_f64(a2.k_new_raw, a2.dtype),
                                     a2.rope_base, positions=r["table"])
    for got_t, ref, raw in ((r["q2"], q2o, a2.q_raw), (r["k2"], k2o, a2.k_new_raw)):
        got = W.values_f64(sio.to_numpy_storage(got_t), a2.dtype)
        x = np.abs(W.values_f64(raw, a2.dtype))
        half = x.shape[-1] // 2
        pair = np.concatenate([x[..., :half] + x[..., half:]] * 2, axis=-1)
        assert np.all(np.abs(got - ref) <= bf16_ulp(ref) + 2.0 ** -21 * pair)
    # pass-2 attention on the device's bytes
    q2 = W.values_f64(sio.to_numpy_storage(r["q2"]), a2.dtype)
    k2 = W.values_f64(sio.to_numpy_storage(r["k2"]), a2.dtype)
    ref = oattn.verify_attention(a2.seqs, a2.tau, q2, W.values_f64(kc, a2.dtype), W.values_f64(vc, a2.dtype), k2,
                                 W.values_f64(a2.v_new, a2.dtype))
    compare_attn(r["o2"], ref, False, False)
