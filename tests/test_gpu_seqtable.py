"""GPU tests of the rotation's position table and of the device-side checks
of the sequence table (SimSD summary, section 3 "Position Encoding
Alignment": each mask slot reuses its data token's RoPE index; section 2
for the attention).

* Position table: ssv_rope_copy with an explicit position per fresh row and
  per data row (mask rows take their data row's) against the fp64 oracle
  given the same table, with the bars of the rotation tests.
* A sequence whose extents leave the call's buffers is skipped by the
  rotation and by both attention kernels: nothing of it is read or written
  (its output rows keep a sentinel), SSV_ERR_INVALID is reported, and the
  other sequences keep oracle parity.
"""
import numpy as np
import pytest
import torch

from diffusion_speculative_verification_gb300 import workloads as W, ssv, io as sio
import oracle.rope as orope
import oracle.attention as oattn
from gpu_common import ensure_built, bf16_ulp, compare_attn, gpu_rope

pytestmark = pytest.mark.gpu

C_, N_, B_, QOFF, KVOFF, TOFF = range(6)   # ssv_seq fields


def setup_module():
    ensure_built()


def _check_rotation(a, got_q, got_k, ref_q, ref_k, rows):
    """The rotation bars (fp32: 1e-5; bf16: one ulp plus the fp32 rotation
    error) on the given rows."""
    for got, ref, raw in ((got_q, ref_q, a.q_raw), (got_k, ref_k, a.k_new_raw)):
        g, r = got[rows], ref[rows]
        err = np.abs(g - r)
        if a.dtype == W.F32:
            assert err.max() <= 1e-5, err.max()
        else:
            x = np.abs(W.values_f64(raw, a.dtype))[rows]
            half = x.shape[-1] // 2
            pair = np.concatenate([x[..., :half] + x[..., half:]] * 2, axis=-1)
            assert np.all(err <= bf16_ulp(r) + 2.0 ** -21 * pair)


@pytest.mark.parametrize("dtype", [W.BF16, W.F32])
def test_rope_position_table(dtype):
    a = W.make_attn_inputs("p", [40, 0, 900], [3, 6, 0], [8, 5, 16], 8, 2, 128, dtype, 51)
    table = np.random.default_rng(52).integers(0, 20000, size=a.total_rows).astype(np.int32)
    for C, N, B, q_off, *_ in a.seqs:
        table[q_off + N + B:q_off + N + 2 * B] = -7   # mask-row entries are never read
    t = sio.attn_to_device(a)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qo, ko = torch.zeros_like(t["q"]), torch.zeros_like(t["k_new"])
    ssv.rope_copy(t["q"], t["k_new"], t["batch"], a.rope_base, q_out=qo, k_out=ko,
                  positions=sio.int_tensor(table, "cuda"), dev_status=st)
    assert ssv.get_status(st) == ssv.SSV_OK
    rq, rk = orope.rope_copy_batch(a.seqs, W.values_f64(a.q_raw, a.dtype), W.values_f64(a.k_new_raw, a.dtype),
                                   a.rope_base, positions=table)
    gq = W.values_f64(sio.to_numpy_storage(qo), a.dtype)
    gk = W.values_f64(sio.to_numpy_storage(ko), a.dtype)
    _check_rotation(a, gq, gk, rq, rk, np.arange(a.total_rows))
    # the table holding the default positions gives the default rotation, bit for bit
    dflt = np.concatenate([orope.rope_positions(int(C), int(N), int(B)) for C, N, B, *_ in a.seqs]).astype(np.int32)
    q2, k2 = torch.zeros_like(t["q"]), torch.zeros_like(t["k_new"])
    ssv.rope_copy(t["q"], t["k_new"], t["batch"], a.rope_base, q_out=q2, k_out=k2,
                  positions=sio.int_tensor(dflt, "cuda"))
    q3, k3 = torch.zeros_like(t["q"]), torch.zeros_like(t["k_new"])
    ssv.rope_copy(t["q"], t["k_new"], t["batch"], a.rope_base, q_out=q3, k_out=k3)
    assert torch.equal(q2, q3) and torch.equal(k2, k3)


def _rows_of(seqs, b):
    C, N, B, q_off = (int(v) for v in seqs[b][:4])
    return np.arange(q_off, q_off + N + 2 * B)


ROPE_BAD = {
    "B_above_64": lambda s, a: s.__setitem__((1, B_), 65),
    "past_last_row": lambda s, a: s.__setitem__((2, N_), a.total_rows),
    "negative_new_len": lambda s, a: s.__setitem__((1, N_), -3),
}


@pytest.mark.parametrize("case", list(ROPE_BAD))
def test_rope_bad_sequence_skipped(case):
    a = W.make_attn_inputs("b", [10, 20, 30], [4, 0, 2], [8, 4, 16], 8, 2, 128, W.BF16, 53)
    t = sio.attn_to_device(a)
    bad = a.seqs.copy()
    ROPE_BAD[case](bad, a)
    badb = [i for i in range(a.batch) if not np.array_equal(bad[i], a.seqs[i])][0]
    t["batch"].dev.copy_(torch.from_numpy(bad))   # host totals stay those of the valid table
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qo = torch.full_like(t["q"], 3.0)
    ko = torch.full_like(t["k_new"], 3.0)
    ssv.rope_copy(t["q"], t["k_new"], t["batch"], a.rope_base, q_out=qo, k_out=ko, dev_status=st)
    assert ssv.get_status(st) == ssv.SSV_ERR_INVALID
    gq = W.values_f64(sio.to_numpy_storage(qo), a.dtype)
    gk = W.values_f64(sio.to_numpy_storage(ko), a.dtype)
    skipped = _rows_of(a.seqs, badb)
    assert np.all(gq[skipped] == 3.0) and np.all(gk[skipped] == 3.0)
    rq, rk = orope.rope_copy_batch(a.seqs, W.values_f64(a.q_raw, a.dtype), W.values_f64(a.k_new_raw, a.dtype),
                                   a.rope_base)
    good = np.concatenate([_rows_of(a.seqs, b) for b in range(a.batch) if b != badb])
    _check_rotation(a, gq, gk, rq, rk, good)


def test_rope_negative_table_entry_skips_its_row():
    a = W.make_attn_inputs("n", [5, 9], [2, 0], [4, 3], 4, 2, 64, W.F32, 55)
    table = np.concatenate([orope.rope_positions(int(C), int(N), int(B)) for C, N, B, *_ in a.seqs]).astype(np.int32)
    table[1] = -1          # fresh row 1 of sequence 0
    table[a.seqs[1][3]] = -5  # data row D_1 of sequence 1: D~_1 uses it too
    t = sio.attn_to_device(a)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qo = torch.full_like(t["q"], 3.0)
    ko = torch.full_like(t["k_new"], 3.0)
    ssv.rope_copy(t["q"], t["k_new"], t["batch"], a.rope_base, q_out=qo, k_out=ko,
                  positions=sio.int_tensor(table, "cuda"), dev_status=st)
    assert ssv.get_status(st) == ssv.SSV_ERR_INVALID
    gq = sio.to_numpy_storage(qo).astype(np.float64)
    gk = sio.to_numpy_storage(ko).astype(np.float64)
    q1 = int(a.seqs[1][3])
    B1 = int(a.seqs[1][2])
    skipped = np.array([1, q1, q1 + B1])
    assert np.all(gq[skipped] == 3.0) and np.all(gk[skipped] == 3.0)
    rq, rk = orope.rope_copy_batch(a.seqs, W.values_f64(a.q_raw, a.dtype), W.values_f64(a.k_new_raw, a.dtype),
                                   a.rope_base)
    good = np.setdiff1d(np.arange(a.total_rows), skipped)
    _check_rotation(a, gq, gk, rq, rk, good)


ATTN_BAD = {
    "kv_past_end": lambda s, a: s.__setitem__((1, KVOFF), a.total_cache - 10),
    "above_max_cache": lambda s, a: (s.__setitem__((1, C_), int(a.seqs[:, 0].max()) + 1),
                                     s.__setitem__((1, KVOFF), 0)),
    "tau_past_end": lambda s, a: s.__setitem__((2, TOFF), len(a.tau) - 2),
    "q_past_end": lambda s, a: s.__setitem__((2, N_), 100),
    "negative_kv_off": lambda s, a: s.__setitem__((0, KVOFF), -1),
}


@pytest.mark.parametrize("dtype,d", [(W.BF16, 128), (W.F32, 64)])
@pytest.mark.parametrize("case", list(ATTN_BAD))
def test_attn_bad_sequence_skipped(case, dtype, d):
    """bf16 / d = 128 runs the tensor-core kernel, fp32 the SIMT kernel."""
    a = W.make_attn_inputs("b", [300, 50, 700], [0, 5, 0], [8, 16, 4], 8, 2, d, dtype, 54)
    qo, ko, t = gpu_rope(a)
    bad = a.seqs.copy()
    ATTN_BAD[case](bad, a)
    badb = [i for i in range(a.batch) if not np.array_equal(bad[i], a.seqs[i])][0]
    t["batch"].dev.copy_(torch.from_numpy(bad))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.full(t["q"].shape, 5.0, dtype=torch.float32, device="cuda")
    ssv.verify_attn(qo, t["k_cache"], t["v_cache"], ko, t["v_new"], t["batch"], t["tau"], out=o, dev_status=st)
    assert ssv.get_status(st) == ssv.SSV_ERR_INVALID
    got = o.cpu().numpy().astype(np.float64)
    assert np.all(got[_rows_of(a.seqs, badb)] == 5.0)
    q64 = W.values_f64(sio.to_numpy_storage(qo), a.dtype)
    k64 = W.values_f64(sio.to_numpy_storage(ko), a.dtype)
    ref = oattn.verify_attention(a.seqs, a.tau, q64, W.values_f64(a.k_cache, a.dtype),
                                 W.values_f64(a.v_cache, a.dtype), k64, W.values_f64(a.v_new, a.dtype))
    good = np.concatenate([_rows_of(a.seqs, b) for b in range(a.batch) if b != badb])
    compare_attn(got[good], ref[good], False, a.dtype == W.F32)
