"""GPU parity of tree (state-set) verification against the oracle (SPOT
review, "How it works" / "How it is used": a draft tree of block states
verified by state equality; SimSD summary section 2 for the mask of a state).

Attention: every defined output row against the fp64 oracle on the same
bytes -- fp32 inputs max abs 1e-5, bf16 inputs with fp32 output max abs
1e-2, bf16 output 1e-2 + 2^-8 |ref| (the verification pass's bars); rows of
committed positions keep what the output held.  Acceptance: n_acc, the
accepted path and the emitted transition bit-exact; the decisions compare
identical fp32 scores, and at every node the walk visits the two best
confidences lie more than 1e-4 apart in the seeded sets (asserted), well
outside the device's fp32 logsumexp error (about 1e-6)."""
import numpy as np
import pytest
import torch

from diffusion_speculative_verification_gb300 import ssv, workloads as W, io as sio
import oracle.tree as otree
from gpu_common import ensure_built, compare_attn

pytestmark = pytest.mark.gpu

CONF_MARGIN = 1e-4


def setup_module():
    ensure_built()


def _attn(t, out_dtype=None, sentinel=7.0, dev_status=None):
    d = sio.tree_to_device(t)
    od = {None: None, "f32": torch.float32, "bf16": torch.bfloat16}[out_dtype]
    out = torch.full((t.total_out, t.Hq, t.d), sentinel, dtype=od or d["q"].dtype, device="cuda")
    ssv.tree_verify_attn(d["q"], d["k_cache"], d["v_cache"], d["k_new"], d["v_new"], d["seqs"], d["parent"],
                         d["pos"], t.total_out, d["max_cache"], out=out, dev_status=dev_status)
    return out


def _oracle_attn(t):
    return otree.tree_attention(t.seqs, t.parent, t.pos, W.values_f64(t.q, t.dtype), W.values_f64(t.k_cache, t.dtype),
                                W.values_f64(t.v_cache, t.dtype), W.values_f64(t.k_new, t.dtype),
                                W.values_f64(t.v_new, t.dtype))


CASES = {
    "f32_d64": lambda: W.make_tree_inputs("a", [30, 0, 7], [3, 5, 0], [8, 4, 16], [10, 3, 25], 4, 2, 64, W.F32, 91),
    "f32_d128_chainish": lambda: W.make_tree_inputs("b", [100], [2], [32], [40], 8, 2, 128, W.F32, 92),
    "bf16_d128_g4": lambda: W.make_tree_inputs("c", [300, 70], [0, 9], [16, 8], [12, 20], 16, 4, 128, W.BF16, 93),
    "bf16_g16": lambda: W.make_tree_inputs("d", [64], [4], [12], [9], 32, 2, 128, W.BF16, 94),
    "bf16_max_tree": lambda: W.make_tree_inputs("e", [40], [0], [64], [63], 8, 8, 128, W.BF16, 95),
    "empty_tree": lambda: W.make_tree_inputs("f", [20, 5], [1, 0], [3, 1], [0, 0], 4, 4, 64, W.BF16, 96),
    "no_prompt": lambda: W.make_tree_inputs("g", [0], [0], [6], [7], 2, 1, 64, W.F32, 97),
}


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_tree_attention_parity(name, out):
    t = CASES[name]()
    if t.dtype == W.F32 and out == "bf16":
        pytest.skip("fp32 inputs produce fp32 outputs")
    got_t = _attn(t, out)
    got = W.values_f64(sio.to_numpy_storage(got_t), W.BF16 if out == "bf16" else W.F32)
    ref = _oracle_attn(t)
    defined = ~np.isnan(ref[:, 0, 0])
    compare_attn(got[defined], ref[defined], out == "bf16", t.dtype == W.F32)
    assert np.all(got[~defined] == 7.0)                     # committed positions: not written


def test_bad_tree_is_skipped():
    t = W.make_tree_inputs("bad", [10, 10], [0, 0], [4, 4], [3, 3], 4, 2, 64, W.F32, 98)
    t.pos[3 + 1] = t.pos[3]            # sequence 1: edge 1 re-commits edge 0's position under it, or a sibling's
    t.parent[3 + 1] = 0                # hang edge 1 under edge 0: its position is then committed already
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _attn(t, "f32", dev_status=st).cpu().numpy().astype(np.float64)
    assert ssv.get_status(st) == ssv.SSV_ERR_INVALID
    s1 = t.seqs[1]
    assert np.all(got[int(s1[8]):int(s1[8]) + int(s1[1]) + (int(s1[3]) + 1) * int(s1[2])] == 7.0)
    good = W.make_tree_inputs("bad", [10, 10], [0, 0], [4, 4], [3, 3], 4, 2, 64, W.F32, 98)
    ref = _oracle_attn(good)
    s0 = t.seqs[0]
    rows = np.arange(int(s0[8]), int(s0[8]) + (int(s0[3]) + 1) * int(s0[2]))
    ok = ~np.isnan(ref[rows, 0, 0])
    compare_attn(got[rows][ok], ref[rows][ok], False, True)


def _accept(t, dev_status=None):
    d = sio.tree_to_device(t)
    n_acc, path, ep, et = ssv.tree_accept(t.mode, t.T, d["logits"], d["seqs"], d["parent"], d["pos"], d["token"],
                                          noise=d["noise"], noise_row=d["noise_row"], pos_off=d["pos_off"],
                                          dev_status=dev_status)
    return n_acc.cpu().numpy(), path.cpu().numpy(), ep.cpu().numpy(), et.cpu().numpy()


def _compare_accept(t, got):
    n_acc, path, ep, et = got
    ref = otree.tree_accept_batch(t.mode, t.T, t.seqs, t.parent, t.pos, t.token, t.logits, t.noise, t.noise_row,
                                  t.pos_off)
    for b, r in enumerate(ref):
        assert all(g > CONF_MARGIN for g in r.gaps), f"seq {b}: a confidence gap inside the band; pick another seed"
        assert n_acc[b] == r.n_acc, f"seq {b}: n_acc {n_acc[b]} vs {r.n_acc}"
        assert path[b, :r.n_acc].tolist() == r.path and np.all(path[b, r.n_acc:] == -1)
        assert (ep[b], et[b]) == (r.emit_pos, r.emit_tok), f"seq {b}: emitted {(ep[b], et[b])} vs {(r.emit_pos, r.emit_tok)}"
        if t.planted is not None:
            assert r.path == t.planted[b][0]


ACC = {
    "argmax_small": dict(mode=W.MODE_ARGMAX, T=0.0, V=700, cache=[5] * 6, blocks=[8, 4, 16, 3, 8, 32],
                         edges=[12, 5, 30, 2, 0, 40]),
    "gumbel_T1": dict(mode=W.MODE_GUMBEL, T=1.0, V=5000, cache=[5] * 4, blocks=[8, 16, 4, 12], edges=[10, 25, 3, 14]),
    "argmax_full_vocab": dict(mode=W.MODE_ARGMAX, T=0.0, V=151936, cache=[5] * 2, blocks=[8, 4], edges=[9, 5]),
    "max_tree": dict(mode=W.MODE_ARGMAX, T=0.0, V=300, cache=[5], blocks=[64], edges=[63]),
    # T != 1: the score divides by T (IEEE division) before the noise is added
    "gumbel_T07": dict(mode=W.MODE_GUMBEL, T=0.7, V=5000, cache=[5] * 3, blocks=[8, 12, 4], edges=[10, 20, 3]),
    # 37 vocabulary chunks: a row's confidence merges more chunks than a warp has lanes
    "argmax_37_chunks": dict(mode=W.MODE_ARGMAX, T=0.0, V=300000, cache=[5] * 2, blocks=[8, 4], edges=[6, 4]),
}


@pytest.mark.parametrize("name", list(ACC))
def test_tree_accept_parity(name):
    c = ACC[name]
    t = W.make_tree_inputs(name, c["cache"], [0] * len(c["blocks"]), c["blocks"], c["edges"], 2, 1, 64, W.F32,
                           seed=sum(map(ord, name)) + 900, V=c["V"], mode=c["mode"], T=c["T"])
    _compare_accept(t, _accept(t))


def test_tree_accept_rejects_bad_tree():
    t = W.make_tree_inputs("badacc", [5, 5], [0, 0], [4, 4], [3, 3], 2, 1, 64, W.F32, seed=920, V=100)
    t.parent[3 + 2] = 2                 # sequence 1, edge 2: hangs under itself
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_acc, path, ep, et = _accept(t, dev_status=st)
    assert ssv.get_status(st) == ssv.SSV_ERR_INVALID
    assert n_acc[1] == -1 and ep[1] == -1
    good = W.make_tree_inputs("badacc", [5, 5], [0, 0], [4, 4], [3, 3], 2, 1, 64, W.F32, seed=920, V=100)
    r0 = otree.tree_accept_batch(good.mode, good.T, good.seqs, good.parent, good.pos, good.token, good.logits)[0]
    assert n_acc[0] == r0.n_acc and (ep[0], et[0]) == (r0.emit_pos, r0.emit_tok)


def test_tree_attention_workspace_reuse():
    """The tensor-core prompt pass leaves its workspace reusable: a second call
    on the same workspace gives identical outputs."""
    t = CASES["bf16_d128_g4"]()
    d = sio.tree_to_device(t)
    a = ssv.tree_attn_args(d["q"], d["k_cache"], d["v_cache"], d["k_new"], d["v_new"],
                           torch.zeros((t.total_out, t.Hq, t.d), dtype=torch.bfloat16, device="cuda"), d["seqs"],
                           d["parent"], d["pos"], t.total_out, d["max_cache"])
    nbytes = ssv.tree_verify_attn_workspace_bytes(a)
    assert nbytes > 0  # bf16, d = 128: the prompt pass runs on the tensor cores
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        o = torch.full((t.total_out, t.Hq, t.d), 7.0, dtype=torch.bfloat16, device="cuda")
        ssv.tree_verify_attn(d["q"], d["k_cache"], d["v_cache"], d["k_new"], d["v_new"], d["seqs"], d["parent"],
                             d["pos"], t.total_out, d["max_cache"], out=o, workspace=ws)
        outs.append(o.float().cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
