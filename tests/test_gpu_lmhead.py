"""GPU parity of ssv_lmhead_accept (LM head over the mask slots fused with
acceptance) against the oracle (SimSD summary, section 4; SPOT review, "How
it is used"; reading: l_k = W h_k, formed exactly and rounded once to fp32).

The device accumulates the exact bf16 products in fp32 in its own order, so
a decision between two tokens whose scores lie within the accumulation bound
(oracle.lmhead.error_bound, divided by T and plus one rounding of the
division and the addition for coupled noise) may go either way.  The bar:
  * per-row decisions (sequences with B = 1 and gamma = 0, whose emitted
    token is the row's decision): equal to the oracle's, or within the bound
    of the oracle's best score; at most 1% of rows may take the second road;
  * planted multi-stage sequences (every decision far outside the bound):
    n_acc, n_out and tokens bit-exact."""
import numpy as np
import pytest

from diffusion_speculative_verification_gb300 import ssv, workloads as W, io as sio
import oracle.accept as oacc
import oracle.lmhead as olm
from gpu_common import ensure_built

pytestmark = pytest.mark.gpu


def setup_module():
    ensure_built()


def _run(x, dev_status=None, workspace=None, w_dev=None, d=None):
    d = sio.lmhead_to_device(x, w=w_dev) if d is None else d
    n_acc, n_out, tokens = ssv.lmhead_accept(d["mode"], d["T"], d["h"], d["w"], d["draft_tokens"], d["tau"],
                                             d["block"], d["gamma"], d["slot_off"], noise=d["noise"],
                                             noise_row=d["noise_row"], dev_status=dev_status, workspace=workspace)
    return n_acc.cpu().numpy(), n_out.cpu().numpy(), tokens.cpu().numpy()


def _decision_inputs(mode, T, V, hidden, rows, seed, w=None):
    """rows sequences of one slot each, gamma = 0: each emits its row's decision."""
    x = W.make_lmhead_inputs("dec", mode, T, V, hidden, [1] * rows, [0] * rows, seed, w=w)
    return x


def _check_decisions(x, tokens):
    a = x.acc
    slots = np.arange(int(np.sum(a.blocks)))
    hv = olm.bf16_values(x.h)
    wv = olm.bf16_values(x.w)
    l64 = olm.lm_head_logits(hv, wv)
    l32 = l64.astype(np.float32)
    bound = olm.error_bound(hv, wv, l64)
    if a.mode == oacc.MODE_GUMBEL and a.T != 0.0:
        g = a.noise[a.noise_row[slots]]
        s = oacc.gumbel_scores(l32, g, a.T).astype(np.float64)
        eps = bound / np.float32(a.T) + 2.0 ** -22 * (np.abs(l32 / np.float32(a.T)) + np.abs(s))
    else:
        s = l32.astype(np.float64)
        eps = bound
    want = np.argmax(s, axis=1)
    got = tokens[slots]
    assert np.all((got >= 0) & (got < a.V))
    differ = np.nonzero(got != want)[0]
    for r in differ:
        t, u = int(want[r]), int(got[r])
        assert s[r, t] - s[r, u] <= eps[r, t] + eps[r, u], \
            f"row {r}: device {u} ({s[r, u]}), oracle {t} ({s[r, t]}), bound {eps[r, t] + eps[r, u]}"
    assert len(differ) <= max(1, len(slots) // 100), f"{len(differ)} of {len(slots)} rows took another token"
    return len(differ)


DECISION_CASES = {
    # (mode, T, V, hidden, rows)
    "argmax_small": (oacc.MODE_ARGMAX, 0.0, 300, 64, 5),           # V % 16 != 0: masked tail columns
    "argmax_two_tiles": (oacc.MODE_ARGMAX, 0.0, 5000, 256, 130),   # ragged second M-tile
    "argmax_odd_vocab": (oacc.MODE_ARGMAX, 0.0, 4099, 128, 40),    # V % 4 != 0
    "gumbel_odd_vocab": (oacc.MODE_GUMBEL, 0.7, 4099, 128, 40),    # scalar noise loads
    "gumbel_vec": (oacc.MODE_GUMBEL, 1.0, 8192, 512, 257),         # 3 M-tiles
    "argmax_full_vocab": (oacc.MODE_ARGMAX, 0.0, 151936, 2048, 64),
    "gumbel_full_vocab": (oacc.MODE_GUMBEL, 1.5, 151936, 1024, 96),
    "argmax_many_tiles": (oacc.MODE_ARGMAX, 0.0, 32768, 4096, 1030),  # 9 M-tiles, K = 4096
    "argmax_tiny_vocab": (oacc.MODE_ARGMAX, 0.0, 100, 64, 3),          # one 112-column piece, one CTA
    "gumbel_max_slots": (oacc.MODE_GUMBEL, 1.0, 512, 64, 2048),        # 2048 sequences: 16 M-tiles
}


@pytest.mark.parametrize("name", list(DECISION_CASES))
def test_lmhead_decisions(name):
    mode, T, V, hidden, rows = DECISION_CASES[name]
    x = _decision_inputs(mode, T, V, hidden, rows, 700 + len(name))
    n_acc, n_out, tokens = _run(x)
    assert np.all(n_acc == 0) and np.all(n_out == 1)
    _check_decisions(x, tokens)


def _check_exact(x, got, seqs=None):
    n_acc, n_out, tokens = got
    ref = olm.accept_lmhead(x)
    assert n_acc.tolist() == ref["n_acc"].tolist()
    assert n_out.tolist() == ref["n_out"].tolist()
    for b in range(len(x.acc.blocks)):
        off, no = int(x.acc.slot_off[b]), int(n_out[b])
        assert tokens[off:off + no].tolist() == ref["tokens"][off:off + no].tolist()
    return ref


PLANTED_CASES = {
    # (mode, T, V, hidden, blocks, gammas)
    "argmax_mixed": (oacc.MODE_ARGMAX, 0.0, 2000, 128, [1, 4, 8, 16, 32, 64, 3], [1, 4, 5, 16, 10, 64, 0]),
    "gumbel_mixed": (oacc.MODE_GUMBEL, 1.5, 3000, 256, [8, 8, 33, 64, 2], [8, 3, 33, 20, 1]),
    "argmax_straddle": (oacc.MODE_ARGMAX, 0.0, 1000, 64, [60, 60, 60, 60], [60, 59, 30, 0]),  # sequences across M-tiles
}


@pytest.mark.parametrize("name", list(PLANTED_CASES))
def test_lmhead_planted(name):
    mode, T, V, hidden, blocks, gammas = PLANTED_CASES[name]
    x = W.make_lmhead_inputs("pl", mode, T, V, hidden, blocks, gammas, 800 + len(name))
    ref = _check_exact(x, _run(x))
    assert max(ref["n_acc"]) > 0  # the planted prefixes are accepted


def test_lmhead_workspace_reuse():
    """Counters are left zero: a second call on the same workspace agrees."""
    import torch
    x = W.make_lmhead_inputs("re", oacc.MODE_GUMBEL, 1.0, 2500, 128, [5, 9, 64, 1], [5, 4, 40, 0], 901)
    d = sio.lmhead_to_device(x)
    a = ssv.lmhead_args(d["mode"], d["T"], d["h"], d["w"], d["draft_tokens"], d["tau"], d["block"], d["gamma"],
                        d["slot_off"], d["draft_tokens"], d["draft_tokens"], d["draft_tokens"], d["noise"],
                        d["noise_row"])
    ws = torch.zeros(ssv.lmhead_accept_workspace_bytes(a), dtype=torch.uint8, device="cuda")
    first = _run(x, workspace=ws, d=d)
    counters = ws[:256].clone()
    second = _run(x, workspace=ws, d=d)
    for u, v in zip(first, second):
        assert np.array_equal(u, v)
    assert int(counters.count_nonzero()) == 0 and int(ws[:256].count_nonzero()) == 0
    _check_exact(x, second)


def _subset(x: W.LmheadInputs, seqs):
    """The chosen sequences of x, repacked (LM head and noise table shared)."""
    a = x.acc
    blocks = a.blocks[seqs]
    slots = np.concatenate([np.arange(a.slot_off[b], a.slot_off[b] + a.blocks[b]) for b in seqs])
    slot_off = np.concatenate([[0], np.cumsum(blocks)[:-1]]).astype(np.int32)
    acc = W.AcceptInputs(a.name, a.mode, a.T, a.V, a.logits_dtype, blocks, a.gammas[seqs], slot_off,
                         a.tau[slots], None, None, a.draft_tokens[slots], a.noise, a.noise_row[slots],
                         a.u_accept[slots], a.u_sample[seqs])
    return W.LmheadInputs(acc, x.hidden, x.h[slots], x.w)


@pytest.mark.parametrize("workload", ["gqa1p7b", "gqa8b", "sweep"])
def test_lmhead_workloads(workload):
    """Full-size workloads through the device; the oracle checks every
    sequence (gqa1p7b) or a seeded sample of sequences (the rest), which the
    rule treats independently."""
    x = W.workload_lmhead(workload)
    got = _run(x)
    batch = len(x.acc.blocks)
    rng = np.random.default_rng(17)
    seqs = np.arange(batch) if batch <= 8 else np.sort(rng.choice(batch, size=6, replace=False))
    sub = _subset(x, seqs)
    n_acc, n_out, tokens = got
    sub_tokens = np.concatenate([tokens[x.acc.slot_off[b]:x.acc.slot_off[b] + x.acc.blocks[b]] for b in seqs])
    ref = _check_exact(sub, (n_acc[seqs], n_out[seqs], sub_tokens))
    assert ref["n_acc"].sum() > 0


@pytest.mark.parametrize("fault", ["bad_tau", "noise_row"])
def test_lmhead_rejects_one_sequence(fault):
    import torch
    x = W.make_lmhead_inputs("f", oacc.MODE_GUMBEL, 1.0, 1500, 64, [6, 5, 7], [6, 2, 3], 902)
    bad = 1
    off = int(x.acc.slot_off[bad])
    if fault == "bad_tau":
        x.acc.tau[off + 1] = x.acc.tau[off]
        want = ssv.SSV_ERR_BAD_TAU
    else:
        x.acc.noise_row[off + int(np.nonzero(x.acc.tau[off:off + 5] == 1)[0][0])] = 10 ** 6
        want = ssv.SSV_ERR_INVALID
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_acc, n_out, tokens = _run(x, dev_status=status)
    assert ssv.get_status(status) == want
    keep = [0, 2]
    sub = _subset(x, np.array(keep))
    sub_tokens = np.concatenate([tokens[x.acc.slot_off[b]:x.acc.slot_off[b] + x.acc.blocks[b]] for b in keep])
    _check_exact(sub, (n_acc[keep], n_out[keep], sub_tokens))


def test_lmhead_host_errors():
    import torch
    x = W.make_lmhead_inputs("h", oacc.MODE_ARGMAX, 0.0, 500, 64, [4, 4], [4, 2], 903)
    d = sio.lmhead_to_device(x)
    outs = [torch.full((2,), 77, dtype=torch.int32, device="cuda"),
            torch.full((2,), 77, dtype=torch.int32, device="cuda"),
            torch.full((8,), 77, dtype=torch.int32, device="cuda")]

    def args():
        return ssv.lmhead_args(d["mode"], d["T"], d["h"], d["w"], d["draft_tokens"], d["tau"], d["block"],
                               d["gamma"], d["slot_off"], *outs)

    ws = torch.zeros(max(256, ssv.lmhead_accept_workspace_bytes(args())), dtype=torch.uint8, device="cuda")

    def call(a, wsb=None):
        return int(ssv.lib().ssv_lmhead_accept(ssv.C.byref(a), ws.data_ptr(), ws.numel() if wsb is None else wsb,
                                               ssv._stream_ptr(None)))

    a = args(); a.mode = ssv.REJECT
    assert call(a) == ssv.SSV_ERR_INVALID
    a = args(); a.hidden = 96
    assert call(a) == ssv.SSV_ERR_INVALID
    a = args(); a.T = float("nan")
    assert call(a) == ssv.SSV_ERR_NOT_FINITE
    a = args(); a.total_slots = 4096
    assert call(a) == ssv.SSV_ERR_UNSUPPORTED
    a = args(); a.lm_head = a.lm_head + 2
    assert call(a) == ssv.SSV_ERR_INVALID
    a = args(); a.mode = ssv.GUMBEL; a.T = 1.0
    assert call(a) == ssv.SSV_ERR_INVALID        # coupled noise without a table
    assert call(args(), wsb=16) == ssv.SSV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert all(int(t[0].item()) == 77 for t in outs)   # nothing was launched
    a = args(); a.batch = 0
    assert call(a) == ssv.SSV_OK
    assert call(args()) == ssv.SSV_OK
    torch.cuda.synchronize()
    _check_exact(x, tuple(t.cpu().numpy() for t in outs))
