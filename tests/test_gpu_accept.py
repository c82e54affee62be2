"""GPU parity of ssv_accept against the oracle (SimSD summary section 4;
SPOT review, "How it is used").  Every mode is bit-exact on n_acc, n_out
and every token.  Greedy and coupled-noise acceptance compare identical fp32
scores.  Rejection sampling: each accept test's log-ratio margin exceeds the
fp32 rounding band of the device's ratio, and each emitted sample's threshold
u'Z lies farther from a CDF boundary than the double-float band of the
device's weights plus the oracle's fp64 summation bound (both derived in
gpu_common); the seeded sets are asserted to contain no decision inside a
band, so the emitted token is unique."""
import numpy as np
import pytest
import torch

from diffusion_speculative_verification_gb300 import workloads as W, ssv
from gpu_common import ensure_built, gpu_accept, compare_accept

pytestmark = pytest.mark.gpu


def setup_module():
    ensure_built()


@pytest.mark.parametrize("which", [0, 1])
def test_tiny(which):
    x = W.workload_accept("tiny", which)
    compare_accept(x, gpu_accept(x))


def test_gqa1p7b_argmax():
    x = W.workload_accept("gqa1p7b")
    compare_accept(x, gpu_accept(x))


def test_gqa8b_reject():
    x = W.workload_accept("gqa8b")
    worst = compare_accept(x, gpu_accept(x))
    assert worst > 1.0


@pytest.fixture(scope="module")
def sweep_inputs():
    return W.workload_accept("sweep", 1)


@pytest.mark.parametrize("T", [0.0, 1.0, 1.5])
def test_sweep_gumbel(sweep_inputs, T):
    x = sweep_inputs
    x.T = T
    compare_accept(x, gpu_accept(x))


EDGE = {
    "gamma0": dict(mode=W.MODE_ARGMAX, T=0.0, V=5000, blocks=[4, 1], gammas=[0, 0]),
    "B1": dict(mode=W.MODE_GUMBEL, T=1.0, V=4097, blocks=[1, 1, 1], gammas=[1, 0, 1]),
    "V1": dict(mode=W.MODE_ARGMAX, T=0.0, V=1, blocks=[3], gammas=[3]),
    "B64": dict(mode=W.MODE_GUMBEL, T=0.7, V=12345, blocks=[64, 2], gammas=[64, 1]),
    "reject_bonus": dict(mode=W.MODE_REJECT, T=1.0, V=9000, blocks=[8, 8, 4], gammas=[3, 8, 1]),
    "reject_T07": dict(mode=W.MODE_REJECT, T=0.7, V=20000, blocks=[16] * 6, gammas=[16] * 6),
    "bf16_logits": dict(mode=W.MODE_GUMBEL, T=1.5, V=30000, blocks=[8, 4], gammas=[8, 2], logits_dtype=W.BF16),
    "bf16_reject": dict(mode=W.MODE_REJECT, T=1.0, V=30000, blocks=[8, 4], gammas=[5, 2], logits_dtype=W.BF16),
}


@pytest.mark.parametrize("name", list(EDGE))
def test_edge_cases(name):
    kw = dict(EDGE[name])
    x = W.make_accept_inputs(name, kw.pop("mode"), kw.pop("T"), kw.pop("V"), kw.pop("blocks"), kw.pop("gammas"),
                             seed=sum(map(ord, name)), **kw)
    compare_accept(x, gpu_accept(x))


def test_ties_resolve_to_lowest_index():
    x = W.make_accept_inputs("ties", W.MODE_ARGMAX, 0.0, 10000, [4], [4], seed=5)
    x.logits[:] = 0.0
    x.logits[:, [17, 4000, 9999]] = 3.0
    n_acc, n_out, tokens = gpu_accept(x)
    compare_accept(x, (n_acc, n_out, tokens))
    assert tokens[0] in (17, x.draft_tokens[np.argmin(x.tau)])


def test_bad_tau_reports_status():
    x = W.make_accept_inputs("bad", W.MODE_ARGMAX, 0.0, 100, [4], [4], seed=6)
    x.tau[:] = [1, 2, 2, 4]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_accept(x, dev_status=st)
    assert ssv.get_status(st) == ssv.SSV_ERR_BAD_TAU


def test_repeated_calls_share_workspace():
    """The arrival counters return to zero, so one workspace serves many calls."""
    x = W.workload_accept("tiny", 1)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        compare_accept(x, gpu_accept(x, workspace=ws))
    assert int(ws[:256].sum()) == 0


def test_reject_sequence_rejected_after_an_emitting_call():
    """Rejection sampling, one workspace for two calls: the first emits a token
    for every sequence; in the second, sequence 1's stage map is not a
    permutation.  Its emission record from the first call must not be acted
    on: its outputs stay untouched, SSV_ERR_BAD_TAU is raised, and the other
    sequences still match the oracle bit for bit."""
    from diffusion_speculative_verification_gb300 import io as sio
    import oracle.accept as oacc
    x = W.make_accept_inputs("stale", W.MODE_REJECT, 1.0, 9000, [8, 8, 4], [6, 7, 3], seed=103)
    ws = torch.zeros(1 << 24, dtype=torch.uint8, device="cuda")
    first = gpu_accept(x, workspace=ws)
    compare_accept(x, first)
    ref = oacc.accept_batch(x)
    assert all(int(r.n_out) > int(r.n_acc) for r in ref["results"]), "every sequence should emit; pick another seed"
    assert ref["results"][1].emit_kind == "residual", "sequence 1 should sample the residual; pick another seed"
    d = sio.accept_to_device(x)
    tau = d["tau"].clone()
    tau[8:16] = torch.tensor([1, 2, 2, 4, 5, 6, 7, 8], dtype=torch.int32)
    out = (torch.full((3,), -7, dtype=torch.int32, device="cuda"), torch.full((3,), -7, dtype=torch.int32, device="cuda"),
           torch.full((20,), -7, dtype=torch.int32, device="cuda"))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_acc, n_out, tokens = ssv.accept(d["mode"], d["T"], d["logits"], d["draft_tokens"], tau, d["block"], d["gamma"],
                                      d["slot_off"], draft_logits=d["draft_logits"], u_accept=d["u_accept"],
                                      u_sample=d["u_sample"], max_block=d["max_block"], dev_status=st,
                                      workspace=ws, out=out)
    n_acc, n_out, tokens = n_acc.cpu().numpy(), n_out.cpu().numpy(), tokens.cpu().numpy()
    assert ssv.get_status(st) == ssv.SSV_ERR_BAD_TAU
    assert n_acc[1] == -7 and n_out[1] == -7 and np.all(tokens[8:16] == -7)
    for b, (off, B) in ((0, (0, 8)), (2, (16, 4))):
        r = ref["results"][b]
        assert n_acc[b] == r.n_acc and n_out[b] == r.n_out
        np.testing.assert_array_equal(tokens[off:off + B], first[2][off:off + B])


def _accept_with_logits_offset(x: W.AcceptInputs, elem_offset: int, dev_status=None):
    """Runs ssv_accept with the logits (and draft logits) stored `elem_offset`
    elements into a larger buffer, so that rows are not 16-byte aligned."""
    from diffusion_speculative_verification_gb300 import io as sio
    d = sio.accept_to_device(x)

    def shifted(t):
        if t is None:
            return None
        buf = torch.zeros(t.numel() + 16, dtype=t.dtype, device=t.device)
        v = buf[elem_offset:elem_offset + t.numel()].view(t.shape)
        v.copy_(t)
        return v

    n_acc, n_out, tokens = ssv.accept(d["mode"], d["T"], shifted(d["logits"]), d["draft_tokens"], d["tau"],
                                      d["block"], d["gamma"], d["slot_off"], draft_logits=shifted(d["draft_logits"]),
                                      noise=d["noise"], noise_row=d["noise_row"], u_accept=d["u_accept"],
                                      u_sample=d["u_sample"], max_block=d["max_block"], dev_status=dev_status,
                                      noise_seed=d["noise_seed"])
    return n_acc.cpu().numpy(), n_out.cpu().numpy(), tokens.cpu().numpy()


UNALIGNED = {
    "argmax_f32": dict(mode=W.MODE_ARGMAX, T=0.0, V=20000, blocks=[8, 16, 4], gammas=[8, 12, 4]),
    "gumbel_f32": dict(mode=W.MODE_GUMBEL, T=1.0, V=20000, blocks=[8, 16, 4], gammas=[8, 16, 2]),
    "reject_bf16": dict(mode=W.MODE_REJECT, T=1.0, V=30000, blocks=[8, 4, 16], gammas=[5, 2, 16],
                        logits_dtype=W.BF16),
}


@pytest.mark.parametrize("name", list(UNALIGNED))
def test_rows_not_16b_aligned(name):
    """Rows that bulk copies cannot address (offset by one element) go
    through the general kernel; the results are the same."""
    kw = dict(UNALIGNED[name])
    x = W.make_accept_inputs(name, kw.pop("mode"), kw.pop("T"), kw.pop("V"), kw.pop("blocks"), kw.pop("gammas"),
                             seed=sum(map(ord, name)) + 3, **kw)
    aligned = gpu_accept(x)
    shifted = _accept_with_logits_offset(x, 1)
    compare_accept(x, aligned)
    compare_accept(x, shifted)
    assert np.array_equal(aligned[0], shifted[0]) and np.array_equal(aligned[1], shifted[1])


def test_many_slots_general_kernel():
    """More slots than the streaming kernel lists (2048) take the general kernel."""
    blocks = [4] * 530  # 2120 slots
    gammas = [int(g) for g in np.random.default_rng(11).integers(0, 5, size=len(blocks))]
    x = W.make_accept_inputs("many", W.MODE_ARGMAX, 0.0, 640, blocks, gammas, seed=12)
    compare_accept(x, gpu_accept(x))


def test_reject_more_sequences_than_one_emission_list():
    """Rejection sampling over 2100 sequences (4200 slots, the general reduce):
    the emission passes list the emitting sequences 2048 at a time, and the
    emission records are cleared before the walks; every token bit-exact."""
    blocks = [2] * 2100
    gammas = [int(g) for g in np.random.default_rng(22).integers(0, 3, size=len(blocks))]
    x = W.make_accept_inputs("manyrej", W.MODE_REJECT, 1.0, 256, blocks, gammas, seed=22)
    compare_accept(x, gpu_accept(x))


def test_reject_vocabulary_of_74_chunks():
    """Rejection sampling at V = 600000: 74 vocabulary chunks (the row merge
    holds 64 per warp and reads the rest again) and 296 emission sub-chunks
    (the normaliser and locating scans run in three blocks); a residual and
    two bonus samples, every token bit-exact."""
    x = W.make_accept_inputs("bigV", W.MODE_REJECT, 1.0, 600000, [4, 3, 2], [3, 3, 1], seed=33)
    compare_accept(x, gpu_accept(x))


@pytest.mark.parametrize("V", [4096, 4097])
def test_bad_noise_row_reports_status(V):
    x = W.make_accept_inputs("badnoise", W.MODE_GUMBEL, 1.0, V, [4, 4], [4, 4], seed=13)
    x.noise_row[1] = x.noise.shape[0] + 5
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_accept(x, dev_status=st)
    assert ssv.get_status(st) == ssv.SSV_ERR_INVALID


def _random_accept(seed):
    """Seeded random batch: mode and temperature, vocabulary size (rows 16-byte
    aligned or not), 1..12 sequences with B in 1..64 and gamma in 0..B, fp32 or
    bf16 logits."""
    rng = np.random.default_rng(seed)
    mode = int(rng.choice([W.MODE_ARGMAX, W.MODE_GUMBEL, W.MODE_REJECT]))
    T = {W.MODE_ARGMAX: 0.0, W.MODE_GUMBEL: float(rng.choice([0.0, 0.7, 1.0, 1.5])),
         W.MODE_REJECT: float(rng.choice([0.7, 1.0, 1.3]))}[mode]
    V = int(rng.choice([int(rng.integers(1, 3000)), int(rng.integers(3000, 40000)), 8 * int(rng.integers(500, 5000))]))
    batch = int(rng.integers(1, 13))
    blocks = [int(rng.integers(1, 65)) for _ in range(batch)]
    gammas = [int(rng.integers(0, b + 1)) for b in blocks]
    dt = W.BF16 if rng.random() < 0.3 else W.F32
    return W.make_accept_inputs(f"random{seed}", mode, T, V, blocks, gammas, seed=3000 + seed, logits_dtype=dt)


@pytest.mark.parametrize("seed", range(10))
def test_accept_random(seed):
    compare_accept(_random_accept(seed), gpu_accept(_random_accept(seed)))
