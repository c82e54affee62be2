"""ssv_verify_step (rotation, verification attention and acceptance in one
call, with programmatic dependent launch between the kernels) against the
three separate calls and against the oracle (SimSD summary sections 2-4)."""
import numpy as np
import pytest
import torch

from diffusion_speculative_verification_gb300 import workloads as W, ssv, io as sio
import oracle.attention as oattn
from gpu_common import ensure_built, compare_attn, compare_accept, random_attn_shape

pytestmark = pytest.mark.gpu

ACC_INDEX = {"tiny": 1, "gqa1p7b": 0, "gqa8b": 0, "sweep": 1}


def setup_module():
    ensure_built()


def _prepare(name):
    a = W.workload_attn(name)
    x = W.workload_accept(name, ACC_INDEX[name])
    t = sio.attn_to_device(a)
    acc = sio.accept_to_device(x)
    return a, x, t, acc


def _run(a, x, t, acc, fused):
    dev = t["q"].device
    qo, ko = torch.empty_like(t["q"]), torch.empty_like(t["k_new"])
    o = torch.empty(t["q"].shape, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = (torch.full((x.batch,), -7, dtype=torch.int32, device=dev),
            torch.full((x.batch,), -7, dtype=torch.int32, device=dev),
            torch.full((len(x.tau),), -7, dtype=torch.int32, device=dev))
    ra = ssv.rope_args(t["q"], t["k_new"], t["batch"], a.rope_base, q_out=qo, k_out=ko)
    aa = ssv.attn_args(qo, t["k_cache"], t["v_cache"], ko, t["v_new"], o, t["batch"], t["tau"], 0.0, st)
    ca = ssv.accept_args(acc["mode"], acc["T"], acc["logits"], acc["draft_tokens"], acc["tau"], acc["block"],
                         acc["gamma"], acc["slot_off"], *outs, acc["draft_logits"], acc["noise"], acc["noise_row"],
                         acc["u_accept"], acc["u_sample"], acc["max_block"], st)
    wa = torch.zeros(max(256, ssv.verify_attn_workspace_bytes(aa)), dtype=torch.uint8, device=dev)
    wc = torch.zeros(ssv.accept_workspace_bytes(ca), dtype=torch.uint8, device=dev)
    if fused:
        for _ in range(2):  # twice: the workspaces must come back clean
            ssv.verify_step(ra, aa, wa, ca, wc)
    else:
        L = ssv.lib()
        import ctypes as C
        assert L.ssv_rope_copy(C.byref(ra), None) == 0
        assert L.ssv_verify_attn(C.byref(aa), wa.data_ptr(), wa.numel(), None) == 0
        assert L.ssv_accept(C.byref(ca), wc.data_ptr(), wc.numel(), None) == 0
    assert ssv.get_status(st) == ssv.SSV_OK
    return o.cpu().numpy(), tuple(v.cpu().numpy() for v in outs), (qo, ko)


@pytest.mark.parametrize("name", ["tiny", "gqa1p7b", "gqa8b"])
def test_step_matches_separate_calls(name):
    a, x, t, acc = _prepare(name)
    o_f, r_f, _ = _run(a, x, t, acc, True)
    o_s, r_s, _ = _run(a, x, t, acc, False)
    assert np.array_equal(o_f, o_s)
    for u, v in zip(r_f, r_s):
        assert np.array_equal(u, v)


def test_step_against_oracle_gqa1p7b():
    """Attention against the oracle on the step's own rotated bytes (the
    rotation itself is checked against the oracle in the rotation tests)."""
    a, x, t, acc = _prepare("gqa1p7b")
    o, res, (qo, ko) = _run(a, x, t, acc, True)
    q64 = W.values_f64(sio.to_numpy_storage(qo), a.dtype)
    k64 = W.values_f64(sio.to_numpy_storage(ko), a.dtype)
    ref = oattn.verify_attention(a.seqs, a.tau, q64, W.values_f64(a.k_cache, a.dtype),
                                 W.values_f64(a.v_cache, a.dtype), k64, W.values_f64(a.v_new, a.dtype))
    compare_attn(o.astype(np.float64), ref, False, False)
    compare_accept(x, res)


def test_step_without_rotation_or_acceptance():
    a, x, t, acc = _prepare("tiny")
    dev = t["q"].device
    o1 = torch.empty(t["q"].shape, dtype=torch.float32, device=dev)
    o2 = torch.empty_like(o1)
    aa1 = ssv.attn_args(t["q"], t["k_cache"], t["v_cache"], t["k_new"], t["v_new"], o1, t["batch"], t["tau"])
    aa2 = ssv.attn_args(t["q"], t["k_cache"], t["v_cache"], t["k_new"], t["v_new"], o2, t["batch"], t["tau"])
    wa = torch.zeros(max(256, ssv.verify_attn_workspace_bytes(aa1)), dtype=torch.uint8, device=dev)
    ssv.verify_step(None, aa1, wa)
    import ctypes as C
    assert ssv.lib().ssv_verify_attn(C.byref(aa2), wa.data_ptr(), wa.numel(), None) == 0
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def _prepare_random(seed):
    """Random batch (shared generator) with coupled-noise acceptance over the
    same sequences and stage maps."""
    a = random_attn_shape(300 + seed)
    blocks = [int(s[2]) for s in a.seqs]
    rng = np.random.default_rng(seed)
    gammas = [int(rng.integers(0, b + 1)) for b in blocks]
    x = W.make_accept_inputs(f"step{seed}", W.MODE_GUMBEL, 1.0, 4000 + 8 * seed, blocks, gammas, seed=4000 + seed,
                             tau=a.tau)
    return a, x, sio.attn_to_device(a), sio.accept_to_device(x)


@pytest.mark.parametrize("seed", range(3))
def test_step_random_against_separate_calls_and_oracle(seed):
    a, x, t, acc = _prepare_random(seed)
    o_f, r_f, (qo, ko) = _run(a, x, t, acc, True)
    o_s, r_s, _ = _run(a, x, t, acc, False)
    assert np.array_equal(o_f, o_s)
    for u, v in zip(r_f, r_s):
        assert np.array_equal(u, v)
    q64 = W.values_f64(sio.to_numpy_storage(qo), a.dtype)
    k64 = W.values_f64(sio.to_numpy_storage(ko), a.dtype)
    ref = oattn.verify_attention(a.seqs, a.tau, q64, W.values_f64(a.k_cache, a.dtype),
                                 W.values_f64(a.v_cache, a.dtype), k64, W.values_f64(a.v_new, a.dtype))
    compare_attn(o_f.astype(np.float64), ref, False, False)
    compare_accept(x, r_f)
