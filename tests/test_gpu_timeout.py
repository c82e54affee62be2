"""Failure detection on the device, without a GPU fault: a bounded wait
that runs out.

ssv_set_fault_injection makes CTA 0 of one kernel leave out one
asynchronous copy and shortens that kernel's wait budget to 2e5 SM cycles
(about 0.1 ms).  The wait for the missing copy runs out; the kernel must
drain what it issued, release its tensor memory, write SSV_ERR_TIMEOUT and
return -- no trap, no fault, no unbounded wait.  A normal call afterwards,
on the same workspace once cleared (the header's rule after a timeout),
must then match the oracle, which shows the context and the SMs' tensor
memory are intact.  Covered: the tensor-core attention, the streaming
acceptance reduce and the fused LM head's GEMM."""
import numpy as np
import pytest
import torch

from diffusion_speculative_verification_gb300 import ssv, workloads as W, io as sio
import oracle.attention as oattn
import oracle.lmhead as olm
from gpu_common import ensure_built, gpu_rope, compare_attn, compare_accept

pytestmark = pytest.mark.gpu

BUDGET = 200_000


def setup_module():
    ensure_built()


def teardown_function():
    ssv.set_fault_injection(None)


@pytest.mark.parametrize("skip", [0, 5])
def test_attention_wait_runs_out(skip):
    # 24 sequences x 8 kv heads: each CTA holds several key blocks (CTA 0 at least 6),
    # and units split across CTAs make other CTAs wait for CTA 0's partials too
    a = W.make_attn_inputs("t", [1024] * 23 + [700], [0] * 23 + [40], [8] * 23 + [4], 16, 8, 128, W.BF16, 81)
    qo, ko, t = gpu_rope(a)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.empty(t["q"].shape, dtype=torch.float32, device="cuda")
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    ssv.set_fault_injection(ssv.FAULT_ATTN, skip, BUDGET)
    ssv.verify_attn(qo, t["k_cache"], t["v_cache"], ko, t["v_new"], t["batch"], t["tau"], out=o, workspace=ws,
                    dev_status=st)
    assert ssv.get_status(st) == ssv.SSV_ERR_TIMEOUT
    ssv.set_fault_injection(None)
    ws.zero_()
    ssv.verify_attn(qo, t["k_cache"], t["v_cache"], ko, t["v_new"], t["batch"], t["tau"], out=o, workspace=ws,
                    dev_status=st)
    assert ssv.get_status(st) == ssv.SSV_OK
    got = o.cpu().numpy().astype(np.float64)
    ref = oattn.verify_attention(a.seqs, a.tau, W.values_f64(sio.to_numpy_storage(qo), a.dtype),
                                 W.values_f64(a.k_cache, a.dtype), W.values_f64(a.v_cache, a.dtype),
                                 W.values_f64(sio.to_numpy_storage(ko), a.dtype), W.values_f64(a.v_new, a.dtype))
    compare_attn(got, ref, False, False)


@pytest.mark.parametrize("mode", [W.MODE_ARGMAX, W.MODE_REJECT])
def test_acceptance_wait_runs_out(mode):
    T = 0.0 if mode == W.MODE_ARGMAX else 1.0
    x = W.make_accept_inputs("t", mode, T, 65536, [8] * 6, [8, 8, 5, 8, 3, 8], seed=82)
    d = sio.accept_to_device(x)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(16 << 20, dtype=torch.uint8, device="cuda")

    def run():
        return ssv.accept(d["mode"], d["T"], d["logits"], d["draft_tokens"], d["tau"], d["block"], d["gamma"],
                          d["slot_off"], draft_logits=d["draft_logits"], noise=d["noise"], noise_row=d["noise_row"],
                          u_accept=d["u_accept"], u_sample=d["u_sample"], max_block=d["max_block"], dev_status=st,
                          workspace=ws)

    ssv.set_fault_injection(ssv.FAULT_ACCEPT, 0, BUDGET)
    run()
    assert ssv.get_status(st) == ssv.SSV_ERR_TIMEOUT
    ssv.set_fault_injection(None)
    ws.zero_()
    n_acc, n_out, tokens = run()
    assert ssv.get_status(st) == ssv.SSV_OK
    compare_accept(x, (n_acc.cpu().numpy(), n_out.cpu().numpy(), tokens.cpu().numpy()))


@pytest.mark.parametrize("skip", [0, 3])
def test_lmhead_wait_runs_out(skip):
    x = W.make_lmhead_inputs("t", W.MODE_ARGMAX, 0.0, 8192, 512, [4, 8, 2, 6], [4, 5, 2, 6], 83)
    d = sio.lmhead_to_device(x)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(32 << 20, dtype=torch.uint8, device="cuda")

    def run():
        return ssv.lmhead_accept(d["mode"], d["T"], d["h"], d["w"], d["draft_tokens"], d["tau"], d["block"],
                                 d["gamma"], d["slot_off"], noise=d["noise"], noise_row=d["noise_row"],
                                 dev_status=st, workspace=ws)

    ssv.set_fault_injection(ssv.FAULT_LMHEAD, skip, BUDGET)
    run()
    assert ssv.get_status(st) == ssv.SSV_ERR_TIMEOUT
    ssv.set_fault_injection(None)
    ws.zero_()
    n_acc, n_out, tokens = run()
    assert ssv.get_status(st) == ssv.SSV_OK
    ref = olm.accept_lmhead(x)
    assert np.array_equal(n_acc.cpu().numpy(), ref["n_acc"]) and np.array_equal(n_out.cpu().numpy(), ref["n_out"])
    assert np.array_equal(tokens.cpu().numpy(), ref["tokens"])


def test_setting_is_validated_and_scoped():
    with pytest.raises(ssv.SsvError):
        ssv.set_fault_injection(ssv.FAULT_ATTN, -2, BUDGET)
    with pytest.raises(ssv.SsvError):
        ssv.set_fault_injection(7, 0, BUDGET)
    with pytest.raises(ssv.SsvError):
        ssv.set_fault_injection(ssv.FAULT_ATTN, 0, 10)
    # a setting for one kernel leaves the others alone
    ssv.set_fault_injection(ssv.FAULT_LMHEAD, 0, BUDGET)
    x = W.make_accept_inputs("s", W.MODE_ARGMAX, 0.0, 65536, [8] * 3, [8] * 3, seed=84)
    d = sio.accept_to_device(x)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_acc, n_out, tokens = ssv.accept(d["mode"], d["T"], d["logits"], d["draft_tokens"], d["tau"], d["block"],
                                      d["gamma"], d["slot_off"], max_block=d["max_block"], dev_status=st)
    assert ssv.get_status(st) == ssv.SSV_OK
    compare_accept(x, (n_acc.cpu().numpy(), n_out.cpu().numpy(), tokens.cpu().numpy()))
