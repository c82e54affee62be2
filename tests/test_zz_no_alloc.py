"""ssv_accept_noalloc: acceptance for callers that cannot allocate device memory.

Some callers have no allocator of their own (a host runtime that owns all
GPU memory, or a path where cudaMalloc is not allowed), so this entry point
takes no workspace and uses the library's fixed 4 MiB per-device scratch
array instead.  These tests call it through the C ABI and check that, on
two calls in a row, it returns exactly what ssv_accept (caller workspace)
returns on the same inputs -- the acceptance tests' tolerance, which is
bit-exact for lengths and tokens -- that a call after one that timed out
(leaving arrival counters non-zero in the shared array) is again exact, and
that a call too large for the array is refused before anything is launched.

Kept in a file of its own that sorts last, so a run that stops at the
first failure has executed every other test before this one.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from diffusion_speculative_verification_gb300 import ssv, io as sio, workloads as W
from gpu_common import ensure_built

pytestmark = pytest.mark.gpu


def _outputs(x):
    dev = "cuda"
    return (torch.full((x.batch,), -7, dtype=torch.int32, device=dev),
            torch.full((x.batch,), -7, dtype=torch.int32, device=dev),
            torch.full((len(x.tau),), -7, dtype=torch.int32, device=dev))


def _args(d, x, out, status):
    return ssv.accept_args(d["mode"], d["T"], d["logits"], d["draft_tokens"], d["tau"], d["block"], d["gamma"],
                           d["slot_off"], *out, d["draft_logits"], d["noise"], d["noise_row"], d["u_accept"],
                           d["u_sample"], d["max_block"], status)


def _run_workspace_path(d, x):
    out = _outputs(x)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = _args(d, x, out, status)
    ws = torch.zeros(ssv.accept_workspace_bytes(a), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert ssv.lib().ssv_accept(C.byref(a), ws.data_ptr(), ws.numel(), stream) == ssv.SSV_OK
    assert ssv.get_status(status) == ssv.SSV_OK
    return [t.cpu().numpy() for t in out]


def _run_noalloc(d, x):
    out = _outputs(x)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = _args(d, x, out, status)
    stream = torch.cuda.current_stream().cuda_stream
    assert ssv.lib().ssv_accept_noalloc(C.byref(a), stream) == ssv.SSV_OK
    assert ssv.get_status(status) == ssv.SSV_OK
    return [t.cpu().numpy() for t in out]


CASES = [
    ("gqa8b_reject", lambda: W.workload_accept("gqa8b")),
    ("gumbel_T1.5", lambda: W.make_accept_inputs("g", W.MODE_GUMBEL, 1.5, 30000, [8, 32, 4, 16], [8, 20, 4, 3],
                                                 seed=71)),
    ("argmax_bf16", lambda: W.make_accept_inputs("a", W.MODE_ARGMAX, 0.0, 151936, [8] * 8, [8] * 8, seed=72,
                                                 logits_dtype=W.BF16)),
]


def test_noalloc_matches_workspace_path_two_calls_in_a_row():
    ensure_built()
    for name, make in CASES:
        x = make()
        d = sio.accept_to_device(x)
        want = _run_workspace_path(d, x)
        first = _run_noalloc(d, x)
        second = _run_noalloc(d, x)
        for w, f, s in zip(want, first, second):
            np.testing.assert_array_equal(f, w, err_msg=name)
            np.testing.assert_array_equal(s, w, err_msg=name)


def test_noalloc_recovers_from_counters_left_non_zero():
    """A call whose reduce times out (a left-out copy, ssv_set_fault_injection)
    leaves arrival counters non-zero in the shared array; the next call clears
    them itself and again returns what the workspace path returns."""
    ensure_built()
    x = W.make_accept_inputs("c", W.MODE_ARGMAX, 0.0, 65536, [8] * 6, [8, 8, 5, 8, 3, 8], seed=73)
    d = sio.accept_to_device(x)
    want = _run_workspace_path(d, x)
    out = _outputs(x)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = _args(d, x, out, status)
    stream = torch.cuda.current_stream().cuda_stream
    try:
        ssv.set_fault_injection(ssv.FAULT_ACCEPT, 0, 200_000)
        assert ssv.lib().ssv_accept_noalloc(C.byref(a), stream) == ssv.SSV_OK
        assert ssv.get_status(status) == ssv.SSV_ERR_TIMEOUT
    finally:
        ssv.set_fault_injection(None)
    for _ in range(2):
        got = _run_noalloc(d, x)
        for w, g in zip(want, got):
            np.testing.assert_array_equal(g, w)


def test_noalloc_refuses_requests_beyond_its_scratch():
    ensure_built()
    # 8000 slots x 19 vocab chunks of 32-byte partial records exceed the 4 MiB
    # array; the refusal happens on the host before any pointer is touched.
    a = ssv.AcceptArgs(ssv.ARGMAX, 0.0, 151936, 8000, 8000, 1, ssv.SSV_F32, 16, None, 16, 16, 16, 16, 16,
                       None, 0, None, None, None, 16, 16, 16, None)
    assert ssv.lib().ssv_accept_noalloc(C.byref(a), None) == ssv.SSV_ERR_WORKSPACE
