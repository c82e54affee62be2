"""C-ABI checks that need no GPU: the library builds for sm_103a, loads, and
exports every entry point include/ssv.h declares; host-side argument
validation rejects bad calls synchronously without touching the device."""
import ctypes as C
import os
import re

import pytest

from diffusion_speculative_verification_gb300 import build, ssv

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ssv.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return ssv.lib()


def declared():
    text = open(HEADER).read()
    return set(re.findall(r"SSV_API\s+[\w\s\*]*?\b(ssv_\w+)\s*\(", text))


def test_header_matches_binding_list():
    assert declared() == set(ssv.EXPORTS)


def test_every_declared_symbol_exported(L):
    for name in declared():
        assert hasattr(L, name), name
    assert ssv.version().startswith("ssv ")


def test_status_strings(L):
    for code in range(8):
        assert ssv.status_string(code) != "unknown status"
    assert ssv.status_string(99) == "unknown status"


def test_rope_rejects_bad_arguments(L):
    a = ssv.RopeArgs(None, None, None, None, ssv.SSV_BF16, 4, 2, 128, 10000.0, None, 1, 10)
    assert L.ssv_rope_copy(C.byref(a), None) == ssv.SSV_ERR_INVALID
    a = ssv.RopeArgs(16, 16, 16, 16, ssv.SSV_BF16, 4, 2, 96, 10000.0, 16, 1, 10)
    assert L.ssv_rope_copy(C.byref(a), None) == ssv.SSV_ERR_UNSUPPORTED
    a = ssv.RopeArgs(16, 16, 24, 16, ssv.SSV_BF16, 4, 2, 128, 10000.0, 16, 1, 10)   # misaligned output
    assert L.ssv_rope_copy(C.byref(a), None) == ssv.SSV_ERR_INVALID
    a = ssv.RopeArgs(16, 16, 16, 16, ssv.SSV_BF16, 4, 2, 128, float("nan"), 16, 1, 10)
    assert L.ssv_rope_copy(C.byref(a), None) == ssv.SSV_ERR_INVALID
    a = ssv.RopeArgs(None, None, None, None, ssv.SSV_BF16, 4, 2, 128, 10000.0, None, 0, 0)
    assert L.ssv_rope_copy(C.byref(a), None) == ssv.SSV_OK   # empty batch: nothing to do


def _attn(**kw):
    base = dict(q=16, k_cache=16, v_cache=16, k_new=16, v_new=16, o=16, in_dtype=ssv.SSV_BF16,
                out_dtype=ssv.SSV_BF16, Hq=32, Hkv=8, d=128, scale=0.0, seqs=16, batch=2, tau=16,
                total_rows=40, total_cache=100, total_slots=20, max_cache=50, max_new=0, max_block=10,
                dev_status=None)
    base.update(kw)
    return ssv.AttnArgs(**base)


def test_attn_validation(L):
    n = C.c_size_t(0)
    assert L.ssv_verify_attn_workspace(C.byref(_attn()), C.byref(n)) == ssv.SSV_OK and n.value >= 0
    cases = [(dict(Hq=30), ssv.SSV_ERR_INVALID), (dict(d=96), ssv.SSV_ERR_UNSUPPORTED),
             (dict(max_block=65), ssv.SSV_ERR_INVALID), (dict(q=None), ssv.SSV_ERR_INVALID),
             (dict(o=8), ssv.SSV_ERR_INVALID), (dict(in_dtype=ssv.SSV_F32), ssv.SSV_ERR_UNSUPPORTED),
             (dict(scale=float("inf")), ssv.SSV_ERR_INVALID), (dict(in_dtype=7), ssv.SSV_ERR_INVALID)]
    for kw, code in cases:
        assert L.ssv_verify_attn(C.byref(_attn(**kw)), None, 0, None) == code, kw
    # workspace missing for a non-empty call
    assert L.ssv_verify_attn(C.byref(_attn()), None, 0, None) == ssv.SSV_ERR_WORKSPACE
    # empty batch is a no-op
    assert L.ssv_verify_attn(C.byref(_attn(batch=0, total_rows=0)), None, 0, None) == ssv.SSV_OK


def _acc(**kw):
    base = dict(mode=ssv.ARGMAX, T=0.0, V=1000, batch=2, total_slots=8, max_block=4, logits_dtype=ssv.SSV_F32,
                logits=16, draft_logits=None, draft_tokens=16, tau=16, block=16, gamma=16, slot_off=16,
                noise=None, n_noise_rows=0, noise_row=None, u_accept=None, u_sample=None, n_acc=16,
                n_out=16, tokens=16, dev_status=None)
    base.update(kw)
    return ssv.AcceptArgs(**base)


def test_accept_validation(L):
    n = C.c_size_t(0)
    assert L.ssv_accept_workspace(C.byref(_acc()), C.byref(n)) == ssv.SSV_OK and n.value > 0
    cases = [(dict(T=float("nan")), ssv.SSV_ERR_NOT_FINITE), (dict(T=-1.0), ssv.SSV_ERR_NOT_FINITE),
             (dict(mode=ssv.REJECT, T=0.0), ssv.SSV_ERR_INVALID),
             (dict(mode=ssv.REJECT, T=1.0), ssv.SSV_ERR_INVALID),          # no draft logits / uniforms
             (dict(mode=ssv.GUMBEL, T=1.0), ssv.SSV_ERR_INVALID),          # no noise table
             (dict(V=0), ssv.SSV_ERR_INVALID), (dict(max_block=0), ssv.SSV_ERR_INVALID),
             (dict(mode=5), ssv.SSV_ERR_INVALID), (dict(tokens=None), ssv.SSV_ERR_INVALID)]
    for kw, code in cases:
        assert L.ssv_accept(C.byref(_acc(**kw)), None, 0, None) == code, kw
    assert L.ssv_accept(C.byref(_acc()), None, 0, None) == ssv.SSV_ERR_WORKSPACE
    assert L.ssv_accept(C.byref(_acc()), 24, 1 << 20, None) == ssv.SSV_ERR_WORKSPACE   # misaligned
    assert L.ssv_accept(C.byref(_acc(batch=0, total_slots=0)), None, 0, None) == ssv.SSV_OK


def test_bench_rejects_unknown_config(L):
    buf = C.create_string_buffer(256)
    assert L.ssv_bench(b"nope", 1, buf, 256) == ssv.SSV_ERR_INVALID
    assert L.ssv_bench(b"tiny", 0, buf, 256) == ssv.SSV_ERR_INVALID
