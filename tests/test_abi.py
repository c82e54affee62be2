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


def test_every_entry_point_has_a_declared_signature(L):
    """Without argtypes ctypes passes a Python int as a 32-bit C int, which
    truncates device addresses: every entry point that takes arguments must
    declare them."""
    for name in ssv.EXPORTS:
        if name == "ssv_version":
            continue
        assert getattr(L, name).argtypes is not None, name


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


def test_accept_workspace_holds_the_emission_exponentials(L):
    """Under rejection sampling the workspace adds 16 bytes per vocabulary
    entry (rounded up to 8192-entry chunks) per sequence, as the header
    states, for the emitted rows' stored exponentials."""
    for V, batch in ((1000, 2), (151936, 16), (8193, 3)):
        g, r = C.c_size_t(0), C.c_size_t(0)
        kw = dict(V=V, batch=batch, total_slots=4 * batch)
        assert L.ssv_accept_workspace(C.byref(_acc(**kw)), C.byref(g)) == ssv.SSV_OK
        rej = _acc(mode=ssv.REJECT, T=1.0, draft_logits=16, u_accept=16, u_sample=16, **kw)
        assert L.ssv_accept_workspace(C.byref(rej), C.byref(r)) == ssv.SSV_OK
        stored = 16 * batch * 8192 * ((V + 8191) // 8192)
        assert stored <= r.value - g.value < stored + 256, (V, batch, r.value - g.value)


def test_bench_rejects_unknown_config(L):
    buf = C.create_string_buffer(256)
    assert L.ssv_bench(b"nope", 1, buf, 256) == ssv.SSV_ERR_INVALID
    assert L.ssv_bench(b"tiny", 0, buf, 256) == ssv.SSV_ERR_INVALID


def _commit(**kw):
    base = dict(k_new=16, v_new=4096, k_dst=1 << 20, v_dst=1 << 21, dtype=ssv.SSV_BF16, Hkv=2, d=128, seqs=16,
                batch=2, tau=16, n_acc=16, dst_off=16, dst_cap=16, new_len=16, total_rows=4, total_slots=4,
                dst_rows=20, dev_status=None)
    base.update(kw)
    return ssv.CommitArgs(**base)


def test_commit_validation(L):
    cases = [(dict(dtype=7), ssv.SSV_ERR_INVALID), (dict(d=96), ssv.SSV_ERR_UNSUPPORTED),
             (dict(batch=-1), ssv.SSV_ERR_INVALID), (dict(Hkv=0), ssv.SSV_ERR_INVALID),
             (dict(total_slots=-1), ssv.SSV_ERR_INVALID), (dict(n_acc=None), ssv.SSV_ERR_INVALID),
             (dict(new_len=None), ssv.SSV_ERR_INVALID), (dict(k_new=24), ssv.SSV_ERR_INVALID),   # misaligned
             (dict(k_dst=16), ssv.SSV_ERR_INVALID),                                             # overlaps k_new
             (dict(v_dst=4096 + 512), ssv.SSV_ERR_INVALID)]                                     # overlaps v_new
    for kw, code in cases:
        assert L.ssv_commit(C.byref(_commit(**kw)), None) == code, kw
    assert L.ssv_commit(C.byref(_commit(batch=0)), None) == ssv.SSV_OK   # nothing to do
    assert L.ssv_commit(None, None) == ssv.SSV_ERR_INVALID


def _lmh(**kw):
    base = dict(mode=ssv.ARGMAX, T=0.0, V=1000, hidden=128, batch=2, total_slots=8, hidden_states=256,
                lm_head=512, draft_tokens=16, tau=16, block=16, gamma=16, slot_off=16, noise=None,
                n_noise_rows=0, noise_row=None, n_acc=16, n_out=16, tokens=16, dev_status=None)
    base.update(kw)
    return ssv.LmheadArgs(**base)


def test_lmhead_validation(L):
    cases = [(dict(mode=ssv.REJECT, T=1.0), ssv.SSV_ERR_INVALID), (dict(T=float("nan")), ssv.SSV_ERR_NOT_FINITE),
             (dict(T=-0.5), ssv.SSV_ERR_NOT_FINITE), (dict(hidden=96), ssv.SSV_ERR_INVALID),
             (dict(hidden=0), ssv.SSV_ERR_INVALID), (dict(V=0), ssv.SSV_ERR_INVALID),
             (dict(total_slots=4096), ssv.SSV_ERR_UNSUPPORTED), (dict(batch=3000), ssv.SSV_ERR_UNSUPPORTED),
             (dict(lm_head=None), ssv.SSV_ERR_INVALID), (dict(hidden_states=520), ssv.SSV_ERR_INVALID),
             (dict(mode=ssv.GUMBEL, T=1.0), ssv.SSV_ERR_INVALID),                 # no noise table
             (dict(mode=ssv.GUMBEL, T=1.0, noise=18, noise_row=16, n_noise_rows=8), ssv.SSV_ERR_INVALID)]
    n = C.c_size_t(0)
    for kw, code in cases:
        assert L.ssv_lmhead_accept(C.byref(_lmh(**kw)), None, 0, None) == code, kw
        assert L.ssv_lmhead_accept_workspace(C.byref(_lmh(**kw)), C.byref(n)) == code, kw
    assert L.ssv_lmhead_accept(C.byref(_lmh(batch=0)), None, 0, None) == ssv.SSV_OK
    assert L.ssv_lmhead_accept_workspace(C.byref(_lmh(total_slots=0)), C.byref(n)) == ssv.SSV_OK and n.value == 0


def test_stream_read_rejects_bad_arguments(L):
    """The read-floor reference validates its arguments on the host."""
    out = 1 << 20
    assert L.ssv_stream_read(None, 64, out, None) == ssv.SSV_ERR_INVALID
    assert L.ssv_stream_read(1 << 20, 64, None, None) == ssv.SSV_ERR_INVALID
    assert L.ssv_stream_read((1 << 20) + 8, 64, out, None) == ssv.SSV_ERR_INVALID  # misaligned
    assert L.ssv_stream_read(1 << 20, 40, out, None) == ssv.SSV_ERR_INVALID        # not a multiple of 16
    assert L.ssv_stream_read(1 << 20, 0, out, None) == ssv.SSV_OK                  # nothing to read


def test_tree_attention_workspace_query(L):
    """fp32 inputs run the prompt part in the node kernel: no workspace."""
    a = ssv.TreeAttnArgs(1 << 20, 1 << 21, 1 << 22, 1 << 23, 1 << 24, 1 << 25, ssv.SSV_F32, ssv.SSV_F32, 4, 2, 64, 0.0,
                         1 << 26, 1, 1 << 27, 1 << 28, 8, 12, 16, 2, 40, 16, None)
    n = C.c_size_t(7)
    assert L.ssv_tree_verify_attn_workspace(C.byref(a), C.byref(n)) == ssv.SSV_OK
    assert n.value == 0
    assert L.ssv_tree_verify_attn_workspace(C.byref(a), None) == ssv.SSV_ERR_INVALID
