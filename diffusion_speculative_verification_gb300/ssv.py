"""ctypes binding of libssv (include/ssv.h).  Argument marshalling only:
every step of the verification pass runs in the library's CUDA kernels.
PyTorch supplies device memory and streams.

The library is loaded from this package's ``lib/libssv.so`` (built in-tree
by ``build.build()``).  If it is missing every call raises ``SsvError``;
there is no CPU fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import numpy as np

from .build import LIB

SSV_OK, SSV_ERR_INVALID, SSV_ERR_UNSUPPORTED, SSV_ERR_CUDA = 0, 1, 2, 3
SSV_ERR_TIMEOUT, SSV_ERR_BAD_TAU, SSV_ERR_WORKSPACE, SSV_ERR_NOT_FINITE = 4, 5, 6, 7
SSV_F32, SSV_BF16 = 0, 1
ARGMAX, GUMBEL, REJECT, GUMBEL_GEN = 0, 1, 2, 3

#: every symbol include/ssv.h declares
EXPORTS = ("ssv_rope_copy", "ssv_verify_attn_workspace", "ssv_verify_attn", "ssv_verify_step", "ssv_accept_workspace",
           "ssv_accept", "ssv_accept_noalloc", "ssv_commit", "ssv_lmhead_accept_workspace", "ssv_lmhead_accept",
           "ssv_get_status", "ssv_status_string", "ssv_version", "ssv_bench", "ssv_set_fault_injection",
           "ssv_tree_verify_attn_workspace", "ssv_tree_verify_attn", "ssv_tree_accept_workspace", "ssv_tree_accept",
           "ssv_stream_read")
FAULT_NONE, FAULT_ATTN, FAULT_ACCEPT, FAULT_LMHEAD = 0, 1, 2, 3


class SsvError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (code {code})")


class SeqC(C.Structure):
    _fields_ = [("cache_len", C.c_int32), ("new_len", C.c_int32), ("block", C.c_int32),
                ("q_off", C.c_int32), ("kv_off", C.c_int32), ("tau_off", C.c_int32)]


class RopeArgs(C.Structure):
    _fields_ = [("q_in", C.c_void_p), ("k_in", C.c_void_p), ("q_out", C.c_void_p), ("k_out", C.c_void_p),
                ("dtype", C.c_int), ("Hq", C.c_int32), ("Hkv", C.c_int32), ("d", C.c_int32),
                ("base", C.c_double), ("seqs", C.c_void_p), ("batch", C.c_int32), ("total_rows", C.c_int32),
                ("positions", C.c_void_p), ("dev_status", C.c_void_p)]


class AttnArgs(C.Structure):
    _fields_ = [("q", C.c_void_p), ("k_cache", C.c_void_p), ("v_cache", C.c_void_p), ("k_new", C.c_void_p),
                ("v_new", C.c_void_p), ("o", C.c_void_p), ("in_dtype", C.c_int), ("out_dtype", C.c_int),
                ("Hq", C.c_int32), ("Hkv", C.c_int32), ("d", C.c_int32), ("scale", C.c_float),
                ("seqs", C.c_void_p), ("batch", C.c_int32), ("tau", C.c_void_p), ("total_rows", C.c_int32),
                ("total_cache", C.c_int32), ("total_slots", C.c_int32), ("max_cache", C.c_int32),
                ("max_new", C.c_int32), ("max_block", C.c_int32), ("dev_status", C.c_void_p)]


class AcceptArgs(C.Structure):
    _fields_ = [("mode", C.c_int), ("T", C.c_float), ("V", C.c_int32), ("batch", C.c_int32),
                ("total_slots", C.c_int32), ("max_block", C.c_int32), ("logits_dtype", C.c_int),
                ("logits", C.c_void_p), ("draft_logits", C.c_void_p), ("draft_tokens", C.c_void_p),
                ("tau", C.c_void_p), ("block", C.c_void_p), ("gamma", C.c_void_p), ("slot_off", C.c_void_p),
                ("noise", C.c_void_p), ("n_noise_rows", C.c_int32), ("noise_row", C.c_void_p),
                ("u_accept", C.c_void_p), ("u_sample", C.c_void_p), ("n_acc", C.c_void_p),
                ("n_out", C.c_void_p), ("tokens", C.c_void_p), ("dev_status", C.c_void_p),
                ("noise_seed", C.c_uint64)]


class CommitArgs(C.Structure):
    _fields_ = [("k_new", C.c_void_p), ("v_new", C.c_void_p), ("k_dst", C.c_void_p), ("v_dst", C.c_void_p),
                ("dtype", C.c_int), ("Hkv", C.c_int32), ("d", C.c_int32), ("seqs", C.c_void_p),
                ("batch", C.c_int32), ("tau", C.c_void_p), ("n_acc", C.c_void_p), ("dst_off", C.c_void_p),
                ("dst_cap", C.c_void_p), ("new_len", C.c_void_p), ("total_rows", C.c_int32),
                ("total_slots", C.c_int32), ("dst_rows", C.c_int32), ("dev_status", C.c_void_p)]


class TreeAttnArgs(C.Structure):
    _fields_ = [("q", C.c_void_p), ("k_cache", C.c_void_p), ("v_cache", C.c_void_p), ("k_new", C.c_void_p),
                ("v_new", C.c_void_p), ("o", C.c_void_p), ("in_dtype", C.c_int), ("out_dtype", C.c_int),
                ("Hq", C.c_int32), ("Hkv", C.c_int32), ("d", C.c_int32), ("scale", C.c_float), ("seqs", C.c_void_p),
                ("batch", C.c_int32), ("parent", C.c_void_p), ("pos", C.c_void_p), ("total_q", C.c_int32),
                ("total_k", C.c_int32), ("total_cache", C.c_int32), ("total_edges", C.c_int32),
                ("total_out", C.c_int32), ("max_cache", C.c_int32), ("dev_status", C.c_void_p)]


class TreeAcceptArgs(C.Structure):
    _fields_ = [("mode", C.c_int), ("T", C.c_float), ("V", C.c_int32), ("seqs", C.c_void_p), ("batch", C.c_int32),
                ("logits_dtype", C.c_int), ("logits", C.c_void_p), ("parent", C.c_void_p), ("pos", C.c_void_p),
                ("token", C.c_void_p), ("total_edges", C.c_int32), ("total_out", C.c_int32),
                ("noise", C.c_void_p), ("n_noise_rows", C.c_int32), ("noise_row", C.c_void_p),
                ("pos_off", C.c_void_p), ("total_positions", C.c_int32), ("n_acc", C.c_void_p), ("path", C.c_void_p),
                ("emit_pos", C.c_void_p), ("emit_tok", C.c_void_p), ("dev_status", C.c_void_p)]


class FaultInjection(C.Structure):
    _fields_ = [("kernel", C.c_int), ("skip", C.c_int32), ("wait_budget_cycles", C.c_int64)]


class LmheadArgs(C.Structure):
    _fields_ = [("mode", C.c_int), ("T", C.c_float), ("V", C.c_int32), ("hidden", C.c_int32),
                ("batch", C.c_int32), ("total_slots", C.c_int32), ("hidden_states", C.c_void_p),
                ("lm_head", C.c_void_p), ("draft_tokens", C.c_void_p), ("tau", C.c_void_p), ("block", C.c_void_p),
                ("gamma", C.c_void_p), ("slot_off", C.c_void_p), ("noise", C.c_void_p),
                ("n_noise_rows", C.c_int32), ("noise_row", C.c_void_p), ("n_acc", C.c_void_p),
                ("n_out", C.c_void_p), ("tokens", C.c_void_p), ("dev_status", C.c_void_p)]


_lib = None


def lib():
    """Load libssv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise SsvError(SSV_ERR_UNSUPPORTED, f"libssv not built ({LIB} missing; run __graft_entry__.build())")
        L = C.CDLL(LIB)
        vp, sz = C.c_void_p, C.c_size_t
        L.ssv_rope_copy.argtypes = [C.POINTER(RopeArgs), vp]
        L.ssv_verify_attn_workspace.argtypes = [C.POINTER(AttnArgs), C.POINTER(sz)]
        L.ssv_verify_attn.argtypes = [C.POINTER(AttnArgs), vp, sz, vp]
        L.ssv_accept_workspace.argtypes = [C.POINTER(AcceptArgs), C.POINTER(sz)]
        L.ssv_accept.argtypes = [C.POINTER(AcceptArgs), vp, sz, vp]
        L.ssv_accept_noalloc.argtypes = [C.POINTER(AcceptArgs), vp]
        L.ssv_commit.argtypes = [C.POINTER(CommitArgs), vp]
        L.ssv_lmhead_accept_workspace.argtypes = [C.POINTER(LmheadArgs), C.POINTER(sz)]
        L.ssv_lmhead_accept.argtypes = [C.POINTER(LmheadArgs), vp, sz, vp]
        L.ssv_verify_step.argtypes = [C.POINTER(RopeArgs), C.POINTER(AttnArgs), vp, sz, C.POINTER(AcceptArgs), vp,
                                      sz, vp]
        L.ssv_get_status.argtypes = [vp, vp]
        L.ssv_status_string.argtypes = [C.c_int]
        L.ssv_status_string.restype = C.c_char_p
        L.ssv_version.restype = C.c_char_p
        L.ssv_bench.argtypes = [C.c_char_p, C.c_int32, C.c_char_p, sz]
        L.ssv_stream_read.argtypes = [vp, sz, vp, vp]
        L.ssv_set_fault_injection.argtypes = [C.POINTER(FaultInjection)]
        L.ssv_tree_verify_attn_workspace.argtypes = [C.POINTER(TreeAttnArgs), C.POINTER(sz)]
        L.ssv_tree_verify_attn.argtypes = [C.POINTER(TreeAttnArgs), vp, sz, vp]
        L.ssv_tree_accept_workspace.argtypes = [C.POINTER(TreeAcceptArgs), C.POINTER(sz)]
        L.ssv_tree_accept.argtypes = [C.POINTER(TreeAcceptArgs), vp, sz, vp]
        for name in ("ssv_rope_copy", "ssv_verify_attn_workspace", "ssv_verify_attn", "ssv_verify_step",
                     "ssv_accept_workspace", "ssv_accept", "ssv_accept_noalloc", "ssv_commit",
                     "ssv_lmhead_accept_workspace", "ssv_lmhead_accept", "ssv_get_status", "ssv_bench",
                     "ssv_set_fault_injection", "ssv_tree_verify_attn_workspace", "ssv_tree_verify_attn",
                     "ssv_tree_accept_workspace", "ssv_tree_accept", "ssv_stream_read"):
            getattr(L, name).restype = C.c_int
        _lib = L
    return _lib


def status_string(code: int) -> str:
    try:
        return lib().ssv_status_string(int(code)).decode()
    except SsvError:
        return "libssv unavailable"


def version() -> str:
    return lib().ssv_version().decode()


def _check(code: int, what: str):
    if code != SSV_OK:
        raise SsvError(code, what)


# ---------------------------------------------------------------------------
# torch plumbing
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return SSV_F32
    if t.dtype == torch.bfloat16:
        return SSV_BF16
    raise SsvError(SSV_ERR_INVALID, f"unsupported dtype {t.dtype}")


class Batch:
    """A packed batch: host ssv_seq table + device copy + the bounds the library needs."""

    def __init__(self, seqs: np.ndarray, device="cuda"):
        torch = _torch()
        self.host = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32).reshape(-1, 6))
        self.dev = torch.from_numpy(self.host.copy()).to(device)
        h = self.host
        self.batch = int(h.shape[0])
        self.total_rows = int(np.sum(h[:, 1] + 2 * h[:, 2])) if self.batch else 0
        self.total_cache = int(np.sum(h[:, 0])) if self.batch else 0
        self.total_slots = int(np.sum(h[:, 2])) if self.batch else 0
        self.max_cache = int(h[:, 0].max()) if self.batch else 0
        self.max_new = int(h[:, 1].max()) if self.batch else 0
        self.max_block = int(h[:, 2].max()) if self.batch else 1


def _workspace(nbytes: int, device, ws=None):
    torch = _torch()
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise SsvError(SSV_ERR_WORKSPACE, "workspace")
        return ws
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------
def rope_args(q, k, batch: Batch, base: float = 10000.0, q_out=None, k_out=None, positions=None, dev_status=None):
    """positions: optional int32 [rows] device table (fresh rows and data rows
    at their entries, mask rows at their data row's)."""
    q_out = q if q_out is None else q_out
    k_out = k if k_out is None else k_out
    return RopeArgs(_ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), _dtype_code(q), q.shape[1], k.shape[1], q.shape[2],
                    float(base), _ptr(batch.dev), batch.batch, q.shape[0], _ptr(positions), _ptr(dev_status))


def rope_copy(q, k, batch: Batch, base: float = 10000.0, q_out=None, k_out=None, stream=None, positions=None,
              dev_status=None):
    """Rotate Q [rows, Hq, d] and K_new [rows, Hkv, d]; returns (q_out, k_out)."""
    a = rope_args(q, k, batch, base, q_out, k_out, positions, dev_status)
    _check(lib().ssv_rope_copy(C.byref(a), _stream_ptr(stream)), "ssv_rope_copy")
    return (q if q_out is None else q_out), (k if k_out is None else k_out)


def verify_step(rope: "RopeArgs | None", attn: AttnArgs, attn_workspace, accept: "AcceptArgs | None" = None,
                accept_workspace=None, stream=None):
    """ssv_verify_step on prepared argument blocks (see rope_args, attn_args,
    accept_args): rotation, verification attention and acceptance as one call."""
    aw = _ptr(attn_workspace)
    awb = 0 if attn_workspace is None else attn_workspace.numel() * attn_workspace.element_size()
    cw = _ptr(accept_workspace)
    cwb = 0 if accept_workspace is None else accept_workspace.numel() * accept_workspace.element_size()
    _check(lib().ssv_verify_step(None if rope is None else C.byref(rope), C.byref(attn), aw, awb,
                                 None if accept is None else C.byref(accept), cw, cwb, _stream_ptr(stream)),
           "ssv_verify_step")


def attn_args(q, k_cache, v_cache, k_new, v_new, out, batch: Batch, tau, scale: float = 0.0, dev_status=None):
    return AttnArgs(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), _ptr(out),
                    _dtype_code(q), _dtype_code(out), q.shape[1], k_new.shape[1], q.shape[2], float(scale),
                    _ptr(batch.dev), batch.batch, _ptr(tau), batch.total_rows,
                    batch.total_cache if k_cache is None else k_cache.shape[0], batch.total_slots, batch.max_cache, batch.max_new, batch.max_block, _ptr(dev_status))


def verify_attn_workspace_bytes(args: AttnArgs) -> int:
    n = C.c_size_t(0)
    _check(lib().ssv_verify_attn_workspace(C.byref(args), C.byref(n)), "ssv_verify_attn_workspace")
    return int(n.value)


def verify_attn(q, k_cache, v_cache, k_new, v_new, batch: Batch, tau, out=None, out_dtype=None,
                scale: float = 0.0, workspace=None, dev_status=None, stream=None):
    """Verification attention; returns O [rows, Hq, d]."""
    torch = _torch()
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    a = attn_args(q, k_cache, v_cache, k_new, v_new, out, batch, tau, scale, dev_status)
    ws = _workspace(verify_attn_workspace_bytes(a), q.device, workspace)
    _check(lib().ssv_verify_attn(C.byref(a), _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream)),
           "ssv_verify_attn")
    return out


def accept_args(mode, T, logits, draft_tokens, tau, block, gamma, slot_off, n_acc, n_out, tokens,
                draft_logits=None, noise=None, noise_row=None, u_accept=None, u_sample=None, max_block=64,
                dev_status=None, noise_seed=0):
    return AcceptArgs(int(mode), float(T), logits.shape[1], block.shape[0], draft_tokens.shape[0], int(max_block),
                      _dtype_code(logits), _ptr(logits), _ptr(draft_logits), _ptr(draft_tokens), _ptr(tau),
                      _ptr(block), _ptr(gamma), _ptr(slot_off), _ptr(noise),
                      0 if noise is None else noise.shape[0], _ptr(noise_row), _ptr(u_accept), _ptr(u_sample),
                      _ptr(n_acc), _ptr(n_out), _ptr(tokens), _ptr(dev_status), int(noise_seed))


def accept_workspace_bytes(args: AcceptArgs) -> int:
    n = C.c_size_t(0)
    _check(lib().ssv_accept_workspace(C.byref(args), C.byref(n)), "ssv_accept_workspace")
    return int(n.value)


def accept(mode, T, logits, draft_tokens, tau, block, gamma, slot_off, draft_logits=None, noise=None,
           noise_row=None, u_accept=None, u_sample=None, max_block=64, workspace=None, dev_status=None,
           stream=None, out=None, noise_seed=0):
    """Acceptance; returns (n_acc [batch], n_out [batch], tokens [slots]) int32 device tensors."""
    torch = _torch()
    dev = logits.device
    if out is None:
        out = (torch.empty(block.shape[0], dtype=torch.int32, device=dev),
               torch.empty(block.shape[0], dtype=torch.int32, device=dev),
               torch.empty(draft_tokens.shape[0], dtype=torch.int32, device=dev))
    n_acc, n_out, tokens = out
    a = accept_args(mode, T, logits, draft_tokens, tau, block, gamma, slot_off, n_acc, n_out, tokens,
                    draft_logits, noise, noise_row, u_accept, u_sample, max_block, dev_status, noise_seed)
    ws = _workspace(accept_workspace_bytes(a), dev, workspace)
    _check(lib().ssv_accept(C.byref(a), _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream)),
           "ssv_accept")
    return n_acc, n_out, tokens


def accept_noalloc(mode, T, logits, draft_tokens, tau, block, gamma, slot_off, draft_logits=None, noise=None,
                   noise_row=None, u_accept=None, u_sample=None, max_block=64, dev_status=None, stream=None,
                   out=None, noise_seed=0):
    """ssv_accept without a workspace: scratch comes from the library's fixed
    per-device array (for callers that cannot allocate).  Output tensors may
    be passed in ``out``; otherwise they are allocated here by torch."""
    torch = _torch()
    dev = logits.device
    if out is None:
        out = (torch.empty(block.shape[0], dtype=torch.int32, device=dev),
               torch.empty(block.shape[0], dtype=torch.int32, device=dev),
               torch.empty(draft_tokens.shape[0], dtype=torch.int32, device=dev))
    n_acc, n_out, tokens = out
    a = accept_args(mode, T, logits, draft_tokens, tau, block, gamma, slot_off, n_acc, n_out, tokens,
                    draft_logits, noise, noise_row, u_accept, u_sample, max_block, dev_status, noise_seed)
    _check(lib().ssv_accept_noalloc(C.byref(a), _stream_ptr(stream)), "ssv_accept_noalloc")
    return n_acc, n_out, tokens


def commit_args(k_new, v_new, k_dst, v_dst, batch: Batch, tau, n_acc, dst_off, dst_cap, new_len,
                dev_status=None):
    return CommitArgs(_ptr(k_new), _ptr(v_new), _ptr(k_dst), _ptr(v_dst), _dtype_code(k_new), k_new.shape[1],
                      k_new.shape[2], _ptr(batch.dev), batch.batch, _ptr(tau), _ptr(n_acc), _ptr(dst_off),
                      _ptr(dst_cap), _ptr(new_len), k_new.shape[0], tau.shape[0], k_dst.shape[0],
                      _ptr(dev_status))


def commit(k_new, v_new, k_dst, v_dst, batch: Batch, tau, n_acc, dst_off, dst_cap, new_len=None, dev_status=None,
           stream=None):
    """Appends each sequence's fresh prompt rows and accepted data rows (stage
    order) to its cache in k_dst / v_dst (in place); returns new_len [batch]
    int32 device (-1 for a sequence rejected on the device)."""
    torch = _torch()
    if k_dst.dtype != k_new.dtype or v_dst.dtype != k_new.dtype or v_new.dtype != k_new.dtype:
        raise SsvError(SSV_ERR_INVALID, "ssv_commit: k_new, v_new, k_dst and v_dst must share one dtype")
    if tuple(k_dst.shape[1:]) != tuple(k_new.shape[1:]) or v_dst.shape != k_dst.shape or v_new.shape != k_new.shape:
        raise SsvError(SSV_ERR_INVALID, "ssv_commit: row shapes differ")
    if new_len is None:
        new_len = torch.empty(batch.batch, dtype=torch.int32, device=k_new.device)
    a = commit_args(k_new, v_new, k_dst, v_dst, batch, tau, n_acc, dst_off, dst_cap, new_len, dev_status)
    _check(lib().ssv_commit(C.byref(a), _stream_ptr(stream)), "ssv_commit")
    return new_len


def lmhead_args(mode, T, hidden_states, lm_head, draft_tokens, tau, block, gamma, slot_off, n_acc, n_out, tokens,
                noise=None, noise_row=None, dev_status=None):
    return LmheadArgs(int(mode), float(T), lm_head.shape[0], lm_head.shape[1], block.shape[0],
                      draft_tokens.shape[0], _ptr(hidden_states), _ptr(lm_head), _ptr(draft_tokens), _ptr(tau),
                      _ptr(block), _ptr(gamma), _ptr(slot_off), _ptr(noise), 0 if noise is None else noise.shape[0],
                      _ptr(noise_row), _ptr(n_acc), _ptr(n_out), _ptr(tokens), _ptr(dev_status))


def lmhead_accept_workspace_bytes(args: LmheadArgs) -> int:
    n = C.c_size_t(0)
    _check(lib().ssv_lmhead_accept_workspace(C.byref(args), C.byref(n)), "ssv_lmhead_accept_workspace")
    return int(n.value)


def lmhead_accept(mode, T, hidden_states, lm_head, draft_tokens, tau, block, gamma, slot_off, noise=None,
                  noise_row=None, workspace=None, dev_status=None, stream=None, out=None):
    """LM head over the slots' hidden states fused with acceptance; returns
    (n_acc [batch], n_out [batch], tokens [slots]) int32 device tensors."""
    torch = _torch()
    if hidden_states.dtype != torch.bfloat16 or lm_head.dtype != torch.bfloat16:
        raise SsvError(SSV_ERR_INVALID, "ssv_lmhead_accept: hidden states and LM head must be bf16")
    if hidden_states.shape[1] != lm_head.shape[1] or hidden_states.shape[0] != draft_tokens.shape[0]:
        raise SsvError(SSV_ERR_INVALID, "ssv_lmhead_accept: shapes")
    dev = hidden_states.device
    if out is None:
        out = (torch.empty(block.shape[0], dtype=torch.int32, device=dev),
               torch.empty(block.shape[0], dtype=torch.int32, device=dev),
               torch.empty(draft_tokens.shape[0], dtype=torch.int32, device=dev))
    n_acc, n_out, tokens = out
    a = lmhead_args(mode, T, hidden_states, lm_head, draft_tokens, tau, block, gamma, slot_off, n_acc, n_out,
                    tokens, noise, noise_row, dev_status)
    ws = _workspace(lmhead_accept_workspace_bytes(a), dev, workspace)
    _check(lib().ssv_lmhead_accept(C.byref(a), _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream)),
           "ssv_lmhead_accept")
    return n_acc, n_out, tokens


def set_fault_injection(kernel=None, skip: int = -1, wait_budget_cycles: int = 1 << 31):
    """Test support: shorten the bounded waits of one kernel and make its CTA 0
    leave out one copy (see ssv_set_fault_injection); kernel None restores the
    defaults."""
    if kernel is None:
        _check(lib().ssv_set_fault_injection(None), "ssv_set_fault_injection")
        return
    f = FaultInjection(int(kernel), int(skip), int(wait_budget_cycles))
    _check(lib().ssv_set_fault_injection(C.byref(f)), "ssv_set_fault_injection")


def tree_attn_args(q, k_cache, v_cache, k_new, v_new, out, seqs, parent, pos, total_out, max_cache,
                   scale: float = 0.0, dev_status=None):
    """seqs: int32 [batch, 9] device tensor of ssv_tree_seq records."""
    return TreeAttnArgs(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), _ptr(out), _dtype_code(q),
                        _dtype_code(out), q.shape[1], k_new.shape[1], q.shape[2], float(scale), _ptr(seqs),
                        seqs.shape[0], _ptr(parent), _ptr(pos), q.shape[0], k_new.shape[0],
                        0 if k_cache is None else k_cache.shape[0], 0 if parent is None else parent.shape[0],
                        int(total_out), int(max_cache), _ptr(dev_status))


def tree_verify_attn_workspace_bytes(args: TreeAttnArgs) -> int:
    n = C.c_size_t(0)
    _check(lib().ssv_tree_verify_attn_workspace(C.byref(args), C.byref(n)), "ssv_tree_verify_attn_workspace")
    return n.value


def tree_verify_attn(q, k_cache, v_cache, k_new, v_new, seqs, parent, pos, total_out, max_cache, out=None,
                     out_dtype=None, scale: float = 0.0, dev_status=None, stream=None, workspace=None):
    """Attention of the tree pass; returns O [total_out, Hq, d] (rows of
    committed positions are left as they were in `out`).  workspace: a zeroed
    uint8 device tensor of tree_verify_attn_workspace_bytes (allocated here
    when not given)."""
    torch = _torch()
    if out is None:
        out = torch.zeros((int(total_out), q.shape[1], q.shape[2]), dtype=out_dtype or q.dtype, device=q.device)
    a = tree_attn_args(q, k_cache, v_cache, k_new, v_new, out, seqs, parent, pos, total_out, max_cache, scale,
                       dev_status)
    ws = _workspace(tree_verify_attn_workspace_bytes(a), q.device, workspace)
    _check(lib().ssv_tree_verify_attn(C.byref(a), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                      _stream_ptr(stream)), "ssv_tree_verify_attn")
    return out


def tree_accept_args(mode, T, logits, seqs, parent, pos, token, n_acc, path, emit_pos, emit_tok, noise=None,
                     noise_row=None, pos_off=None, dev_status=None):
    return TreeAcceptArgs(int(mode), float(T), logits.shape[1], _ptr(seqs), seqs.shape[0], _dtype_code(logits),
                          _ptr(logits), _ptr(parent), _ptr(pos), _ptr(token),
                          0 if parent is None else parent.shape[0], logits.shape[0], _ptr(noise),
                          0 if noise is None else noise.shape[0], _ptr(noise_row), _ptr(pos_off),
                          0 if noise_row is None else noise_row.shape[0], _ptr(n_acc), _ptr(path), _ptr(emit_pos),
                          _ptr(emit_tok), _ptr(dev_status))


def tree_accept(mode, T, logits, seqs, parent, pos, token, noise=None, noise_row=None, pos_off=None, workspace=None,
                dev_status=None, stream=None):
    """Acceptance of the tree by state equality; returns (n_acc [batch],
    path [batch, 64], emit_pos [batch], emit_tok [batch]) int32 device tensors."""
    torch = _torch()
    dev = logits.device
    b = seqs.shape[0]
    n_acc = torch.empty(b, dtype=torch.int32, device=dev)
    path = torch.empty((b, 64), dtype=torch.int32, device=dev)
    ep = torch.empty(b, dtype=torch.int32, device=dev)
    et = torch.empty(b, dtype=torch.int32, device=dev)
    a = tree_accept_args(mode, T, logits, seqs, parent, pos, token, n_acc, path, ep, et, noise, noise_row, pos_off,
                         dev_status)
    n = C.c_size_t(0)
    _check(lib().ssv_tree_accept_workspace(C.byref(a), C.byref(n)), "ssv_tree_accept_workspace")
    ws = _workspace(int(n.value), dev, workspace)
    _check(lib().ssv_tree_accept(C.byref(a), _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream)),
           "ssv_tree_accept")
    return n_acc, path, ep, et


def stream_read(buf, out, stream=None):
    """Reads every byte of the device tensor `buf` once (measurement reference
    for memory-bound kernels); XOR checksum into the int32 device tensor `out`."""
    nbytes = buf.numel() * buf.element_size()
    _check(lib().ssv_stream_read(_ptr(buf), nbytes, _ptr(out), _stream_ptr(stream)), "ssv_stream_read")


def get_status(dev_status, stream=None) -> int:
    """Waits for the stream and returns (and clears) the device status word."""
    return int(lib().ssv_get_status(_ptr(dev_status), _stream_ptr(stream)))


def bench(config: str, iters: int = 20) -> str:
    buf = C.create_string_buffer(4096)
    _check(lib().ssv_bench(config.encode(), int(iters), buf, 4096), "ssv_bench")
    return buf.value.decode()
