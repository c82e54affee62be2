"""Moves seeded workload arrays (numpy) into torch tensors and back."""
from __future__ import annotations

import numpy as np

from . import workloads as W
from .ssv import Batch


def _torch():
    import torch
    return torch


def tensor(arr: np.ndarray, dtype: str, device, pin: bool = False):
    """numpy storage (bf16 bit patterns or fp32) -> torch tensor of that dtype."""
    torch = _torch()
    if dtype == W.BF16:
        t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))
    if pin:
        return t.pin_memory()
    return t.to(device)


def to_numpy_storage(t) -> np.ndarray:
    """torch tensor -> numpy storage (bf16 as uint16 bit patterns)."""
    torch = _torch()
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def int_tensor(arr, device):
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.int32)).to(device)


def f32_tensor(arr, device):
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)


def attn_to_device(a: W.AttnInputs, device="cuda") -> dict:
    return dict(
        batch=Batch(a.seqs, device),
        tau=int_tensor(a.tau, device),
        q=tensor(a.q_raw, a.dtype, device),
        k_new=tensor(a.k_new_raw, a.dtype, device),
        v_new=tensor(a.v_new, a.dtype, device),
        k_cache=tensor(a.k_cache, a.dtype, device),
        v_cache=tensor(a.v_cache, a.dtype, device),
    )


def accept_to_device(x: W.AcceptInputs, device="cuda") -> dict:
    d = dict(
        mode=x.mode, T=x.T,
        logits=tensor(x.logits, x.logits_dtype, device),
        draft_tokens=int_tensor(x.draft_tokens, device),
        tau=int_tensor(x.tau, device),
        block=int_tensor(x.blocks, device),
        gamma=int_tensor(x.gammas, device),
        slot_off=int_tensor(x.slot_off, device),
        noise_row=int_tensor(x.noise_row, device),
        u_accept=f32_tensor(x.u_accept, device),
        u_sample=f32_tensor(x.u_sample, device),
        max_block=int(np.max(x.blocks)) if len(x.blocks) else 1,
        noise_seed=int(getattr(x, "noise_seed", 0)),
    )
    d["draft_logits"] = None if x.draft_logits is None else tensor(x.draft_logits, x.logits_dtype, device)
    d["noise"] = None if x.noise is None else f32_tensor(x.noise, device)
    return d


def lmhead_to_device(x: W.LmheadInputs, device="cuda", w=None) -> dict:
    """Device copies of a fused LM-head input set (`w`: an LM head already on
    the device, reused)."""
    a = x.acc
    d = dict(
        mode=a.mode, T=a.T,
        h=tensor(x.h, W.BF16, device),
        w=tensor(x.w, W.BF16, device) if w is None else w,
        draft_tokens=int_tensor(a.draft_tokens, device),
        tau=int_tensor(a.tau, device),
        block=int_tensor(a.blocks, device),
        gamma=int_tensor(a.gammas, device),
        slot_off=int_tensor(a.slot_off, device),
        noise_row=int_tensor(a.noise_row, device),
    )
    d["noise"] = None if a.noise is None else f32_tensor(a.noise, device)
    return d


def tree_to_device(t: W.TreeInputs, device="cuda") -> dict:
    """Device copies of a tree input set (attention inputs, and acceptance
    inputs when they were drawn)."""
    d = dict(
        seqs=int_tensor(t.seqs, device),
        parent=int_tensor(t.parent, device),
        pos=int_tensor(t.pos, device),
        token=int_tensor(t.token, device),
        q=tensor(t.q, t.dtype, device),
        k_new=tensor(t.k_new, t.dtype, device),
        v_new=tensor(t.v_new, t.dtype, device),
        k_cache=tensor(t.k_cache, t.dtype, device),
        v_cache=tensor(t.v_cache, t.dtype, device),
        total_out=t.total_out,
        max_cache=int(t.seqs[:, 0].max()) if t.batch else 0,
    )
    d["logits"] = None if t.logits is None else f32_tensor(t.logits, device)
    d["noise"] = None if t.noise is None else f32_tensor(t.noise, device)
    d["noise_row"] = None if t.noise_row is None else int_tensor(t.noise_row, device)
    d["pos_off"] = None if t.pos_off is None else int_tensor(t.pos_off, device)
    return d
