"""The work models bench.py divides by (algorithmic bytes and flops of the
commit and of the fused LM head), checked against hand counts."""
import importlib.util
import os

import numpy as np

from diffusion_speculative_verification_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_commit_bytes_hand_count():
    b = _bench()
    a = W.make_attn_inputs("w", [5, 0], [3, 7], [4, 2], 4, 2, 64, W.BF16, 1)
    # K and V, read and write, (N + n_acc) rows of Hkv * d bf16 elements
    want = 2 * 2 * ((3 + 1) + (7 + 2)) * 2 * 64 * 2
    assert b.commit_bytes(a, [1, 2]) == want


def test_lmhead_work_hand_count():
    b = _bench()
    V, H = 300, 64
    x = W.make_lmhead_inputs("w", W.MODE_GUMBEL, 1.0, V, H, [4, 8, 2], [4, 3, 0], 2)
    nbytes, flops, ver = b.lmhead_work(x)
    assert ver == 4 + 4 + 1                      # min(gamma + 1, B) per sequence
    assert flops == 2.0 * ver * V * H
    assert nbytes == V * H * 2 + 14 * H * 2 + ver * V * 4   # LM head, hidden states, noise rows
    x0 = W.make_lmhead_inputs("w", W.MODE_ARGMAX, 0.0, V, H, [4, 8, 2], [4, 3, 0], 2)
    assert b.lmhead_work(x0)[0] == V * H * 2 + 14 * H * 2   # greedy: no noise


def test_commit_layout_has_room():
    a = W.make_attn_inputs("w", [5, 0, 9], [3, 7, 0], [4, 2, 16], 4, 2, 64, W.BF16, 3)
    n_acc, off, cap, rows, _ = W.commit_layout(a, 4)
    C, N, B = (a.seqs[:, i] for i in range(3))
    assert np.all(cap >= C + N + B) and np.all(n_acc <= B) and np.all(n_acc >= 0)
    assert np.all(off[1:] >= off[:-1] + cap[:-1]) and off[-1] + cap[-1] <= rows   # disjoint, inside
