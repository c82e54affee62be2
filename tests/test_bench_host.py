"""bench.py's algorithmic work formulas against direct counts (CPU only).

The attention FLOP count uses the closed form for allowed (row, key) pairs
per sequence; it must equal the number of ones in the oracle's dense mask.
Byte counts follow the stated rule: KV cache once per kv head, Q, K/V_new,
O, and every logits / noise / draft row the acceptance needs.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from diffusion_speculative_verification_gb300 import workloads as W  # noqa: E402
from oracle.mask import verify_mask  # noqa: E402


def test_attention_pairs_match_dense_mask():
    a = W.make_attn_inputs("t", [5, 0, 17], [3, 9, 0], [4, 1, 7], 4, 2, 64, W.F32, seed=3)
    pairs = 0
    for C, N, B, _q, _k, toff in a.seqs:
        pairs += int(verify_mask(int(C), int(N), int(B), a.tau[toff:toff + B]).sum())
    _, flops = bench.attn_work(a, 4)
    assert flops == pairs * a.Hq * 4 * a.d


def test_attention_bytes():
    a = W.make_attn_inputs("t", [100, 30], [0, 2], [8, 3], 8, 2, 128, W.BF16, seed=4)
    by, _ = bench.attn_work(a, 2)
    rows = a.total_rows
    want = (130 * 2 * 128 * 2 * 2) + rows * 8 * 128 * 2 + rows * 2 * 128 * 2 * 2 + rows * 8 * 128 * 2
    assert by == want


def test_accept_bytes_per_mode():
    g = W.make_accept_inputs("g", W.MODE_GUMBEL, 1.0, 1000, [4, 8], [4, 3], seed=1)
    assert bench.accept_bytes(g) == (4 + 4) * 1000 * 4 + (4 + 4) * 1000 * 4
    g.T = 0.0
    assert bench.accept_bytes(g) == (4 + 4) * 1000 * 4
    r = W.make_accept_inputs("r", W.MODE_REJECT, 1.0, 1000, [4, 8], [4, 3], seed=2)
    assert bench.accept_bytes(r) == (4 + 4) * 1000 * 4 + (4 + 3) * 1000 * 4
    assert bench.kernel_launches(r) == 7 and bench.kernel_launches(g) == 4 and bench.kernel_launches(None) == 2


def test_rope_bytes():
    a = W.make_attn_inputs("t", [1], [2], [3], 4, 2, 64, W.F32, seed=5)
    assert bench.rope_bytes(a) == 2 * 8 * 6 * 64 * 4


def test_code_digest_ignores_comments_only():
    src = "__global__ void k(float* x) {  // scale\n  /* one */ x[0] = 2.f * x[0];\n  const char* s = \"a // b\";\n}\n"
    same = "// header comment\n__global__ void k(float* x) {\n    x[0] = 2.f * x[0];   // twice\n  const char* s = \"a // b\";\n}"
    other = src.replace("2.f", "3.f")
    lit = src.replace("a // b", "a // c")
    assert bench.strip_comments(src) == bench.strip_comments(same)
    assert bench.strip_comments(src) != bench.strip_comments(other)
    assert bench.strip_comments(src) != bench.strip_comments(lit)
    for kern in bench.KERNEL_SOURCES:
        assert len(bench.code_digest(kern)) == 16
